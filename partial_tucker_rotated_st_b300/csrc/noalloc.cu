// jolt_sweep_candidates_noalloc: the candidate sweep for callers that cannot
// allocate device memory (for example code running where cudaMalloc is not
// permitted, or a caller whose memory is owned by an allocator it may not
// call from this point).  The sweep's only scratch beyond the caller's
// buffers, the per-tile partial sums, lives in a fixed-size array of device
// memory that belongs to the library.
#include "jolt_internal.cuh"

#include <mutex>

namespace jolt {
namespace {

// Static scratch for the per-tile partial sums: every GPU that loads the
// library holds these bytes until the process exits.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)16 << 20;
__device__ __align__(256) float g_noalloc_scratch[NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int MAX_DEVICES = 64;
float* g_scratch_ptr[MAX_DEVICES];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device.  In host code the symbol is only a host-side stand-in, so the
// address must come from cudaGetSymbolAddress with the device current.
jolt_status scratch_for_current_device(float** out) {
  int dev = 0;
  JOLT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= MAX_DEVICES) return JOLT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    JOLT_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    g_scratch_ptr[dev] = (float*)p;
  }
  *out = g_scratch_ptr[dev];
  return JOLT_OK;
}

}  // namespace
}  // namespace jolt

using namespace jolt;

extern "C" jolt_status jolt_sweep_candidates_noalloc(const jolt_config* cfg, int n_units,
                                                     const void* X, const int8_t* signs,
                                                     void* ws, size_t ws_bytes, double* dist,
                                                     int64_t* cost, void* stream) {
  Layout L;
  jolt_status s = make_layout(cfg, &L);
  if (s != JOLT_OK) return s;
  if (n_units < 1 || n_units > 65535 || !X || !signs || !dist || !cost) return JOLT_ERR_INVALID;
  if (!ws || ((uintptr_t)ws % 256) || ws_bytes < (size_t)n_units * L.unit_total)
    return JOLT_ERR_WORKSPACE;
  const size_t need = (size_t)n_units * L.ntiles * (L.ncand + 1) * sizeof(float);
  if (need > NOALLOC_SCRATCH_BYTES) return JOLT_ERR_TOO_LARGE;
  float* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != JOLT_OK) return s;
  return sweep_run(L, n_units, X, signs, (char*)ws, dist, cost, (cudaStream_t)stream, scratch);
}

extern "C" size_t jolt_noalloc_scratch_bytes(void) { return NOALLOC_SCRATCH_BYTES; }
