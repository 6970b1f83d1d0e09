// Gram matrices of the factor step on the 5th-generation tensor cores:
// tcgen05.mma (bf16 x bf16 -> fp32 in TMEM), operands staged by TMA with
// 128-byte swizzle, one elected thread issuing MMAs, a 4-stage mbarrier
// pipeline, fp32 epilogue through tcgen05.ld.  bf16 inputs multiply exactly,
// so these Grams are the exact sums of products up to fp32 accumulation.
//
//   token Gram   S_T[u] = sum_h X_h X_h^T            (T x T, K = H*D)
//     ["Technical Summary: A JOLT for the KV Cache", Methodology 1 and 4:
//      the token-mode SVD of the unfolding, the expensive one on long
//      contexts]  Tiles of 128 x 128 on and above the diagonal; the lower
//      triangle is written as the mirror.  Operands are K-major (rows of X_h).
//   feature Gram S_d[u] = sum_{h,t} x x^T             (D x D, K = H*T)
//     ["Joint Tucker-rank and residual-bit KV allocator", Implementation
//      notes: SVD of the feature unfolding]  Split over row ranges, each CTA
//      writes one fp32 partial, summed afterwards in f64.  Operands are
//      MN-major: X's rows are read as stored, no transpose.
//
// Warp roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues
// MMAs, warps 2-5 drain the accumulator.  All mbarrier waits are bounded; a
// timeout sets the unit's status word and the CTA still frees its TMEM.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

#include <string.h>


namespace jolt {

namespace tc {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapDataType dt) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, rank, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

using tc::encode_fn;
using tc::make_map;

namespace {

constexpr int STAGES = 4;
constexpr int TILE = 128;
constexpr int KCH = 64;                       // bf16 elements per 128-byte row
constexpr int TILE_BYTES = TILE * KCH * 2;    // 16 KB
constexpr int TC_THREADS = 192;

struct TcArgs {
  int T, D, H;
  int nt;             // token tiles per dim (T / 128 rounded up)
  int rows_per;       // feature Gram: rows per split
  int nsplit;
  float* out;         // unit 0 base of the output (S_T or the partials)
  long long out_us;   // output unit stride, floats
  char* ws;
  size_t ub, o_status;
};

struct Smem {
  // operand stages come first (1024-byte aligned by the launch)
  uint64_t full[STAGES], empty[STAGES], accum;
  uint32_t tmem;
};

__device__ __forceinline__ void set_err(const TcArgs& a, int u) {
  atomicOr((int*)(a.ws + (size_t)u * a.ub + a.o_status), ST_TIMEOUT);
}

// Drain one 128 x 128 fp32 accumulator: warp q (of 4) owns TMEM lanes
// 32q..32q+31 = tile rows; calls f(row_in_tile, col_in_tile, v[32]) per
// 32-column slab.
template <typename F>
__device__ __forceinline__ void drain(uint32_t tmem, int q, F&& f) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int c = 0; c < TILE / 32; ++c) {
    float v[32];
    tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(c * 32), v);
    f(32 * q + lane, c * 32, v);
  }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
gram_tok_tc_kernel(const __grid_constant__ CUtensorMap tm, TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  Smem* S = (Smem*)(base + STAGES * 2 * TILE_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int u = blockIdx.y;
  // upper-triangular tile (mi <= ni)
  int mi = 0, idx = blockIdx.x;
  while (idx >= a.nt - mi) { idx -= a.nt - mi; ++mi; }
  const int ni = mi + idx;
  const bool diag = (mi == ni);
  const int nk = a.H * (a.D / KCH);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&S->accum), 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&S->tmem), TILE);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    const uint32_t bytes = diag ? TILE_BYTES : 2 * TILE_BYTES;
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % STAGES, r = kk / STAGES;
      if (r > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[s]), (r - 1) & 1)) { ok = false; break; }
      const int h = kk / (a.D / KCH), k0 = (kk % (a.D / KCH)) * KCH;
      const uint32_t fb = tc::smem_u32(&S->full[s]);
      tc::mbar_expect_tx(fb, bytes);
      const uint32_t sa = tc::smem_u32(base + s * 2 * TILE_BYTES);
      tc::tma_load_3d(sa, &tm, k0, mi * TILE, u * a.H + h, fb);
      if (!diag) tc::tma_load_3d(sa + TILE_BYTES, &tm, k0, ni * TILE, u * a.H + h, fb);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::idesc_bf16(TILE, TILE, 0, 0);
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % STAGES, r = kk / STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[s]), r & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + s * 2 * TILE_BYTES);
      const uint32_t sb = diag ? sa : sa + TILE_BYTES;
#pragma unroll
      for (int k4 = 0; k4 < KCH / 16; ++k4) {
        const uint64_t ad = tc::sdesc_sw128(sa + 32 * k4, 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(sb + 32 * k4, 16, 1024);
        tc::mma_f16(tmem, ad, bd, idesc, (kk | k4) != 0);
      }
      tc::mma_commit(tc::smem_u32(&S->empty[s]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  } else if (warp >= 2) {
    const int q = warp & 3;
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) {
      ok = false;
    } else {
      tc::tc_fence_after();
      float* C = a.out + (long long)u * a.out_us;
      const int T = a.T;
      drain(tmem, q, [&](int rt, int c0, const float (&v)[32]) {
        const int row = mi * TILE + rt;
        if (row < T) {
          float* cr = C + (long long)row * T + ni * TILE + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (ni * TILE + c0 + j < T) cr[j] = v[j];
        }
        if (!diag) {
          // mirror: lanes hold consecutive rows, so each column is one
          // coalesced 128-byte store
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = ni * TILE + c0 + j;
            if (col < T && row < T) C[(long long)col * T + row] = v[j];
          }
        }
      });
    }
  }
  if (!ok) set_err(a, u);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, TILE);
}

// Feature Gram partials, D = 128: rows [s*rows_per, (s+1)*rows_per) of unit u.
// One stage = 64 rows x 128 features in two 64-feature swizzle atoms (8 KB
// each); the A and B operands are the same tile (MN-major, LBO = 8 KB between
// the feature atoms, SBO = 1 KB between 8-row groups).
__global__ void __launch_bounds__(TC_THREADS, 1)
gram_feat_tc_kernel(const __grid_constant__ CUtensorMap tm, TcArgs a) {
  constexpr int SBYTES = 2 * 64 * 128;   // 16 KB per stage
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  Smem* S = (Smem*)(base + STAGES * SBYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int u = blockIdx.y, sp = blockIdx.x;
  const long long row0 = (long long)u * a.H * a.T + (long long)sp * a.rows_per;
  const int nk = a.rows_per / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&S->accum), 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&S->tmem), TILE);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % STAGES, r = kk / STAGES;
      if (r > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[s]), (r - 1) & 1)) { ok = false; break; }
      const uint32_t fb = tc::smem_u32(&S->full[s]);
      tc::mbar_expect_tx(fb, SBYTES);
      const uint32_t sa = tc::smem_u32(base + s * SBYTES);
      const int rr = (int)(row0 + (long long)kk * 64);
      tc::tma_load_2d(sa, &tm, 0, rr, fb);
      tc::tma_load_2d(sa + SBYTES / 2, &tm, 64, rr, fb);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::idesc_bf16(TILE, TILE, 1, 1);
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % STAGES, r = kk / STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[s]), r & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + s * SBYTES);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const uint64_t d = tc::sdesc_sw128(sa + 2048 * k4, SBYTES / 2, 1024);
        tc::mma_f16(tmem, d, d, idesc, (kk | k4) != 0);
      }
      tc::mma_commit(tc::smem_u32(&S->empty[s]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  } else if (warp >= 2) {
    const int q = warp & 3;
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) {
      ok = false;
    } else {
      tc::tc_fence_after();
      float* P = a.out + (long long)u * a.out_us + (long long)sp * 128 * 128;
      drain(tmem, q, [&](int rt, int c0, const float (&v)[32]) {
        float4* pr = reinterpret_cast<float4*>(P + rt * 128 + c0);
#pragma unroll
        for (int j = 0; j < 8; ++j) pr[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      });
    }
  }
  if (!ok) set_err(a, u);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, TILE);
}

// Z[u] (T x L) = S[u] (T x T) V[u] (T x L) on kind::tf32 with three
// products: S V + S V_lo + S_lo V, where x_lo = x - trunc_tf32(x) is exact in
// fp32; the dropped S_lo V_lo and the truncation of the lo parts leave about
// 2^-21 relative error per product, the size of fp32 accumulation itself.
// One CTA per 128-row tile of one unit.  Both operands are K-major: S rows,
// and V^T (64 x T) written by split_v_kernel.
constexpr int SV_STAGES = 3;
constexpr int SV_A = TILE * 32 * 4;          // 16 KB: 128 rows x 32 k (fp32)
constexpr int SV_B = 64 * 32 * 4;            // 8 KB: 64 rows (n) x 32 k
constexpr int SV_STAGE = 2 * SV_A + 2 * SV_B;

struct SvArgs {
  int T, L;
  float* Z;
  long long z_us;      // floats
  const int* flags;
  long long f_us;      // ints
  char* ws;
  size_t ub, o_status;
};

__global__ void __launch_bounds__(TC_THREADS, 1)
sv_tc_kernel(const __grid_constant__ CUtensorMap tS, const __grid_constant__ CUtensorMap tSl,
             const __grid_constant__ CUtensorMap tV, const __grid_constant__ CUtensorMap tVl,
             SvArgs a) {
  const int u = blockIdx.y, mi = blockIdx.x;
  if (a.flags && a.flags[u * a.f_us]) return;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  struct Bars { uint64_t full[SV_STAGES], empty[SV_STAGES], accum; uint32_t tmem; };
  Bars* S = (Bars*)(base + SV_STAGES * SV_STAGE);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int nk = (a.T + 31) / 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SV_STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&S->accum), 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&S->tmem), 64);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;
  if (warp == 0 && lane == 0) {
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % SV_STAGES, r = kk / SV_STAGES;
      if (r > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[s]), (r - 1) & 1)) { ok = false; break; }
      const uint32_t fb = tc::smem_u32(&S->full[s]);
      tc::mbar_expect_tx(fb, SV_STAGE);
      const uint32_t sa = tc::smem_u32(base + s * SV_STAGE);
      tc::tma_load_3d(sa, &tS, kk * 32, mi * TILE, u, fb);
      tc::tma_load_3d(sa + SV_A, &tSl, kk * 32, mi * TILE, u, fb);
      tc::tma_load_3d(sa + 2 * SV_A, &tV, kk * 32, 0, u, fb);
      tc::tma_load_3d(sa + 2 * SV_A + SV_B, &tVl, kk * 32, 0, u, fb);
    }
  } else if (warp == 1 && lane == 0) {
    // kind::tf32, fp32 accumulate, A and B K-major, M = 128, N = 64
    constexpr uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                               ((uint32_t)(64 >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % SV_STAGES, r = kk / SV_STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[s]), r & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + s * SV_STAGE);
      const uint32_t sb = sa + 2 * SV_A;
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const uint64_t ah = tc::sdesc_sw128(sa + 32 * k4, 16, 1024);
        const uint64_t al = tc::sdesc_sw128(sa + SV_A + 32 * k4, 16, 1024);
        const uint64_t bh = tc::sdesc_sw128(sb + 32 * k4, 16, 1024);
        const uint64_t bl = tc::sdesc_sw128(sb + SV_B + 32 * k4, 16, 1024);
        tc::mma_tf32(tmem, ah, bh, idesc, (kk | k4) != 0);
        tc::mma_tf32(tmem, ah, bl, idesc, 1);
        tc::mma_tf32(tmem, al, bh, idesc, 1);
      }
      tc::mma_commit(tc::smem_u32(&S->empty[s]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  } else if (warp >= 2) {
    const int q = warp & 3;
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) {
      ok = false;
    } else {
      tc::tc_fence_after();
      const int row = mi * TILE + 32 * q + lane;
      float* zr = a.Z + (long long)u * a.z_us + (long long)row * 64;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(c * 32), v);
        if (row < a.T) {
          float4* z4 = reinterpret_cast<float4*>(zr + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) z4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
    }
  }
  if (!ok) atomicOr((int*)(a.ws + (size_t)u * a.ub + a.o_status), ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 64);
}

// lo[i] = x[i] - trunc_tf32(x[i]) over n floats per unit.
__global__ void tf32_lo_kernel(const char* ws, size_t ub, size_t o_in, size_t o_out, long long n,
                               const int* flags, long long f_us) {
  const int u = blockIdx.y;
  if (flags && flags[u * f_us]) return;
  const float* x = (const float*)(ws + (size_t)u * ub + o_in);
  float* y = (float*)((char*)ws + (size_t)u * ub + o_out);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float v = x[i];
    y[i] = v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  }
}

// V^T and its tf32 low part (64 x T each) from V (T x 64), via a 32 x 32
// shared-memory transpose per block.
__global__ void split_v_kernel(const char* ws, size_t ub, size_t o_V, size_t o_Vt, size_t o_Vtl,
                               int T, const int* flags, long long f_us) {
  const int u = blockIdx.z;
  if (flags && flags[u * f_us]) return;
  __shared__ float tile[32][33];
  const float* V = (const float*)(ws + (size_t)u * ub + o_V);
  float* Vt = (float*)((char*)ws + (size_t)u * ub + o_Vt);
  float* Vtl = (float*)((char*)ws + (size_t)u * ub + o_Vtl);
  const int t0 = blockIdx.x * 32, n0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int t = t0 + r;
    tile[r][tx] = t < T ? V[(long long)t * 64 + n0 + tx] : 0.f;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int n = n0 + r, t = t0 + tx;
    if (t < T) {
      const float v = tile[tx][r];
      Vt[(long long)n * T + t] = v;
      Vtl[(long long)n * T + t] = v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
    }
  }
}

// Token Grams of the truncated feature ranks: for problem p = u * ndt + id,
// S[p] = A A^T with A = Yt[u][:, :H rd[id]] (T x H rd[id]), on kind::tf32
// with the three-product split (A_hi A_hi^T + A_hi A_lo^T + A_lo A_hi^T).
// Yt[u] is [T][RD*H] fp32 with column j*H + h = Y[u][h][:, j], so that the
// feature ranks j < rd of one Gram are a leading column range.  Upper-
// triangular 128 x 128 tiles, mirrored into the lower triangle.
constexpr int YG_STAGES = 2;
constexpr int YG_A = TILE * 32 * 4;          // 16 KB: 128 rows x 32 k
constexpr int YG_STAGE = 4 * YG_A;           // A hi, A lo, B hi, B lo

struct YgArgs {
  int T, ndt, nt;
  int k1s[JOLT_MAX_GRID];   // column count H * rd[id] of each truncated rank
  float* S;
  long long s_us;
  char* ws;
  size_t ub, o_status;
};

__global__ void __launch_bounds__(TC_THREADS, 1)
ygram_tc_kernel(const __grid_constant__ CUtensorMap tH, const __grid_constant__ CUtensorMap tL,
                YgArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  struct Bars { uint64_t full[YG_STAGES], empty[YG_STAGES], accum; uint32_t tmem; };
  Bars* S = (Bars*)(base + YG_STAGES * YG_STAGE);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int p = blockIdx.y, u = p / a.ndt;
  int mi = 0, idx = blockIdx.x;
  while (idx >= a.nt - mi) { idx -= a.nt - mi; ++mi; }
  const int ni = mi + idx;
  const bool diag = (mi == ni);
  const int klen = a.k1s[p % a.ndt];
  const int nk = (klen + 31) / 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < YG_STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&S->accum), 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&S->tmem), TILE);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;
  if (warp == 0 && lane == 0) {
    const uint32_t bytes = diag ? 2 * YG_A : 4 * YG_A;
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % YG_STAGES, r = kk / YG_STAGES;
      if (r > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[s]), (r - 1) & 1)) { ok = false; break; }
      const uint32_t fb = tc::smem_u32(&S->full[s]);
      tc::mbar_expect_tx(fb, bytes);
      const uint32_t sa = tc::smem_u32(base + s * YG_STAGE);
      const int kc = kk * 32;
      tc::tma_load_3d(sa, &tH, kc, mi * TILE, u, fb);
      tc::tma_load_3d(sa + YG_A, &tL, kc, mi * TILE, u, fb);
      if (!diag) {
        tc::tma_load_3d(sa + 2 * YG_A, &tH, kc, ni * TILE, u, fb);
        tc::tma_load_3d(sa + 3 * YG_A, &tL, kc, ni * TILE, u, fb);
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                               ((uint32_t)(TILE >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
    bool first = true;
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % YG_STAGES, r = kk / YG_STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[s]), r & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + s * YG_STAGE);
      const uint32_t sb = diag ? sa : sa + 2 * YG_A;
      const int steps = min(4, (klen - kk * 32) / 8);   // K ranges are multiples of 8
      for (int k4 = 0; k4 < steps; ++k4) {
        const uint64_t ah = tc::sdesc_sw128(sa + 32 * k4, 16, 1024);
        const uint64_t al = tc::sdesc_sw128(sa + YG_A + 32 * k4, 16, 1024);
        const uint64_t bh = tc::sdesc_sw128(sb + 32 * k4, 16, 1024);
        const uint64_t bl = tc::sdesc_sw128(sb + YG_A + 32 * k4, 16, 1024);
        tc::mma_tf32(tmem, ah, bh, idesc, first ? 0u : 1u);
        tc::mma_tf32(tmem, ah, bl, idesc, 1);
        tc::mma_tf32(tmem, al, bh, idesc, 1);
        first = false;
      }
      tc::mma_commit(tc::smem_u32(&S->empty[s]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  } else if (warp >= 2) {
    const int q = warp & 3;
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) {
      ok = false;
    } else {
      tc::tc_fence_after();
      float* C = a.S + (long long)p * a.s_us;
      const int T = a.T;
      drain(tmem, q, [&](int rt, int c0, const float (&v)[32]) {
        const int row = mi * TILE + rt;
        if (row < T) {
          float* cr = C + (long long)row * T + ni * TILE + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (ni * TILE + c0 + j < T) cr[j] = v[j];
        }
        if (!diag) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = ni * TILE + c0 + j;
            if (col < T && row < T) {
              C[(long long)col * T + row] = v[j];
            }
          }
        }
      });
    }
  }
  if (!ok) atomicOr((int*)(a.ws + (size_t)p * a.ub + a.o_status), ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, TILE);
}

// Yt[u][t][j*H + h] = Y[u][h][t][j] and its tf32 low part.
__global__ void ytrans_kernel(const char* ws, size_t ub, size_t o_Y, size_t o_Yt, int H, int T,
                              int RD) {
  const int u = blockIdx.y;
  const float* Y = (const float*)(ws + (size_t)u * ub + o_Y);
  float* Yt = (float*)((char*)ws + (size_t)u * ub + o_Yt);
  float* Ytl = Yt + (size_t)T * RD * H;
  const int K = RD * H;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < (long long)T * K;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / K), c = (int)(e % K), j = c / H, h = c % H;
    const float v = Y[((long long)h * T + t) * RD + j];
    Yt[e] = v;
    Ytl[e] = v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  }
}

// ---------------------------------------------------------------- sweep (TC)
// The candidate sweep with the dense products on the tensor cores, for bf16
// X with D = 128 and truncated ranks <= 32.  One CTA scores 128 tokens of one
// head with two threads per token row, each owning one 64-column half (warps
// w and w + 4 read the same TMEM lane quarter; the row maximum is exchanged
// through shared memory between the pair):
//   * QX = X (diag(sigma) H) by kind::f16 MMAs (bf16 X and the +-1 matrix are
//     exact; fp32 accumulate) into TMEM columns [0, 128);
//   * every reconstruction in the rotated domain, U_T W or Y16 (Q U_d)^T at a
//     rank checkpoint r, as K[:, :r] B[:r, :] by kind::tf32 MMAs (K, fp16
//     values, is exact in tf32; B split hi + lo) into TMEM columns [128, 256),
//     recomputed from k = 0 for each checkpoint (columns r..8*ceil(r/8) of K
//     zeroed meanwhile);
//   * each thread then reads its half row y = QX / sqrt(D) - P back in
//     16-column chunks and scores every b exactly as the SIMT sweep does (row
//     max, fp16 scale, round-half-even by the magic constant, squared error).
// The K and B operands are written by the threads in the 128-byte swizzled
// K-major layout (16-byte unit u of row r at u ^ (r % 8)), X and the sign
// matrix arrive by TMA in the same layout.
constexpr int STC_ROWS = 128, STC_THREADS = 256;
constexpr int STC_XBYTES = STC_ROWS * 256;       // 128 rows x 128 bf16
constexpr int STC_KBYTES = STC_ROWS * 128;       // 128 rows x 32 fp32

struct SweepTcArgs {
  int H, T, nT, nd, nb, nTt, ndt, RT, RD, hasFullT, hasFullD;
  int rT[JOLT_MAX_GRID], rd[JOLT_MAX_GRID], b[4];
  float rq[4];
  int ncand, tiles_t;
  char* ws;
  size_t ub, o_UT16, o_W, o_Y16, o_QUd, o_status;
  float* part;
  long long part_us;
};

__device__ __forceinline__ uint32_t sw128(int r, int byte) {
  return (uint32_t)(r * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15)));
}

// 16 columns of this thread's TMEM lane into registers, without waiting.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}
// Wait for this thread's TMEM loads, tied to the registers it makes valid
// (so that no use of them can be scheduled before it).
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16], uint32_t (&q)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(q[0]), "+r"(q[1]),
                 "+r"(q[2]), "+r"(q[3]), "+r"(q[4]), "+r"(q[5]), "+r"(q[6]), "+r"(q[7]),
                 "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]), "+r"(q[12]), "+r"(q[13]),
                 "+r"(q[14]), "+r"(q[15])
               :
               : "memory");
}

// One pass over this thread's 64-column half row (`trow` carries the half's
// column offset), STC_CH columns at a time, with the loads of the next
// STC_CH columns in flight while the current ones are used:
// f(y0, y1) is called on consecutive pairs of y = QX rs - P (with_qx) or
// y = P rs.
constexpr int STC_CH = 16;
template <typename F>
__device__ __forceinline__ void stc_pass(uint32_t trow, bool with_qx, float rs, F&& f) {
  const float2 rs2 = make_float2(rs, rs);
  uint32_t pa[STC_CH], qa[STC_CH], pb[STC_CH], qb[STC_CH];
  auto issue = [&](uint32_t addr, uint32_t (&r)[STC_CH]) { tmem_ld16_issue(addr, r); };
  issue(trow + 128, pa);
  if (with_qx) issue(trow, qa);
  if (with_qx) tmem_ld_wait(pa, qa); else tmem_ld_wait(pa);
  auto use = [&](const uint32_t (&p)[STC_CH], const uint32_t (&q)[STC_CH]) {
#pragma unroll
    for (int j = 0; j < STC_CH; j += 2) {
      const float2 pp = make_float2(__uint_as_float(p[j]), __uint_as_float(p[j + 1]));
      const float2 y = with_qx
                           ? __ffma2_rn(make_float2(__uint_as_float(q[j]), __uint_as_float(q[j + 1])),
                                        rs2, make_float2(-pp.x, -pp.y))
                           : __fmul2_rn(pp, rs2);
      f(y);
    }
  };
#pragma unroll
  for (int c = 0; c < 64; c += 2 * STC_CH) {
    // columns c .. c + STC_CH - 1 are in (pa, qa); fetch the next STC_CH
    // into (pb, qb)
    issue(trow + 128 + c + STC_CH, pb);
    if (with_qx) issue(trow + c + STC_CH, qb);
    use(pa, qa);
    if (with_qx) tmem_ld_wait(pb, qb); else tmem_ld_wait(pb);
    if (c + 2 * STC_CH < 64) {
      issue(trow + 128 + c + 2 * STC_CH, pa);
      if (with_qx) issue(trow + c + 2 * STC_CH, qa);
    }
    use(pb, qb);
    if (c + 2 * STC_CH < 64) {
      if (with_qx) tmem_ld_wait(pa, qa); else tmem_ld_wait(pa);
    }
  }
}

// Score one candidate from TMEM: half row `trow` (this thread's lane
// address and column offset); y = QX rs - P (with_qx) or y = P rs (the
// whole-modes residual).  The two halves of a row meet on the row maximum
// through rmax[half][lr] and a 64-thread named barrier of their warp pair;
// the squared errors of the halves add in the cells.  The caller separates
// consecutive calls by a CTA barrier (rmax is rewritten by the next call).
__device__ __forceinline__ void stc_score(uint32_t trow, bool with_qx, float rs,
                                          const SweepTcArgs& a, float* cells, int cell0,
                                          float* rmax, int lr, int half, int pair) {
  float m0 = 0.f, m1 = 0.f;
  float2 e0 = make_float2(0.f, 0.f);
  stc_pass(trow, with_qx, rs, [&](float2 y) {
    m0 = fmaxf(m0, fabsf(y.x));
    m1 = fmaxf(m1, fabsf(y.y));
    e0 = __ffma2_rn(y, y, e0);
  });
  float m = fmaxf(m0, m1);
  rmax[half * STC_ROWS + lr] = m;
  asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
  m = fmaxf(m, rmax[(half ^ 1) * STC_ROWS + lr]);
  float s[4], inv[4];
#pragma unroll
  for (int ib = 0; ib < 4; ++ib) {
    s[ib] = 0.f; inv[ib] = 0.f;
    if (ib < a.nb && a.b[ib] > 0) {
      s[ib] = round_f16(m * a.rq[ib]);
      float r;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s[ib]));
      inv[ib] = s[ib] > 0.f ? r : 0.f;
    }
  }
  const float2 M2 = make_float2(12582912.0f, 12582912.0f), nM2 = make_float2(-12582912.0f, -12582912.0f);
  float2 eb[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  stc_pass(trow, with_qx, rs, [&](float2 y) {
#pragma unroll
    for (int ib = 0; ib < 4; ++ib) {
      if (ib >= a.nb || a.b[ib] == 0) continue;
      const float2 i2 = make_float2(inv[ib], inv[ib]), ns2 = make_float2(-s[ib], -s[ib]);
      const float2 qq = __fadd2_rn(__ffma2_rn(y, i2, M2), nM2);
      const float2 d = __ffma2_rn(ns2, qq, y);
      eb[ib] = __ffma2_rn(d, d, eb[ib]);
    }
  });
  float v[4];
#pragma unroll
  for (int ib = 0; ib < 4; ++ib) v[ib] = (ib < a.nb && a.b[ib] == 0) ? e0.x + e0.y : eb[ib].x + eb[ib].y;
#pragma unroll
  for (int ib = 0; ib < 4; ++ib)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[ib] += __shfl_xor_sync(0xffffffffu, v[ib], o);
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int ib = 0; ib < 4; ++ib)
      if (ib < a.nb) atomicAdd(&cells[cell0 + ib], v[ib]);
}

__global__ void __launch_bounds__(STC_THREADS, 2)
sweep_tc_kernel(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tHs,
                SweepTcArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  unsigned char* sX = base;                       // X tile (2 chunks), later K operand
  unsigned char* sH = base + STC_XBYTES;          // sign matrix (2 chunks), later B hi / lo
  float* cells = (float*)(base + 2 * STC_XBYTES); // [ncand + 1]
  struct Bars { uint64_t tma, mma; uint32_t tmem; int nz; };
  Bars* S = (Bars*)(cells + 260);
  float* rmax = cells + 260 + 16;                 // [2][128] half-row maxima
  const int t = threadIdx.x, warp = t >> 5;
  const int lr = t & (STC_ROWS - 1), half = t >> 7;  // token row, column half
  const int tt = blockIdx.x, h = blockIdx.y, u = blockIdx.z;
  const int t0 = tt * STC_ROWS, row = t0 + lr;
  const bool in = row < a.T;
  char* ub = a.ws + (size_t)u * a.ub;
  for (int i = t; i <= a.ncand; i += STC_THREADS) cells[i] = 0.f;
  if (t == 0) {
    tc::mbar_init(tc::smem_u32(&S->tma), 1);
    tc::mbar_init(tc::smem_u32(&S->mma), 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&S->tmem), 256);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 64 * half;
  bool ok = true;
  uint32_t mma_phase = 0;
  auto mma_wait = [&]() {
    if (!tc::mbar_wait(tc::smem_u32(&S->mma), mma_phase & 1)) ok = false;
    ++mma_phase;
    tc::tc_fence_after();
  };
  // ---- X and the sign matrix by TMA; QX = X Hs into TMEM [0, 128)
  if (t == 0) {
    const uint32_t fb = tc::smem_u32(&S->tma);
    tc::mbar_expect_tx(fb, 2 * STC_XBYTES);
    const int xr = u * a.H + h;
    tc::tma_load_3d(tc::smem_u32(sX), &tX, 0, t0, xr, fb);
    tc::tma_load_3d(tc::smem_u32(sX + STC_XBYTES / 2), &tX, 64, t0, xr, fb);
    tc::tma_load_3d(tc::smem_u32(sH), &tHs, 0, 0, u, fb);
    tc::tma_load_3d(tc::smem_u32(sH + STC_XBYTES / 2), &tHs, 64, 0, u, fb);
  }
  if (!tc::mbar_wait(tc::smem_u32(&S->tma), 0)) ok = false;
  constexpr uint32_t idesc16 = tc::idesc_bf16(128, 128, 0, 0);
  constexpr uint32_t idesc32 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(128 >> 3) << 17) |
                               ((uint32_t)(128 >> 4) << 24);
  auto mma_x = [&](uint32_t dcol) {   // D[dcol..] = sX sH^T over K = 128 (bf16)
    if (t == 0) {
      tc::tc_fence_after();
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sX + kc * (STC_XBYTES / 2)) + 32 * k, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sH + kc * (STC_XBYTES / 2)) + 32 * k, 16, 1024);
          tc::mma_f16(tmem + dcol, ad, bd, idesc16, (kc | k) != 0);
        }
      tc::mma_commit(tc::smem_u32(&S->mma));
    }
  };
  mma_x(0);
  mma_wait();
  // ---- ||x||^2 and the whole-modes residual x - fp16(x) (in place, bf16-exact)
  const float rs = rsqrtf(128.f);
  {
    float xn = 0.f;
    int nz = 0;
#pragma unroll 4
    for (int c = 0; c < 64; c += 8) {
      unsigned char* p = sX + half * (STC_XBYTES / 2) + sw128(lr, c * 2);
      uint4 v = *reinterpret_cast<uint4*>(p);
      __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x = __bfloat162float(e[i]);
        xn = fmaf(x, x, xn);
        const float r = x - round_f16(x);
        nz |= (r != 0.f);
        e[i] = __float2bfloat16_rn(r);
      }
      *reinterpret_cast<uint4*>(p) = v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) xn += __shfl_xor_sync(0xffffffffu, xn, o);
    if ((t & 31) == 0) atomicAdd(&cells[a.ncand], xn);
    nz = __syncthreads_or(nz);
    if (a.hasFullT && a.hasFullD && nz) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      mma_x(128);
      mma_wait();
      stc_score(trow, false, rs, a, cells, ((a.nT - 1) * a.nd + (a.nd - 1)) * a.nb, rmax, lr,
                half, warp & 3);
    }
  }
  // ---- rank chains: P = K[:, :r] B[:r, :] for each checkpoint r
  unsigned char* sK = sX;                 // 128 x 32 fp32
  unsigned char* sBh = sH;                // 128 (n) x 32 fp32
  unsigned char* sBl = sH + STC_KBYTES;
  auto run_chain = [&](const __half* Kg, long long k_ld, int kn, const float* Bg, int nck,
                       const int* ranks, int cellbase, int cellstride) {
    tc::tc_fence_before();
    __syncthreads();   // previous MMAs and TMEM reads done, operands free
    // K rows (this thread's token row, columns 16 half .. 16 half + 15),
    // fp16 -> fp32, zero past kn / T
    const int k0 = 16 * half;
    if (kn == 32 && (k_ld & 7) == 0) {
      uint4 raw[2];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        raw[i] = in ? reinterpret_cast<const uint4*>(Kg + (long long)row * k_ld + k0)[i] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const __half* hv = reinterpret_cast<const __half*>(&raw[i]);
        float4 v0, v1;
        v0.x = __half2float(hv[0]); v0.y = __half2float(hv[1]); v0.z = __half2float(hv[2]); v0.w = __half2float(hv[3]);
        v1.x = __half2float(hv[4]); v1.y = __half2float(hv[5]); v1.z = __half2float(hv[6]); v1.w = __half2float(hv[7]);
        *reinterpret_cast<float4*>(sK + sw128(lr, (k0 + 8 * i) * 4)) = v0;
        *reinterpret_cast<float4*>(sK + sw128(lr, (k0 + 8 * i + 4) * 4)) = v1;
      }
    } else {
      for (int k = k0; k < k0 + 16; k += 4) {
        float4 v;
        float* pv = reinterpret_cast<float*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          pv[i] = (in && k + i < kn) ? __half2float(Kg[(long long)row * k_ld + k + i]) : 0.f;
        *reinterpret_cast<float4*>(sK + sw128(lr, k * 4)) = v;
      }
    }
    // B^T rows: n = lr, B^T[n][k] = B[k][n] for this half's k, split hi + lo
    for (int k = k0; k < k0 + 16; k += 4) {
      float4 hi, lo;
      float* ph = reinterpret_cast<float*>(&hi);
      float* pl = reinterpret_cast<float*>(&lo);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float b = (k + i < kn) ? Bg[(long long)(k + i) * 128 + lr] : 0.f;
        const float bh = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
        ph[i] = bh;
        pl[i] = b - bh;
      }
      *reinterpret_cast<float4*>(sBh + sw128(lr, k * 4)) = hi;
      *reinterpret_cast<float4*>(sBl + sw128(lr, k * 4)) = lo;
    }
    for (int ci = 0; ci < nck; ++ci) {
      const int r = ranks[ci];
      const int ks = (r + 7) >> 3;
      // zero K columns r .. 8 ks - 1 of this row for this checkpoint (each
      // half its own columns)
      float saved[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = r + i;
        saved[i] = 0.f;
        if (k < 8 * ks && (k >> 4) == half) {
          float* p = reinterpret_cast<float*>(sK + sw128(lr, k * 4));
          saved[i] = *p;
          *p = 0.f;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc::tc_fence_before();
      __syncthreads();
      if (t == 0) {
        tc::tc_fence_after();
        for (int k = 0; k < ks; ++k) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sK) + 32 * k, 16, 1024);
          const uint64_t bh = tc::sdesc_sw128(tc::smem_u32(sBh) + 32 * k, 16, 1024);
          const uint64_t bl = tc::sdesc_sw128(tc::smem_u32(sBl) + 32 * k, 16, 1024);
          tc::mma_tf32(tmem + 128, ad, bh, idesc32, k != 0);
          tc::mma_tf32(tmem + 128, ad, bl, idesc32, 1);
        }
        tc::mma_commit(tc::smem_u32(&S->mma));
      }
      mma_wait();
      stc_score(trow, true, rs, a, cells, cellbase + ci * cellstride, rmax, lr, half, warp & 3);
      // restore the zeroed columns for the next checkpoint
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = r + i;
        if (k < 8 * ks && (k >> 4) == half) *reinterpret_cast<float*>(sK + sw128(lr, k * 4)) = saved[i];
      }
      tc::tc_fence_before();
      __syncthreads();
    }
  };
  if (a.hasFullT && a.ndt > 0) {
    const __half* Yh = (const __half*)(ub + a.o_Y16) + (long long)h * a.T * a.RD;
    run_chain(Yh, a.RD, a.RD, (const float*)(ub + a.o_QUd), a.ndt, a.rd,
              ((a.nT - 1) * a.nd) * a.nb, a.nb);
  }
  if (a.nTt > 0) {
    for (int id = 0; id < a.nd; ++id) {
      const __half* Ug = (const __half*)(ub + a.o_UT16) + (long long)id * a.T * a.RT;
      const float* Wg = (const float*)(ub + a.o_W) + ((long long)id * a.H + h) * a.RT * 128;
      run_chain(Ug, a.RT, a.RT, Wg, a.nTt, a.rT, id * a.nb, a.nd * a.nb);
    }
  }
  if (!ok) atomicOr((int*)(ub + a.o_status), ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
  float* part = a.part + u * a.part_us + ((long long)h * a.tiles_t + tt) * (a.ncand + 1);
  for (int i = t; i <= a.ncand; i += STC_THREADS) part[i] = cells[i];
}

size_t tc_smem(int stage_bytes) { return (size_t)STAGES * stage_bytes + 1024 + sizeof(Smem) + 64; }

}  // namespace

bool gram_tc_supported(const Layout& L) {
  return L.dtype == JOLT_BF16 && L.D == 128 && encode_fn() != nullptr;
}

// S_T of problem u = sum_h X_h X_h^T of unit u, T x T fp32.
jolt_status gram_tok_tc(const Layout& L, int U, const void* X, char* pbase, size_t pstride,
                        cudaStream_t st) {
  CUtensorMap tm;
  const cuuint64_t dims[3] = {(cuuint64_t)L.D, (cuuint64_t)L.T, (cuuint64_t)U * L.H};
  const cuuint64_t strides[2] = {(cuuint64_t)L.D * 2, (cuuint64_t)L.T * L.D * 2};
  const cuuint32_t box[3] = {KCH, TILE, 1};
  if (!make_map(&tm, X, 3, dims, strides, box)) return JOLT_ERR_CUDA;
  TcArgs a;
  a.T = L.T; a.D = L.D; a.H = L.H;
  a.nt = (L.T + TILE - 1) / TILE;
  a.rows_per = 0; a.nsplit = 0;
  a.out = (float*)(pbase + L.p_ST);
  a.out_us = (long long)pstride / 4;
  a.ws = pbase; a.ub = pstride; a.o_status = L.p_status;
  const size_t smem = tc_smem(2 * TILE_BYTES);
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(gram_tok_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  dim3 grid(a.nt * (a.nt + 1) / 2, U);
  gram_tok_tc_kernel<<<grid, TC_THREADS, smem, st>>>(tm, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

// Feature-Gram partials Sdp[u][s] (128 x 128 fp32) over L.nsplit row ranges.
jolt_status gram_feat_tc(const Layout& L, int U, const void* X, char* ws, cudaStream_t st) {
  const long long rows = (long long)U * L.H * L.T;
  const int rows_per = (L.H / L.nsplit) * L.T;
  if (rows_per % 64) return JOLT_ERR_INVALID;
  CUtensorMap tm;
  const cuuint64_t dims[2] = {(cuuint64_t)L.D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)L.D * 2};
  const cuuint32_t box[2] = {64, 64};
  if (!make_map(&tm, X, 2, dims, strides, box)) return JOLT_ERR_CUDA;
  TcArgs a;
  a.T = L.T; a.D = L.D; a.H = L.H; a.nt = 0;
  a.rows_per = rows_per; a.nsplit = L.nsplit;
  a.out = (float*)(ws + L.o_Sdp);
  a.out_us = (long long)L.unit_bytes / 4;
  a.ws = ws; a.ub = L.unit_bytes; a.o_status = L.o_status;
  const size_t smem = tc_smem(2 * 64 * 128);
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(gram_feat_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  dim3 grid(L.nsplit, U);
  gram_feat_tc_kernel<<<grid, TC_THREADS, smem, st>>>(tm, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

bool sv_tc_supported(const Layout& L) {
  return L.L == 64 && L.T % 4 == 0 && encode_fn() != nullptr && L.p_STs != 0;
}

// S_lo = S - trunc_tf32(S) for every problem (after its S_T is final).
jolt_status split_tok_gram(const Layout& L, int np, char* pbase, size_t pstride, cudaStream_t st) {
  dim3 grid(256, np);
  tf32_lo_kernel<<<grid, 256, 0, st>>>(pbase, pstride, L.p_ST, L.p_STs, (long long)L.T * L.T,
                                       nullptr, 0);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

// Z = S V for every problem not flagged (T x 64 blocks at p_V / o_Z).
jolt_status sv_tc(const Layout& L, int np, char* pbase, size_t pstride, size_t o_Z,
                  cudaStream_t st) {
  const int* flags = (const int*)(pbase + L.p_flag);
  const long long f_us = (long long)pstride / 4;
  dim3 g2((L.T + 31) / 32, 2, np);
  split_v_kernel<<<g2, dim3(32, 8), 0, st>>>(pbase, pstride, L.p_V, L.p_Vs,
                                             L.p_Vs + (size_t)L.T * 64 * 4, L.T, flags, f_us);
  JOLT_LAUNCH_CHECK();
  CUtensorMap tS, tSl, tV, tVl;
  const cuuint64_t dS[3] = {(cuuint64_t)L.T, (cuuint64_t)L.T, (cuuint64_t)np};
  const cuuint64_t sS[2] = {(cuuint64_t)L.T * 4, (cuuint64_t)pstride};
  const cuuint32_t bS[3] = {32, TILE, 1};
  const cuuint64_t dV[3] = {(cuuint64_t)L.T, 64, (cuuint64_t)np};
  const cuuint64_t sV[2] = {(cuuint64_t)L.T * 4, (cuuint64_t)pstride};
  const cuuint32_t bV[3] = {32, 64, 1};
  const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (!make_map(&tS, pbase + L.p_ST, 3, dS, sS, bS, f32) ||
      !make_map(&tSl, pbase + L.p_STs, 3, dS, sS, bS, f32) ||
      !make_map(&tV, pbase + L.p_Vs, 3, dV, sV, bV, f32) ||
      !make_map(&tVl, pbase + L.p_Vs + (size_t)L.T * 64 * 4, 3, dV, sV, bV, f32))
    return JOLT_ERR_CUDA;
  SvArgs a;
  a.T = L.T; a.L = 64;
  a.Z = (float*)(pbase + o_Z);
  a.z_us = f_us;
  a.flags = flags;
  a.f_us = f_us;
  a.ws = pbase; a.ub = pstride; a.o_status = L.p_status;
  const size_t smem = (size_t)SV_STAGES * SV_STAGE + 1024 + 256;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(sv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem));
    attr = true;
  }
  dim3 grid((L.T + TILE - 1) / TILE, np);
  sv_tc_kernel<<<grid, TC_THREADS, smem, st>>>(tS, tSl, tV, tVl, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

bool ygram_tc_supported(const Layout& L) {
  if (!(L.o_Yt != 0 && encode_fn() != nullptr)) return false;
  for (int i = 0; i < L.ndt; ++i)
    if ((L.rd[i] * L.H) % 8) return false;
  return true;
}

// Yt = relayout of Y (once per factor call).
jolt_status ytrans(const Layout& L, int U, char* ws, cudaStream_t st) {
  dim3 grid(512, U);
  ytrans_kernel<<<grid, 256, 0, st>>>(ws, L.unit_bytes, L.o_Y, L.o_Yt, L.H, L.T, L.RD);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

// S_T of every truncated problem p = u * ndt + id: the Gram of feature ranks
// [0, rd[id]) of unit u's Y, one launch for all.
jolt_status ygram_tc(const Layout& L, int U, const char* ws, char* pbase, size_t pstride,
                     cudaStream_t st) {
  const size_t ub = L.unit_bytes;
  const int K = L.RD * L.H;
  if (L.ndt < 1 || L.ndt > JOLT_MAX_GRID) return JOLT_ERR_INVALID;
  CUtensorMap tH, tL;
  const cuuint64_t d[3] = {(cuuint64_t)K, (cuuint64_t)L.T, (cuuint64_t)U};
  const cuuint64_t sd[2] = {(cuuint64_t)K * 4, (cuuint64_t)ub};
  const cuuint32_t box[3] = {32, TILE, 1};
  const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (!make_map(&tH, ws + L.o_Yt, 3, d, sd, box, f32) ||
      !make_map(&tL, ws + L.o_Yt + (size_t)L.T * K * 4, 3, d, sd, box, f32))
    return JOLT_ERR_CUDA;
  YgArgs a;
  memset(&a, 0, sizeof(a));
  a.T = L.T;
  a.ndt = L.ndt;
  for (int i = 0; i < L.ndt; ++i) a.k1s[i] = L.rd[i] * L.H;
  a.nt = (L.T + TILE - 1) / TILE;
  a.S = (float*)(pbase + L.p_ST);
  a.s_us = (long long)pstride / 4;
  a.ws = pbase; a.ub = pstride; a.o_status = L.p_status;
  const size_t smem = (size_t)YG_STAGES * YG_STAGE + 1024 + 256;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(ygram_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  dim3 grid(a.nt * (a.nt + 1) / 2, U * L.ndt);
  ygram_tc_kernel<<<grid, TC_THREADS, smem, st>>>(tH, tL, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

// ---- tensor-core sweep
bool sweep_tc_supported(const Layout& L) {
  if (!(L.dtype == JOLT_BF16 && L.D == 128 && L.RT <= 32 && L.RD <= 32 && L.o_Hs != 0 &&
        encode_fn() != nullptr && L.ncand + 1 <= 260 && L.nb <= 4))
    return false;
  return true;
}

jolt_status sweep_tc_run(const Layout& L, int U, const void* X, char* ws, float* part,
                         long long part_us, int* tiles_t_out, cudaStream_t st) {
  CUtensorMap tX;
  const cuuint64_t dX[3] = {128, (cuuint64_t)L.T, (cuuint64_t)U * L.H};
  const cuuint64_t sX[2] = {256, (cuuint64_t)L.T * 256};
  const cuuint32_t bX[3] = {64, 128, 1};
  if (!make_map(&tX, X, 3, dX, sX, bX)) return JOLT_ERR_CUDA;
  // the sign matrices sit one per unit region: a 3-D map (128 cols, 128 rows, unit)
  CUtensorMap tH3;
  const cuuint64_t dH3[3] = {128, 128, (cuuint64_t)U};
  const cuuint64_t sH3[2] = {256, (cuuint64_t)L.unit_bytes};
  const cuuint32_t bH3[3] = {64, 128, 1};
  if (!make_map(&tH3, ws + L.o_Hs, 3, dH3, sH3, bH3)) return JOLT_ERR_CUDA;
  SweepTcArgs a;
  memset(&a, 0, sizeof(a));
  a.H = L.H; a.T = L.T; a.nT = L.nT; a.nd = L.nd; a.nb = L.nb; a.nTt = L.nTt; a.ndt = L.ndt;
  a.RT = L.RT; a.RD = L.RD; a.hasFullT = L.hasFullT; a.hasFullD = L.hasFullD;
  for (int i = 0; i < JOLT_MAX_GRID; ++i) {
    a.rT[i] = i < L.nTt ? L.rT[i] : -1;
    a.rd[i] = i < L.ndt ? L.rd[i] : -1;
  }
  for (int i = 0; i < 4; ++i) {
    a.b[i] = L.b[i];
    a.rq[i] = L.b[i] > 0 ? 1.f / (float)((1 << (L.b[i] - 1)) - 1) : 0.f;
  }
  a.ncand = L.ncand;
  a.tiles_t = (L.T + STC_ROWS - 1) / STC_ROWS;
  a.ws = ws; a.ub = L.unit_bytes;
  a.o_UT16 = L.o_UT16; a.o_W = L.o_W; a.o_Y16 = L.o_Y16; a.o_QUd = L.o_QUd; a.o_status = L.o_status;
  a.part = part; a.part_us = part_us;
  // cells (260 floats), barriers (64 bytes), row maxima (256 floats), and
  // the 1024-byte alignment slack; 2 CTAs per SM by TMEM (256 columns each)
  const size_t smem = 2 * STC_XBYTES + 260 * 4 + 64 + 2 * STC_ROWS * 4 + 1024;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(sweep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem));
    attr = true;
  }
  dim3 grid(a.tiles_t, L.H, U);
  sweep_tc_kernel<<<grid, STC_THREADS, smem, st>>>(tX, tH3, a);
  JOLT_LAUNCH_CHECK();
  *tiles_t_out = a.tiles_t;
  return JOLT_OK;
}

}  // namespace jolt
