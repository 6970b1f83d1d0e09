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
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  if (rank < 1 || rank > 5) return false;
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

// The same Grams for every truncated feature rank of a unit from one pass
// over its Yt columns: the slab of feature ranks [rd[i-1], rd[i]) (columns
// [H rd[i-1], H rd[i])) is accumulated into TMEM accumulator i (up to four,
// 128 columns each), and the epilogue writes S(rd[i]) = sum over i' <= i of
// slab i' (nested feature ranks: each Gram is a prefix sum of the slabs).
// One CTA per upper-triangular 128 x 128 tile and unit; half the tensor work
// of one product per rank.
__global__ void __launch_bounds__(TC_THREADS, 1)
ygram_pre_tc_kernel(const __grid_constant__ CUtensorMap tH, const __grid_constant__ CUtensorMap tL,
                    YgArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  struct Bars { uint64_t full[YG_STAGES], empty[YG_STAGES], accum; uint32_t tmem; };
  Bars* S = (Bars*)(base + YG_STAGES * YG_STAGE);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int u = blockIdx.y;
  int mi = 0, idx = blockIdx.x;
  while (idx >= a.nt - mi) { idx -= a.nt - mi; ++mi; }
  const int ni = mi + idx;
  const bool diag = (mi == ni);
  const int klen = a.k1s[a.ndt - 1];
  const int nk = (klen + 31) / 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < YG_STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&S->accum), 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&S->tmem), 512);
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
    int slab = 0;
    bool first = true;
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % YG_STAGES, r = kk / YG_STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[s]), r & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + s * YG_STAGE);
      const uint32_t sb = diag ? sa : sa + 2 * YG_A;
      for (int k4 = 0; k4 < 4; ++k4) {
        const int col = kk * 32 + 8 * k4;     // slab boundaries are multiples of 8
        if (col >= klen) break;
        if (col >= a.k1s[slab]) { ++slab; first = true; }
        const uint32_t d = tmem + 128u * (uint32_t)slab;
        const uint64_t ah = tc::sdesc_sw128(sa + 32 * k4, 16, 1024);
        const uint64_t al = tc::sdesc_sw128(sa + YG_A + 32 * k4, 16, 1024);
        const uint64_t bh = tc::sdesc_sw128(sb + 32 * k4, 16, 1024);
        const uint64_t bl = tc::sdesc_sw128(sb + YG_A + 32 * k4, 16, 1024);
        tc::mma_tf32(d, ah, bh, idesc, first ? 0u : 1u);
        tc::mma_tf32(d, ah, bl, idesc, 1);
        tc::mma_tf32(d, al, bh, idesc, 1);
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
      const int T = a.T;
      const int rt = 32 * q + lane, row = mi * TILE + rt;
#pragma unroll 1
      for (int c = 0; c < TILE / 32; ++c) {
        float sum[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) sum[j] = 0.f;
        for (int i = 0; i < a.ndt; ++i) {
          float v[32];
          tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 128u * (uint32_t)i + (uint32_t)(c * 32), v);
#pragma unroll
          for (int j = 0; j < 32; ++j) sum[j] += v[j];
          float* C = a.S + (long long)(u * a.ndt + i) * a.s_us;
          if (row < T) {
            float* cr = C + (long long)row * T + ni * TILE + c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (ni * TILE + c * 32 + j < T) cr[j] = sum[j];
          }
          if (!diag) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = ni * TILE + c * 32 + j;
              if (col < T && row < T) C[(long long)col * T + row] = sum[j];
            }
          }
        }
      }
    }
  }
  if (!ok) atomicOr((int*)(a.ws + (size_t)(u * a.ndt) * a.ub + a.o_status), ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// Yt[u][t][k] = Y[u][h][t][j] and its tf32 low part, the columns k over the
// feature-rank slabs [jb[s], jb[s + 1]) of the truncated ranks, each slab
// head-major: k = H jb[s] + h w_s + (j - jb[s]), w_s = jb[s + 1] - jb[s]
// (every truncated rank's Gram is then the prefix k < H rd).
struct Slabs { int n; int jb[JOLT_MAX_GRID + 1]; };
__global__ void ytrans_kernel(const char* ws, size_t ub, size_t o_Y, size_t o_Yt, int H, int T,
                              int RD, Slabs sl) {
  const int u = blockIdx.y;
  const float* Y = (const float*)(ws + (size_t)u * ub + o_Y);
  float* Yt = (float*)((char*)ws + (size_t)u * ub + o_Yt);
  float* Ytl = Yt + (size_t)T * RD * H;
  const int K = RD * H;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < (long long)T * K;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / K), c = (int)(e % K);
    int s = 0;
    while (s + 1 < sl.n && c >= H * sl.jb[s + 1]) ++s;
    const int j0 = sl.jb[s], w = sl.jb[s + 1] - j0, off = c - H * j0;
    const int h = off / w, j = j0 + off % w;
    const float v = Y[((long long)h * T + t) * RD + j];
    Yt[e] = v;
    Ytl[e] = v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  }
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
                  cudaStream_t st, bool vs_ready) {
  const int* flags = (const int*)(pbase + L.p_flag);
  const long long f_us = (long long)pstride / 4;
  if (!vs_ready) {
    dim3 g2((L.T + 31) / 32, 2, np);
    split_v_kernel<<<g2, dim3(32, 8), 0, st>>>(pbase, pstride, L.p_V, L.p_Vs,
                                               L.p_Vs + (size_t)L.T * 64 * 4, L.T, flags, f_us);
    JOLT_LAUNCH_CHECK();
  }
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
  Slabs sl;
  sl.n = L.ndt;
  sl.jb[0] = 0;
  for (int s = 0; s < L.ndt; ++s) sl.jb[s + 1] = L.rd[s];
  dim3 grid(512, U);
  ytrans_kernel<<<grid, 256, 0, st>>>(ws, L.unit_bytes, L.o_Y, L.o_Yt, L.H, L.T, L.RD, sl);
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
  if (L.ndt <= 4) {
    // one pass per unit: the ranks' Grams as prefix sums of slabs
    static bool attr_pre = false;
    if (!attr_pre) {
      JOLT_CUDA_TRY(cudaFuncSetAttribute(ygram_pre_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
      attr_pre = true;
    }
    dim3 grid(a.nt * (a.nt + 1) / 2, U);
    ygram_pre_tc_kernel<<<grid, TC_THREADS, smem, st>>>(tH, tL, a);
    JOLT_LAUNCH_CHECK();
    return JOLT_OK;
  }
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


}  // namespace jolt
