// Feature-mode projection Y = X U_d[:, :RD] and the Tucker cores on the
// 5th-generation tensor cores, for bf16 X with D = 128.
//
// ["Technical Summary: A JOLT for the KV Cache", Methodology 1: sequential
//  truncation, the token mode is taken on the tensor already projected onto
//  the feature factor; "Joint Tucker-rank and residual-bit KV allocator",
//  Mathematical statement: X~ = G x_2 U_T x_3 U_d.]
//
// X is bf16 (exact in the products); U_d (fp32 eigenvectors) is split into
// three bf16 parts u = u1 + u2 + u3 (each the bf16 rounding of what the
// earlier parts leave, 27 bits together), stacked as the N = 96 columns of
// one kind::f16 product per 128-token tile and head:
//   D[t][32 p + j] = sum_d X[t][d] u_p[d][j]      (exact products, fp32 sums)
//   Y[t][j] = (D[t][64 + j] + D[t][32 + j]) + D[t][j].
// One CTA covers one 128-token tile of HB heads of one unit (HB = 2: two CTAs
// per SM); X tiles and the split factor arrive by TMA (128-byte swizzle).  The epilogue (one thread per
// token row) writes, per head, Y16 = fp16(Y) [H][T][RD] and, when asked, Y in
// fp32 [H][T][RD]; and the token-Gram relayout Yt[t][k] with its tf32 low
// part.  Yt's columns k run over the feature-rank slabs [rd_{s-1}, rd_s) of
// the truncated ranks, each slab head-major: k = H rd_{s-1} + h w_s + (j - rd_{s-1})
// with w_s = rd_s - rd_{s-1}, so that every truncated rank's Gram is a prefix
// k < H rd_s and a CTA's HB heads own one contiguous run per slab.  The rows
// are staged in shared memory and each warp writes its 32 rows' runs with
// consecutive lanes on consecutive columns.
//
// Cores (after the token mode):
//   G(r_d)[h] = U_T(r_d)^T X_h U_d[:, :r_d]   (U_d = I for the whole feature rank)
// as Z = X_h^T [U_T(r_d) of every feature rank], one MN-major kind::f16
// product per head over K = T: X_h (bf16, exact) and each U_T split into three
// bf16 parts (N = 96 per rank, up to 480 TMEM columns).  The whole-feature
// core is Z itself; a truncated core is the small product U_d[:, :r_d]^T Z in
// fp32 on the CUDA cores from shared memory.  Cores and U_T are written in
// fp16 (the storage type) directly.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

#include <string.h>

namespace jolt {

namespace {

constexpr int PJ_ROWS = 128, PJ_THREADS = 128;
constexpr int PJ_XBYTES = PJ_ROWS * 256;   // 128 rows x 128 bf16, two 64-column swizzle atoms
constexpr int PJ_RDP = 32;                 // factor columns per part
constexpr int PJ_N = 3 * PJ_RDP;           // MMA N: three parts

struct ProjArgs {
  int H, T, RD;
  char* ws;
  size_t ub, o_Y, o_Y16, o_Yt, o_status;
  int write_y;
  int nsl;                        // slabs of Yt: feature ranks [jb[s], jb[s + 1])
  int jb[JOLT_MAX_GRID + 1];
};

// Vs3[u][p * 32 + j][d] = bf16 part p of V_d[d][j] (zero for j >= RD), K-major
// rows of the product's B operand; and U_d16[d][j] = fp16(V_d[d][j]).
__global__ void split_ud_kernel(char* ws, size_t ub, size_t o_Vd, size_t o_Vs3, size_t o_Ud16,
                                int D, int RD) {
  const int u = blockIdx.y;
  const float* Vd = (const float*)(ws + (size_t)u * ub + o_Vd);
  __nv_bfloat16* Vs = (__nv_bfloat16*)(ws + (size_t)u * ub + o_Vs3);
  __half* Ud16 = (__half*)(ws + (size_t)u * ub + o_Ud16);
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < PJ_RDP * D; e += gridDim.x * blockDim.x) {
    const int j = e / D, d = e % D;
    const float v = j < RD ? Vd[(size_t)d * D + j] : 0.f;
    const __nv_bfloat16 b1 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(b1);
    const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(b2);
    Vs[(size_t)j * D + d] = b1;
    Vs[(size_t)(PJ_RDP + j) * D + d] = b2;
    Vs[(size_t)(2 * PJ_RDP + j) * D + d] = __float2bfloat16_rn(r2);
    if (j < RD) Ud16[(size_t)d * RD + j] = __float2half_rn(v);
  }
}

template <int HB>
__global__ void __launch_bounds__(PJ_THREADS, HB >= 4 ? 1 : 2)
proj_tc_kernel(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tB,
               ProjArgs a) {
  constexpr int BCHUNK = PJ_N * 128;                  // one 64-column chunk of the B rows
  constexpr uint32_t TCOLS = HB * PJ_N <= 128 ? 128 : (HB * PJ_N <= 256 ? 256 : 512);
  constexpr int SROW = 32 * HB + (HB >= 4 ? 4 : HB);  // staging row stride (floats)
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  unsigned char* sX = base;                           // HB tiles, later the Yt staging
  unsigned char* sB = base + HB * PJ_XBYTES;
  struct Bars { uint64_t tma, mma; uint32_t tmem; };
  Bars* S = (Bars*)(sB + 2 * BCHUNK);
  const int t = threadIdx.x, warp = t >> 5;
  const int tt = blockIdx.x, hg = blockIdx.y, u = blockIdx.z;
  const int t0 = tt * PJ_ROWS, row = t0 + t;
  const bool in = row < a.T;
  const int h0 = hg * HB;
  char* wu = a.ws + (size_t)u * a.ub;

  if (t == 0) {
    tc::mbar_init(tc::smem_u32(&S->tma), 1);
    tc::mbar_init(tc::smem_u32(&S->mma), 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&S->tmem), TCOLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;

  if (t == 0) {
    const uint32_t fb = tc::smem_u32(&S->tma);
    tc::mbar_expect_tx(fb, HB * PJ_XBYTES + 2 * BCHUNK);
#pragma unroll
    for (int i = 0; i < HB; ++i) {
      const int xr = u * a.H + h0 + i;
      tc::tma_load_3d(tc::smem_u32(sX + i * PJ_XBYTES), &tX, 0, t0, xr, fb);
      tc::tma_load_3d(tc::smem_u32(sX + i * PJ_XBYTES + PJ_XBYTES / 2), &tX, 64, t0, xr, fb);
    }
    tc::tma_load_3d(tc::smem_u32(sB), &tB, 0, 0, u, fb);
    tc::tma_load_3d(tc::smem_u32(sB + BCHUNK), &tB, 64, 0, u, fb);
    if (!tc::mbar_wait(fb, 0)) ok = false;
    tc::tc_fence_after();
    if (ok) {
      constexpr uint32_t idesc = tc::idesc_bf16(PJ_ROWS, PJ_N, 0, 0);
#pragma unroll
      for (int i = 0; i < HB; ++i)
#pragma unroll
        for (int kc = 0; kc < 2; ++kc)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = tc::sdesc_sw128(
                tc::smem_u32(sX + i * PJ_XBYTES + kc * (PJ_XBYTES / 2)) + 32 * k, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sB + kc * BCHUNK) + 32 * k, 16, 1024);
            tc::mma_f16(tmem + (uint32_t)(i * PJ_N), ad, bd, idesc, (kc | k) != 0);
          }
    }
    // committed even after a failed load, so that no thread waits in vain
    tc::mma_commit(tc::smem_u32(&S->mma));
  }
  if (!tc::mbar_wait(tc::smem_u32(&S->mma), 0)) ok = false;
  tc::tc_fence_after();

  // ---- epilogue: thread t owns token row t of the tile (TMEM lane t)
  const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
  float* stg = reinterpret_cast<float*>(sX) + (size_t)t * SROW;   // this row's staging
  const int RD = a.RD;
#pragma unroll 1
  for (int i = 0; i < HB; ++i) {
    float c0[32], c1[32], c2[32];
    tc::tmem_ld32(tl + (uint32_t)(i * PJ_N), c0);
    tc::tmem_ld32(tl + (uint32_t)(i * PJ_N + PJ_RDP), c1);
    tc::tmem_ld32(tl + (uint32_t)(i * PJ_N + 2 * PJ_RDP), c2);
    float y[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      y[j] = (c2[j] + c1[j]) + c0[j];
      if (!ok) y[j] = __int_as_float(0x7fc00000);
    }
    const size_t r = ((size_t)(h0 + i) * a.T + (in ? row : 0)) * RD;
    if (in) {
      __half* y16 = (__half*)(wu + a.o_Y16) + r;
      float* y32 = (float*)(wu + a.o_Y) + r;
      if (RD == 32) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 v;
          __half2* hv = reinterpret_cast<__half2*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) hv[e] = __floats2half2_rn(y[j + 2 * e], y[j + 2 * e + 1]);
          *reinterpret_cast<uint4*>(y16 + j) = v;
        }
        if (a.write_y) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(y32 + j) = make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < RD) {
            y16[j] = __float2half_rn(y[j]);
            if (a.write_y) y32[j] = y[j];
          }
      }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) stg[j * HB + i] = y[j];
  }
  // ---- Yt and its tf32 low part: this CTA's HB heads own, per slab s, the
  // run of HB w_s columns at H jb[s] + h0 w_s of each row; element e of the
  // concatenated runs is (head h0 + i, rank j).  Lane l writes elements l,
  // l + 32, ... of each of its warp's rows (staged by that warp's threads).
  if (a.o_Yt) {
    __syncwarp();
    const size_t K = (size_t)RD * a.H;
    float* ytb = (float*)(wu + a.o_Yt);
    const int lane = t & 31;
    constexpr int EMAX = (HB * PJ_RDP + 31) / 32;
    int col[EMAX], src[EMAX];
#pragma unroll
    for (int c = 0; c < EMAX; ++c) {
      const int e = lane + 32 * c;
      col[c] = -1;
      src[c] = 0;
      int s = 0;
      while (s < a.nsl && e >= HB * a.jb[s + 1]) ++s;
      if (s < a.nsl) {
        const int j0 = a.jb[s], w = a.jb[s + 1] - j0, off = e - HB * j0;
        const int i = off / w, j = j0 + off % w;
        col[c] = a.H * j0 + (h0 + i) * w + (j - j0);
        src[c] = j * HB + i;
      }
    }
#pragma unroll 2
    for (int r = 0; r < 32; ++r) {
      const int rr = warp * 32 + r, grow = t0 + rr;
      if (grow >= a.T) break;
      const float* sr = reinterpret_cast<const float*>(sX) + (size_t)rr * SROW;
      float* yt = ytb + (size_t)grow * K;
#pragma unroll
      for (int c = 0; c < EMAX; ++c) {
        if (col[c] < 0) continue;
        const float v = sr[src[c]];
        yt[col[c]] = v;
        yt[(size_t)a.T * K + col[c]] = v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
      }
    }
  }
  if (!ok) atomicOr((int*)(wu + a.o_status), ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
}


// ---------------------------------------------------------------- cores
constexpr int CT_THREADS = 192;             // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
constexpr int CT_KT = 64;                   // tokens per stage
constexpr int CT_XST = CT_KT * 256;         // X stage: 64 tokens x 128 features (two atoms)
constexpr int CT_NATOM = CT_KT * 128;       // one 64-column atom of the U_T parts
constexpr int CT_NMAX = 512;                // columns of the U_T part rows
constexpr int CT_STAGES = 2;
constexpr int CT_ZROW = 36;                 // padded row (floats) of the staged Z and U_d

struct CoresArgs {
  int H, T, RT, nd, ntot, natoms;
  int rd[JOLT_MAX_GRID];
  int full_id;                  // index of the whole feature rank, or -1
  char* ws;
  size_t ub, o_Vd, o_G16, o_status, o_cap;
};

// Sum over the warp's lanes of v[j] for each j, lane j receiving the sum of
// index j (recursive halving: 31 exchanges instead of 32 x 5).
__device__ __forceinline__ double warp_reduce_scatter32(double (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const double send = up ? v[k] : v[k + o];
      const double keep = up ? v[k + o] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// Ub3[u][t][96 id + 32 p + j] = bf16 part p of U_T(id)[t][j] (zero for
// j >= RT and for the columns past nd * 96); U_T16[id][t][j] = fp16(U_T).
__global__ void split_ut_kernel(char* ws, size_t ub, size_t o_UT32, size_t o_UT16, size_t o_Ub3,
                                int T, int RT, int nd) {
  const int u = blockIdx.y;
  const float* U32 = (const float*)(ws + (size_t)u * ub + o_UT32);
  __half* U16 = (__half*)(ws + (size_t)u * ub + o_UT16);
  __nv_bfloat16* Ub = (__nv_bfloat16*)(ws + (size_t)u * ub + o_Ub3);
  const long long n = (long long)T * CT_NMAX;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / CT_NMAX), c = (int)(e % CT_NMAX);
    const int id = c / 96, p = (c % 96) / 32, j = c % 32;
    float v = 0.f;
    if (id < nd && j < RT) v = U32[((size_t)id * T + t) * RT + j];
    const float r1 = v - __bfloat162float(__float2bfloat16_rn(v));
    const float r2 = r1 - __bfloat162float(__float2bfloat16_rn(r1));
    const float part = p == 0 ? v : (p == 1 ? r1 : r2);
    Ub[e] = __float2bfloat16_rn(part);
    if (p == 0 && id < nd && j < RT) U16[((size_t)id * T + t) * RT + j] = __float2half_rn(v);
  }
}

__global__ void __launch_bounds__(CT_THREADS, 1)
cores_tc_kernel(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tU,
                CoresArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const int stage_bytes = CT_XST + a.natoms * CT_NATOM;
  // the stages, later the epilogue's Z and U_d staging; the barriers after both
  const int epi_bytes = (a.nd + 1) * 128 * CT_ZROW * 4;
  const int region = CT_STAGES * stage_bytes > epi_bytes ? CT_STAGES * stage_bytes : epi_bytes;
  struct Bars {
    uint64_t full[CT_STAGES], empty[CT_STAGES], accum;
    double cap[(CT_NMAX / 96) * 32];   // per-block captured energy of the truncated ranks
    uint32_t tmem;
  };
  Bars* S = (Bars*)(base + region);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int h = blockIdx.x, u = blockIdx.y;
  const int nk = (a.T + CT_KT - 1) / CT_KT;
  char* wu = a.ws + (size_t)u * a.ub;
  if (threadIdx.x == 0) {
    for (int s = 0; s < CT_STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&S->accum), 1);
    tc::fence_barrier_init();
  }
  for (int i = threadIdx.x; i < (CT_NMAX / 96) * 32; i += CT_THREADS) S->cap[i] = 0.0;
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&S->tmem), 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;
  if (warp == 0 && lane == 0) {
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % CT_STAGES, r = kk / CT_STAGES;
      if (r > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[s]), (r - 1) & 1)) { ok = false; break; }
      const uint32_t fb = tc::smem_u32(&S->full[s]);
      tc::mbar_expect_tx(fb, stage_bytes);
      const uint32_t sa = tc::smem_u32(base + s * stage_bytes);
      const int xr = u * a.H + h;
      tc::tma_load_3d(sa, &tX, 0, kk * CT_KT, xr, fb);
      tc::tma_load_3d(sa + CT_XST / 2, &tX, 64, kk * CT_KT, xr, fb);
      for (int at = 0; at < a.natoms; ++at)
        tc::tma_load_3d(sa + CT_XST + at * CT_NATOM, &tU, 64 * at, kk * CT_KT, u, fb);
    }
  } else if (warp == 1 && lane == 0) {
    const int n1 = a.ntot < 256 ? a.ntot : 256, n2 = a.ntot - n1;
    const uint32_t id1 = tc::idesc_bf16(128, n1, 1, 1);
    const uint32_t id2 = tc::idesc_bf16(128, n2 > 0 ? n2 : 16, 1, 1);
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % CT_STAGES, r = kk / CT_STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[s]), r & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + s * stage_bytes);
      const uint32_t sb = sa + CT_XST;
#pragma unroll
      for (int k4 = 0; k4 < CT_KT / 16; ++k4) {
        const uint64_t ad = tc::sdesc_sw128(sa + 2048 * k4, CT_XST / 2, 1024);
        const uint64_t b1 = tc::sdesc_sw128(sb + 2048 * k4, CT_NATOM, 1024);
        tc::mma_f16(tmem, ad, b1, id1, (kk | k4) != 0);
        if (n2 > 0) {
          const uint64_t b2 = tc::sdesc_sw128(sb + 4 * CT_NATOM + 2048 * k4, CT_NATOM, 1024);
          tc::mma_f16(tmem + 256, ad, b2, id2, (kk | k4) != 0);
        }
      }
      tc::mma_commit(tc::smem_u32(&S->empty[s]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  }
  // ---- epilogue: thread e (warps 2-5) owns feature row d = TMEM lane
  const int e = threadIdx.x - 64;
  float* Zs = reinterpret_cast<float*>(base);                      // [truncated id][d][36]
  float* Vs = Zs + (size_t)a.nd * 128 * CT_ZROW;                    // [d][36]
  const int RT = a.RT;
  if (warp >= 2) {
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) ok = false;
    tc::tc_fence_after();
    const int q = warp & 3, d = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    int it = 0;
    for (int id = 0; id < a.nd; ++id) {
      float c0[32], c1[32], c2[32];
      tc::tmem_ld32(tl + (uint32_t)(96 * id), c0);
      tc::tmem_ld32(tl + (uint32_t)(96 * id + 32), c1);
      tc::tmem_ld32(tl + (uint32_t)(96 * id + 64), c2);
      float z[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = ok ? (c2[j] + c1[j]) + c0[j] : __int_as_float(0x7fc00000);
      if (id == a.full_id) {
        // G(D)[h][j][d] = Z[d][j]
        __half* G = (__half*)(wu + a.o_G16) + (size_t)id * a.H * RT * 128 + (size_t)h * RT * 128;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < RT) G[(size_t)j * 128 + d] = __float2half_rn(z[j]);
        double sq[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) sq[j] = (double)z[j] * (double)z[j];
        const double cj = warp_reduce_scatter32(sq, lane);
        if (lane < RT) atomicAdd((double*)(wu + a.o_cap) + id * RT + lane, cj);
      } else {
        float* zr = Zs + ((size_t)it * 128 + d) * CT_ZROW;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(zr + j) = make_float4(z[j], z[j + 1], z[j + 2], z[j + 3]);
        ++it;
      }
    }
    // U_d[d][:32] (unrounded, fp32)
    const float* Vd = (const float*)(wu + a.o_Vd) + (size_t)d * 128;
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4*>(Vs + (size_t)d * CT_ZROW + j) = *reinterpret_cast<const float4*>(Vd + j);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
  // ---- truncated cores G(r_d)[h][jt][jd] = sum_d Z[d][jt] U_d[d][jd], one
  // 4 x 4 block per thread and step
  if (warp >= 2) {
    int tot = 0;
    for (int id = 0; id < a.nd; ++id)
      if (id != a.full_id) tot += (RT / 4) * (a.rd[id] / 4);
    for (int tile = e; tile < tot; tile += 128) {
      int rem = tile, it = 0, id = 0;
      for (id = 0; id < a.nd; ++id) {
        if (id == a.full_id) continue;
        const int n = (RT / 4) * (a.rd[id] / 4);
        if (rem < n) break;
        rem -= n;
        ++it;
      }
      const int rd = a.rd[id];
      const int jt0 = (rem / (rd / 4)) * 4, jd0 = (rem % (rd / 4)) * 4;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
      const float* zb = Zs + (size_t)it * 128 * CT_ZROW + jt0;
      const float* vb = Vs + jd0;
#pragma unroll 4
      for (int d = 0; d < 128; ++d) {
        const float4 zv = *reinterpret_cast<const float4*>(zb + (size_t)d * CT_ZROW);
        const float4 vv = *reinterpret_cast<const float4*>(vb + (size_t)d * CT_ZROW);
        const float zz[4] = {zv.x, zv.y, zv.z, zv.w}, ww[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(zz[i], ww[j], acc[i][j]);
      }
      __half* G = (__half*)(wu + a.o_G16) + (size_t)id * a.H * RT * 128 + (size_t)h * RT * rd;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        double c = 0.0;
#pragma unroll
        for (int j = 0; j < 4; ++j) c += (double)acc[i][j] * (double)acc[i][j];
        atomicAdd(&S->cap[id * 32 + jt0 + i], c);
        __half2 p0 = __floats2half2_rn(acc[i][0], acc[i][1]);
        __half2 p1 = __floats2half2_rn(acc[i][2], acc[i][3]);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t*>(&p0);
        v.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(G + (size_t)(jt0 + i) * rd + jd0) = v;
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int k = e; k < a.nd * 32; k += 128) {
      const int id = k / 32, j = k % 32;
      if (id != a.full_id && j < RT)
        atomicAdd((double*)(wu + a.o_cap) + id * RT + j, S->cap[k]);
    }
  }
  if (!ok) atomicOr((int*)(wu + a.o_status), ST_TIMEOUT);
}

size_t cores_smem(int natoms, int nd) {
  const size_t stages = (size_t)CT_STAGES * (CT_XST + natoms * CT_NATOM);
  const size_t epi = (size_t)(nd + 1) * 128 * CT_ZROW * 4;
  return 1024 + (stages > epi ? stages : epi) + 64 + (CT_NMAX / 96) * 32 * 8 + 64;
}

template <int HB>
size_t proj_smem() {
  return 1024 + (size_t)HB * PJ_XBYTES + 2 * PJ_N * 128 + 64;
}

template <int HB>
jolt_status launch_proj(dim3 grid, const CUtensorMap& tX, const CUtensorMap& tB,
                        const ProjArgs& a, cudaStream_t st) {
  const size_t smem = proj_smem<HB>();
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(proj_tc_kernel<HB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  proj_tc_kernel<HB><<<grid, PJ_THREADS, smem, st>>>(tX, tB, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace

bool proj_tc_supported(const Layout& L) {
  return L.dtype == JOLT_BF16 && L.D == 128 && L.RD > 0 && L.RD <= PJ_RDP && L.o_Vs3 != 0 &&
         tc::encode_fn() != nullptr;
}

jolt_status proj_tc(const Layout& L, int U, const void* X, char* ws, bool write_y,
                    cudaStream_t st) {
  if (!proj_tc_supported(L)) return JOLT_ERR_INVALID;
  split_ud_kernel<<<dim3(16, U), 256, 0, st>>>(ws, L.unit_bytes, L.o_Vd, L.o_Vs3, L.o_Ud16, L.D,
                                               L.RD);
  JOLT_LAUNCH_CHECK();
  CUtensorMap tX, tB;
  const cuuint64_t dX[3] = {128, (cuuint64_t)L.T, (cuuint64_t)U * L.H};
  const cuuint64_t sX[2] = {256, (cuuint64_t)L.T * 256};
  const cuuint32_t bX[3] = {64, PJ_ROWS, 1};
  if (!tc::make_map(&tX, X, 3, dX, sX, bX)) return JOLT_ERR_CUDA;
  const cuuint64_t dB[3] = {128, PJ_N, (cuuint64_t)U};
  const cuuint64_t sB[2] = {256, (cuuint64_t)L.unit_bytes};
  const cuuint32_t bB[3] = {64, PJ_N, 1};
  if (!tc::make_map(&tB, ws + L.o_Vs3, 3, dB, sB, bB)) return JOLT_ERR_CUDA;
  ProjArgs a;
  a.H = L.H; a.T = L.T; a.RD = L.RD;
  a.ws = ws; a.ub = L.unit_bytes;
  a.o_Y = L.o_Y; a.o_Y16 = L.o_Y16; a.o_Yt = L.o_Yt; a.o_status = L.o_status;
  a.write_y = write_y ? 1 : 0;
  a.nsl = L.ndt;
  a.jb[0] = 0;
  for (int s = 0; s < L.ndt; ++s) a.jb[s + 1] = L.rd[s];
  // two heads per CTA: two CTAs per SM (TMEM 256 columns, 88 KB of shared
  // memory each) overlap one CTA's loads with the other's epilogue
  const int tiles = (L.T + PJ_ROWS - 1) / PJ_ROWS;
  if (L.H % 2 == 0) return launch_proj<2>(dim3(tiles, L.H / 2, U), tX, tB, a, st);
  return launch_proj<1>(dim3(tiles, L.H, U), tX, tB, a, st);
}


bool cores_tc_supported(const Layout& L) {
  if (!(L.dtype == JOLT_BF16 && L.D == 128 && L.RT > 0 && L.RT <= 32 && L.RT % 4 == 0 &&
        L.nd * 96 <= CT_NMAX && L.o_Ub3 != 0 && tc::encode_fn() != nullptr))
    return false;
  for (int i = 0; i < L.nd; ++i)
    if (L.rd[i] != L.D && (L.rd[i] % 4 || L.rd[i] > 32)) return false;
  return true;
}

jolt_status cores_tc(const Layout& L, int U, const void* X, char* ws, cudaStream_t st) {
  if (!cores_tc_supported(L)) return JOLT_ERR_INVALID;
  split_ut_kernel<<<dim3(256, U), 256, 0, st>>>(ws, L.unit_bytes, L.o_UT32, L.o_UT16, L.o_Ub3,
                                                L.T, L.RT, L.nd);
  JOLT_LAUNCH_CHECK();
  CoresArgs a;
  memset(&a, 0, sizeof(a));
  a.H = L.H; a.T = L.T; a.RT = L.RT; a.nd = L.nd;
  a.ntot = 96 * L.nd;
  a.natoms = (a.ntot + 63) / 64;
  a.full_id = -1;
  for (int i = 0; i < L.nd; ++i) {
    a.rd[i] = L.rd[i];
    if (L.rd[i] == L.D) a.full_id = i;
  }
  a.ws = ws; a.ub = L.unit_bytes; a.o_Vd = L.o_Vd; a.o_G16 = L.o_G16; a.o_status = L.o_status;
  a.o_cap = L.o_cap;
  CUtensorMap tX, tU;
  const cuuint64_t dX[3] = {128, (cuuint64_t)L.T, (cuuint64_t)U * L.H};
  const cuuint64_t sX[2] = {256, (cuuint64_t)L.T * 256};
  const cuuint32_t bX[3] = {64, CT_KT, 1};
  if (!tc::make_map(&tX, X, 3, dX, sX, bX)) return JOLT_ERR_CUDA;
  const cuuint64_t dU[3] = {CT_NMAX, (cuuint64_t)L.T, (cuuint64_t)U};
  const cuuint64_t sU[2] = {CT_NMAX * 2, (cuuint64_t)L.unit_bytes};
  const cuuint32_t bU[3] = {64, CT_KT, 1};
  if (!tc::make_map(&tU, ws + L.o_Ub3, 3, dU, sU, bU)) return JOLT_ERR_CUDA;
  const size_t smem = cores_smem(a.natoms, a.nd);
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(cores_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)cores_smem(CT_NMAX / 64, CT_NMAX / 96)));
    attr = true;
  }
  cores_tc_kernel<<<dim3(L.H, U), CT_THREADS, smem, st>>>(tX, tU, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace jolt
