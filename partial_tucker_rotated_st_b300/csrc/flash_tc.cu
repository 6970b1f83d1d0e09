// FlashJoLT's randomized token-mode solve with every product over X on the
// 5th-generation tensor cores (bf16 X, D = 128).
//
// ["Technical Summary: A JOLT for the KV Cache", Methodology 4 (FlashJoLT:
//  a randomized range finder with p = 8 oversampling columns and q = 2 power
//  steps for the token mode); Methodology 1 (the token mode of the tensor
//  projected onto the feature factor, Y = X x_3 U_d^T).]
//
// For a feature rank r_d the token-mode matrix is A = [A_1 .. A_H] with
// A_h = X_h V (V = U_d[:, :r_d], or the identity for the whole feature rank).
// Every product of the range finder is taken against X itself, with the
// small factor moved to the other side:
//   Z = A Omega           = sum_h X_h (V Omega_h)
//   P_h = A_h^T Q         = V^T (X_h^T Q)
//   Z = A (A^T Q)         = sum_h X_h (V V^T X_h^T Q)
//   Rayleigh-Ritz matrix  = sum_h P_h^T P_h
// so each step is one pass over the bf16 X (exact in the products) against
// fp32 matrices split into three bf16 parts (27 bits), with fp32 accumulation:
//   * the "Z pass" (flash_z_kernel): one CTA per 128-token tile, K = H x D
//     over every head, N = 3 parts x the ranks' sketch columns;
//   * the "C pass" (flash_c_kernel): C_h = X_h^T Q for every head, one CTA per
//     head, K = T (the cores kernel's MN-major product);
// and the ranks of one call move in lockstep, their columns side by side in
// one product.  The small products (V Omega_h, V^T C_h, V P_h, the Gram of
// the P_h) run on the CUDA cores; the orthonormalisations (CholeskyQR2) and
// the Rayleigh-Ritz eigen-solve are the library's usual ones.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

#include <string.h>

namespace jolt {

namespace {

constexpr int FL_THREADS = 192;     // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
constexpr int FL_WMAX = 160;        // sketch columns of the ranks of one call
constexpr int FL_BROWS = 512;       // rows of one head's B block (Z pass)
constexpr int FL_STAGES = 2;
// Z pass: stage = one 64-feature atom of the X tile (128 tokens) and of B
constexpr int FZ_XATOM = 128 * 128;         // bytes
constexpr int FZ_BATOM = 512 * 128;
constexpr int FZ_STAGE = FZ_XATOM + FZ_BATOM;
// C pass: stage = 64 tokens of X_h (two 64-feature atoms) and of the Q parts
constexpr int FC_KT = 64;
constexpr int FC_XST = FC_KT * 256;
constexpr int FC_NATOM = FC_KT * 128;
constexpr int FC_QCOLS = 512;

struct FlashSet {
  int nr, ell, W;              // ranks, sketch width, part width (multiple of 32, >= nr ell)
  int rdv[4];                  // feature rank (D = the whole feature rank: V = I)
  int pidx0[4], pmul;          // problem of (unit u, rank r) = u * pmul + pidx0[r]
  int H, T, D;
  int hs;                      // head groups of the Rayleigh-Ritz partial Grams (divides H)
  char* ws;                    // units
  size_t ub, o_Vd, o_Bx, o_Qs, o_C, o_status;
  char* pbase;                 // problems
  size_t pb, p_Z, p_V, p_Hm, p_status;
};

__device__ __forceinline__ char* prob(const FlashSet& s, int u, int r) {
  return s.pbase + (size_t)(u * s.pmul + s.pidx0[r]) * s.pb;
}

// bf16 parts of v: v = p0 + p1 + p2 up to 2^-27 |v|
__device__ __forceinline__ void split3(float v, __nv_bfloat16 (&p)[3]) {
  p[0] = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(p[0]);
  p[1] = __float2bfloat16_rn(r1);
  p[2] = __float2bfloat16_rn(r1 - __bfloat162float(p[1]));
}

// Bx[u][h][p W + r ell + k][d] = part p of B_r[d][k] (K-major rows of the Z
// pass), where B_r = V_r Omega_h[:rdv] (mode 0) or B_r = V_r V_r^T C_h,r
// (mode 1; the whole feature rank: B = Omega_h or C_h,r).  One CTA per (head,
// unit); Omega_h is [D][ell] rows of the unit's sketch, C_h is
// [D][nr ell] at o_C.
__global__ void __launch_bounds__(256)
flash_b_kernel(FlashSet s, const float* __restrict__ sketch, int mode) {
  const int h = blockIdx.x, u = blockIdx.y, t = threadIdx.x;
  const int D = s.D, ell = s.ell, NC = s.nr * ell;
  extern __shared__ float fb_sm[];
  float* In = fb_sm;                    // [D][NC]: Omega_h (every rank) or C_h
  float* Pm = In + D * NC;              // [32][NC]: V_r^T C_h,r of the truncated ranks
  float* Vs = Pm + 32 * NC;             // [32][D]: U_d[:, :32] transposed
  const char* wu = s.ws + (size_t)u * s.ub;
  const float* Vg = (const float*)(wu + s.o_Vd);
  for (int e = t; e < D * 32; e += 256) Vs[(e & 31) * D + (e >> 5)] = Vg[(size_t)(e >> 5) * D + (e & 31)];
  for (int e = t; e < D * NC; e += 256) {
    const int d = e / NC, c = e % NC;
    In[e] = mode == 0 ? sketch[(((size_t)u * s.H + h) * D + d) * ell + c % ell]
                      : ((const float*)(wu + s.o_C))[(((size_t)h * D) + d) * NC + c];
  }
  __syncthreads();
  // mode 1: Pm[j][r ell + k] = sum_d V[d][j] C[d][r ell + k], j < rdv_r
  if (mode == 1) {
    for (int e = t; e < 32 * NC; e += 256) {
      const int j = e / NC, c = e % NC, r = c / ell;
      float a = 0.f;
      if (s.rdv[r] < D && j < s.rdv[r])
        for (int d = 0; d < D; ++d) a = fmaf(Vs[j * D + d], In[d * NC + c], a);
      Pm[e] = a;
    }
    __syncthreads();
  }
  __nv_bfloat16* Bx = (__nv_bfloat16*)(s.ws + (size_t)u * s.ub + s.o_Bx) + (size_t)h * FL_BROWS * D;
  for (int e = t; e < D * s.W; e += 256) {
    const int d = e % D, c = e / D;           // consecutive threads: consecutive d
    float v = 0.f;
    if (c < NC) {
      const int r = c / ell, k = c % ell, rd = s.rdv[r];
      if (rd >= D) {
        v = In[d * NC + c];                   // V = I
      } else if (mode == 0) {
        for (int j = 0; j < rd; ++j) v = fmaf(Vs[j * D + d], In[j * NC + c], v);
      } else {
        for (int j = 0; j < rd; ++j) v = fmaf(Vs[j * D + d], Pm[j * NC + r * ell + k], v);
      }
    }
    __nv_bfloat16 p[3];
    split3(v, p);
#pragma unroll
    for (int q = 0; q < 3; ++q) Bx[(size_t)(q * s.W + c) * D + d] = p[q];
  }
}

// Qs[u][t][p W + r ell + k] = part p of Q_r[t][k] (the problem's p_V, T x ell).
__global__ void flash_qsplit_kernel(FlashSet s) {
  const int u = blockIdx.y;
  __nv_bfloat16* Qs = (__nv_bfloat16*)(s.ws + (size_t)u * s.ub + s.o_Qs);
  const long long n = (long long)s.T * s.W;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / s.W), c = (int)(e % s.W);
    float v = 0.f;
    if (c < s.nr * s.ell) {
      const int r = c / s.ell, k = c % s.ell;
      v = ((const float*)(prob(s, u, r) + s.p_V))[(size_t)t * s.ell + k];
    }
    __nv_bfloat16 p[3];
    split3(v, p);
#pragma unroll
    for (int q = 0; q < 3; ++q) Qs[(size_t)t * FC_QCOLS + q * s.W + c] = p[q];
  }
}

// Z pass: Z_r[t][k] = sum_h sum_d X_h[t][d] B_r,h[d][k] for one 128-token tile
// of one unit, the ranks side by side (columns p W + r ell + k of the
// product, the three parts summed in the epilogue) into each problem's p_Z.
__global__ void __launch_bounds__(FL_THREADS, 1)
flash_z_kernel(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tB,
               FlashSet s) {
  extern __shared__ __align__(1024) unsigned char fz_raw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)fz_raw + 1023) & ~(uintptr_t)1023);
  struct Bars { uint64_t full[FL_STAGES], empty[FL_STAGES], accum; uint32_t tmem; };
  Bars* S = (Bars*)(base + FL_STAGES * FZ_STAGE);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int tt = blockIdx.x, u = blockIdx.y;
  const int ntot = 3 * s.W;
  const int nld = ntot > 256 ? 2 : 1;          // B loads of 256 rows per atom
  const int stage_tx = FZ_XATOM + nld * 256 * 128;
  const int nk = 2 * s.H;                      // stages: (head, feature atom)
  if (threadIdx.x == 0) {
    for (int i = 0; i < FL_STAGES; ++i) {
      tc::mbar_init(tc::smem_u32(&S->full[i]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[i]), 1);
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
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int st = kk % FL_STAGES, rr = kk / FL_STAGES;
      if (rr > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[st]), (rr - 1) & 1)) { ok = false; break; }
      const uint32_t fb = tc::smem_u32(&S->full[st]);
      tc::mbar_expect_tx(fb, stage_tx);
      const uint32_t sa = tc::smem_u32(base + st * FZ_STAGE);
      const int h = kk >> 1, at = kk & 1;
      tc::tma_load_3d(sa, &tX, 64 * at, tt * 128, u * s.H + h, fb);
      for (int l = 0; l < nld; ++l)
        tc::tma_load_4d(sa + FZ_XATOM + l * 256 * 128, &tB, 64 * at, 256 * l, h, u, fb);
    }
  } else if (warp == 1 && lane == 0) {
    const int n1 = ntot < 256 ? ntot : 256, n2 = ntot - n1;
    const uint32_t id1 = tc::idesc_bf16(128, n1, 0, 0);
    const uint32_t id2 = tc::idesc_bf16(128, n2 > 0 ? n2 : 16, 0, 0);
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int st = kk % FL_STAGES, rr = kk / FL_STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[st]), rr & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + st * FZ_STAGE);
      const uint32_t sb = sa + FZ_XATOM;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = tc::sdesc_sw128(sa + 32 * k, 16, 1024);
        tc::mma_f16(tmem, ad, tc::sdesc_sw128(sb + 32 * k, 16, 1024), id1, (kk | k) != 0);
        if (n2 > 0)
          tc::mma_f16(tmem + 256, ad, tc::sdesc_sw128(sb + 256 * 128 + 32 * k, 16, 1024), id2,
                      (kk | k) != 0);
      }
      tc::mma_commit(tc::smem_u32(&S->empty[st]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  }
  if (warp >= 2) {
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) ok = false;
    tc::tc_fence_after();
    const int q = warp & 3, row = 32 * q + lane;
    const int t = tt * 128 + row;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const int NC = s.nr * s.ell;
    for (int k = 0; k < s.W / 32; ++k) {
      float c0[32], c1[32], c2[32];
      tc::tmem_ld32(tl + (uint32_t)(32 * k), c0);
      tc::tmem_ld32(tl + (uint32_t)(s.W + 32 * k), c1);
      tc::tmem_ld32(tl + (uint32_t)(2 * s.W + 32 * k), c2);
      if (t < s.T) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const int c = 32 * k + i;
          if (c >= NC) break;
          const int r = c / s.ell, kc = c % s.ell;   // ell is a multiple of 4
          float4 v;
          v.x = ok ? (c2[i] + c1[i]) + c0[i] : __int_as_float(0x7fc00000);
          v.y = ok ? (c2[i + 1] + c1[i + 1]) + c0[i + 1] : __int_as_float(0x7fc00000);
          v.z = ok ? (c2[i + 2] + c1[i + 2]) + c0[i + 2] : __int_as_float(0x7fc00000);
          v.w = ok ? (c2[i + 3] + c1[i + 3]) + c0[i + 3] : __int_as_float(0x7fc00000);
          *reinterpret_cast<float4*>((float*)(prob(s, u, r) + s.p_Z) + (size_t)t * s.ell + kc) = v;
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
  if (!ok) atomicOr((int*)(s.ws + (size_t)u * s.ub + s.o_status), ST_TIMEOUT);
}

// C pass: C[u][h][d][r ell + k] = sum_t X_h[t][d] Q_r[t][k] (MN-major A = X_h^T
// and B = the Q parts, K = T), one CTA per (head, unit).
__global__ void __launch_bounds__(FL_THREADS, 1)
flash_c_kernel(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tQ,
               FlashSet s) {
  extern __shared__ __align__(1024) unsigned char fc_raw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)fc_raw + 1023) & ~(uintptr_t)1023);
  const int ntot = 3 * s.W;
  const int natoms = (ntot + 63) / 64;
  const int stage_bytes = FC_XST + natoms * FC_NATOM;
  struct Bars { uint64_t full[FL_STAGES], empty[FL_STAGES], accum; uint32_t tmem; };
  Bars* S = (Bars*)(base + FL_STAGES * (FC_XST + 8 * FC_NATOM));
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int h = blockIdx.x, u = blockIdx.y;
  const int nk = (s.T + FC_KT - 1) / FC_KT;
  if (threadIdx.x == 0) {
    for (int i = 0; i < FL_STAGES; ++i) {
      tc::mbar_init(tc::smem_u32(&S->full[i]), 1);
      tc::mbar_init(tc::smem_u32(&S->empty[i]), 1);
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
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int st = kk % FL_STAGES, rr = kk / FL_STAGES;
      if (rr > 0 && !tc::mbar_wait(tc::smem_u32(&S->empty[st]), (rr - 1) & 1)) { ok = false; break; }
      const uint32_t fb = tc::smem_u32(&S->full[st]);
      tc::mbar_expect_tx(fb, stage_bytes);
      const uint32_t sa = tc::smem_u32(base + st * stage_bytes);
      const int xr = u * s.H + h;
      tc::tma_load_3d(sa, &tX, 0, kk * FC_KT, xr, fb);
      tc::tma_load_3d(sa + FC_XST / 2, &tX, 64, kk * FC_KT, xr, fb);
      for (int at = 0; at < natoms; ++at)
        tc::tma_load_3d(sa + FC_XST + at * FC_NATOM, &tQ, 64 * at, kk * FC_KT, u, fb);
    }
  } else if (warp == 1 && lane == 0) {
    const int n1 = ntot < 256 ? ntot : 256, n2 = ntot - n1;
    const uint32_t id1 = tc::idesc_bf16(128, n1, 1, 1);
    const uint32_t id2 = tc::idesc_bf16(128, n2 > 0 ? n2 : 16, 1, 1);
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int st = kk % FL_STAGES, rr = kk / FL_STAGES;
      if (!tc::mbar_wait(tc::smem_u32(&S->full[st]), rr & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(base + st * stage_bytes);
      const uint32_t sb = sa + FC_XST;
#pragma unroll
      for (int k4 = 0; k4 < FC_KT / 16; ++k4) {
        const uint64_t ad = tc::sdesc_sw128(sa + 2048 * k4, FC_XST / 2, 1024);
        tc::mma_f16(tmem, ad, tc::sdesc_sw128(sb + 2048 * k4, FC_NATOM, 1024), id1, (kk | k4) != 0);
        if (n2 > 0)
          tc::mma_f16(tmem + 256, ad, tc::sdesc_sw128(sb + 4 * FC_NATOM + 2048 * k4, FC_NATOM, 1024),
                      id2, (kk | k4) != 0);
      }
      tc::mma_commit(tc::smem_u32(&S->empty[st]));
    }
    tc::mma_commit(tc::smem_u32(&S->accum));
  }
  if (warp >= 2) {
    if (!tc::mbar_wait(tc::smem_u32(&S->accum), 0)) ok = false;
    tc::tc_fence_after();
    const int q = warp & 3, d = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    const int NC = s.nr * s.ell;
    float* C = (float*)(s.ws + (size_t)u * s.ub + s.o_C) + ((size_t)h * s.D + d) * NC;
    for (int k = 0; k < s.W / 32; ++k) {
      float c0[32], c1[32], c2[32];
      tc::tmem_ld32(tl + (uint32_t)(32 * k), c0);
      tc::tmem_ld32(tl + (uint32_t)(s.W + 32 * k), c1);
      tc::tmem_ld32(tl + (uint32_t)(2 * s.W + 32 * k), c2);
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const int c = 32 * k + i;
        if (c >= NC) break;
        float4 v;
        v.x = ok ? (c2[i] + c1[i]) + c0[i] : __int_as_float(0x7fc00000);
        v.y = ok ? (c2[i + 1] + c1[i + 1]) + c0[i + 1] : __int_as_float(0x7fc00000);
        v.z = ok ? (c2[i + 2] + c1[i + 2]) + c0[i + 2] : __int_as_float(0x7fc00000);
        v.w = ok ? (c2[i + 3] + c1[i + 3]) + c0[i + 3] : __int_as_float(0x7fc00000);
        *reinterpret_cast<float4*>(C + c) = v;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
  if (!ok) atomicOr((int*)(s.ws + (size_t)u * s.ub + s.o_status), ST_TIMEOUT);
}

// Rayleigh-Ritz matrix of problem (u, r): Hm = sum_h P_h^T P_h with P_h =
// V_r^T C_h,r (rdv x ell; C_h,r itself for the whole feature rank), one
// partial per group of H / hs heads into the problem's p_Hm + g ell^2 (the
// eigen-solve sums the partials).  One CTA per (head group, rank, unit).
__global__ void __launch_bounds__(256)
flash_rr_kernel(FlashSet s) {
  const int g = blockIdx.x, r = blockIdx.y, u = blockIdx.z, t = threadIdx.x;
  const int D = s.D, ell = s.ell, NC = s.nr * ell, rd = s.rdv[r];
  const int rows = rd < D ? rd : D;
  const int hper = s.H / s.hs;
  extern __shared__ float fr_sm[];
  float* Ch = fr_sm;                 // [D][ell]
  float* Ph = Ch + D * ell;          // [32][ell]
  float* Vs = Ph + 32 * ell;         // [32][D]: U_d[:, :32] transposed
  const char* wu = s.ws + (size_t)u * s.ub;
  const float* Cg = (const float*)(wu + s.o_C);
  if (rd < D) {
    const float* Vg = (const float*)(wu + s.o_Vd);
    for (int e = t; e < D * 32; e += 256) Vs[(e & 31) * D + (e >> 5)] = Vg[(size_t)(e >> 5) * D + (e & 31)];
  }
  float acc[16];                     // entries t + 256 i of the ell x ell matrix (ell <= 64)
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int h = g * hper; h < (g + 1) * hper; ++h) {
    __syncthreads();
    for (int e = t; e < D * ell; e += 256) {
      const int d = e / ell, k = e % ell;
      Ch[e] = Cg[((size_t)h * D + d) * NC + r * ell + k];
    }
    __syncthreads();
    if (rd < D) {
      for (int e = t; e < rows * ell; e += 256) {
        const int j = e / ell, k = e % ell;
        float a = 0.f;
        for (int d = 0; d < D; ++d) a = fmaf(Vs[j * D + d], Ch[d * ell + k], a);
        Ph[e] = a;
      }
      __syncthreads();
    }
    const float* P = rd < D ? Ph : Ch;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = t + 256 * i;
      if (e < ell * ell) {
        const int a = e / ell, b = e % ell;
        float v = acc[i];
        for (int j = 0; j < rows; ++j) v = fmaf(P[j * ell + a], P[j * ell + b], v);
        acc[i] = v;
      }
    }
  }
  float* Hm = (float*)(prob(s, u, r) + s.p_Hm) + (size_t)g * ell * ell;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = t + 256 * i;
    if (e < ell * ell) Hm[e] = acc[i];
  }
}

}  // namespace

bool flash_tc_supported(const Layout& L) {
  return L.dtype == JOLT_BF16 && L.D == 128 && L.token_mode == JOLT_TOKEN_RANDOMIZED &&
         L.RT > 0 && L.ell % 4 == 0 && L.o_Bx != 0 && tc::encode_fn() != nullptr;
}

// One lockstep call: the ranks rid[0..nr) (indices into the rank grid) of every
// unit, problems at pbase + (u * pmul + pidx0[r]) * pb.
jolt_status flash_tc_solve(const Layout& L, int U, const void* X, const float* sketch, char* ws,
                           char* pbase, int pmul, const int* pidx0, const int* rid, int nr,
                           cudaStream_t st) {
  if (!flash_tc_supported(L) || nr < 1 || nr > 4) return JOLT_ERR_INVALID;
  FlashSet s;
  memset(&s, 0, sizeof(s));
  s.nr = nr; s.ell = L.ell;
  s.W = ((nr * L.ell + 31) / 32) * 32;
  if (s.W > FL_WMAX) return JOLT_ERR_INVALID;
  for (int r = 0; r < nr; ++r) {
    s.rdv[r] = L.rd[rid[r]];
    s.pidx0[r] = pidx0[r];
  }
  s.pmul = pmul;
  s.H = L.H; s.T = L.T; s.D = L.D; s.hs = L.hs;
  s.ws = ws; s.ub = L.unit_bytes; s.o_Vd = L.o_Vd; s.o_Bx = L.o_Bx; s.o_Qs = L.o_Qs;
  s.o_C = L.o_C; s.o_status = L.o_status;
  s.pbase = pbase; s.pb = L.prob_bytes; s.p_Z = L.p_Z; s.p_V = L.p_V; s.p_Hm = L.p_Hm;
  s.p_status = L.p_status;
  const int NC = nr * L.ell;

  CUtensorMap tXz, tB, tXc, tQ;
  {
    const cuuint64_t d[3] = {128, (cuuint64_t)L.T, (cuuint64_t)U * L.H};
    const cuuint64_t sd[2] = {256, (cuuint64_t)L.T * 256};
    const cuuint32_t bz[3] = {64, 128, 1};
    const cuuint32_t bc[3] = {64, FC_KT, 1};
    if (!tc::make_map(&tXz, X, 3, d, sd, bz) || !tc::make_map(&tXc, X, 3, d, sd, bc))
      return JOLT_ERR_CUDA;
  }
  {
    // H heads of 512 rows per unit, units at the unit stride
    const cuuint64_t d[4] = {128, FL_BROWS, (cuuint64_t)L.H, (cuuint64_t)U};
    const cuuint64_t sd[3] = {256, (cuuint64_t)FL_BROWS * 256, (cuuint64_t)L.unit_bytes};
    const cuuint32_t b[4] = {64, 256, 1, 1};
    if (!tc::make_map(&tB, ws + L.o_Bx, 4, d, sd, b)) return JOLT_ERR_CUDA;
  }
  {
    // U units of T x 512 rows at the unit stride
    const cuuint64_t d[3] = {FC_QCOLS, (cuuint64_t)L.T, (cuuint64_t)U};
    const cuuint64_t sd[2] = {FC_QCOLS * 2, (cuuint64_t)L.unit_bytes};
    const cuuint32_t b[3] = {64, FC_KT, 1};
    if (!tc::make_map(&tQ, ws + L.o_Qs, 3, d, sd, b)) return JOLT_ERR_CUDA;
  }
  const size_t zsm = 1024 + (size_t)FL_STAGES * FZ_STAGE + 128;
  const size_t csm = 1024 + (size_t)FL_STAGES * (FC_XST + 8 * FC_NATOM) + 128;
  const size_t bsm = ((size_t)L.D * NC + 32 * NC + (size_t)L.D * 32) * 4;
  const size_t rsm = ((size_t)L.D * L.ell + 32 * L.ell + (size_t)L.D * 32) * 4;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(flash_z_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)zsm));
    JOLT_CUDA_TRY(cudaFuncSetAttribute(flash_c_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm));
    JOLT_CUDA_TRY(cudaFuncSetAttribute(flash_b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(((size_t)128 * FL_WMAX + 32 * FL_WMAX + 128 * 32) * 4)));
    JOLT_CUDA_TRY(cudaFuncSetAttribute(flash_rr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(((size_t)128 * 64 + 32 * 64 + 128 * 32) * 4)));
    attr = true;
  }
  const dim3 gh(L.H, U), gz((L.T + 127) / 128, U);
  auto zpass = [&]() -> jolt_status {
    flash_z_kernel<<<gz, FL_THREADS, zsm, st>>>(tXz, tB, s);
    JOLT_LAUNCH_CHECK();
    return JOLT_OK;
  };
  auto cpass = [&]() -> jolt_status {
    flash_qsplit_kernel<<<dim3(64, U), 256, 0, st>>>(s);
    JOLT_LAUNCH_CHECK();
    flash_c_kernel<<<gh, FL_THREADS, csm, st>>>(tXc, tQ, s);
    JOLT_LAUNCH_CHECK();
    return JOLT_OK;
  };
  // the problems of rank r of every unit: a strided set
  bool contiguous = pmul == nr;
  for (int r = 0; r < nr; ++r) contiguous = contiguous && pidx0[r] == r;
  auto orth_all = [&]() -> jolt_status {
    if (contiguous) return cholqr2_set(L, pbase, L.prob_bytes, U * nr, st);
    for (int r = 0; r < nr; ++r) {
      const jolt_status e = cholqr2_set(L, pbase + (size_t)pidx0[r] * L.prob_bytes,
                                        (size_t)pmul * L.prob_bytes, U, st);
      if (e != JOLT_OK) return e;
    }
    return JOLT_OK;
  };
  // Z = A Omega, Q = orth(Z)
  flash_b_kernel<<<gh, 256, bsm, st>>>(s, sketch, 0);
  JOLT_LAUNCH_CHECK();
  if (jolt_status e = zpass()) return e;
  if (jolt_status e = orth_all()) return e;
  for (int q = 0; q <= L.power_iters; ++q) {
    if (jolt_status e = cpass()) return e;        // C_h = X_h^T Q
    if (q == L.power_iters) break;
    flash_b_kernel<<<gh, 256, bsm, st>>>(s, sketch, 1);   // B = V V^T C_h
    JOLT_LAUNCH_CHECK();
    if (jolt_status e = zpass()) return e;        // Z = A (A^T Q)
    if (jolt_status e = orth_all()) return e;
  }
  flash_rr_kernel<<<dim3(L.hs, nr, U), 256, rsm, st>>>(s);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace jolt
