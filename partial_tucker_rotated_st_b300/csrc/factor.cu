// Partial Tucker factors of a batch of units by ST-HOSVD over the feature and
// token modes, head axis kept.
//
// ["Joint Tucker-rank and residual-bit KV allocator", Mathematical statement
//  and Implementation notes: partial Tucker approximation over the token and
//  feature axes, sequential or randomized SVD of the unfoldings;
//  "Technical Summary: A JOLT for the KV Cache", Methodology 1 (ST-HOSVD,
//  head and layer axes kept) and 4 (FlashJoLT: randomized token-mode SVD).]
//
// Order (feature mode first, then the token mode of the projected tensor):
//   S_d = sum_{h,t} x x^T            split over head groups, f64 reduction
//   U_d = leading eigenvectors of S_d (Jacobi)
//   Y   = X U_d[:, :RD]              all truncated feature ranks at once
//   per feature rank r_d (ascending, untruncated last):
//     exact:      S_T(r_d) = sum_h Y_h[:, :r_d] Y_h[:, :r_d]^T (prefix sums over
//                 r_d; the untruncated mode uses X), then block subspace
//                 iteration with Rayleigh-Ritz to the leading RT eigenvectors
//                 (a direct Jacobi solve when T <= 128)
//     randomized: range finder Z = A Omega, q power steps A (A^T Q) each
//                 re-orthonormalised by CholeskyQR2, Rayleigh-Ritz on
//                 (A^T Q)^T (A^T Q)
//     cores G(r_d)[h] = U_T^T Y_h[:, :r_d]   (U_T^T X_h for r_d = D)
//   factors and cores rounded to fp16 (the storage type).
#include "jolt_internal.cuh"

#include <string.h>

#include <mutex>
#include <vector>

namespace jolt {

void* g_factor_ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};

namespace {

constexpr int SUB_STEPS = 5;        // power steps between Rayleigh-Ritz checks
constexpr float SUB_SHIFT = 1e-5f;  // shift of the equilibrated first CholeskyQR pass (f32)
constexpr int SUB_MAX_BLOCKS = 25;
int g_sub_blocks = SUB_MAX_BLOCKS;   // subspace-iteration block cap (host-settable)
constexpr float RITZ_TOL_REL = 1e-4f;
constexpr float RITZ_TOL_ABS = 1e-5f;

// Sd[u] = sum_s Sdp[u][s], in f64 (kept in f64 and rounded to fp32).
__global__ void reduce_splits_kernel(char* ws, size_t ub, size_t o_part, size_t o_out,
                                     size_t o_out64, int nsplit, int n) {
  const int u = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const float* p = (const float*)(ws + u * ub + o_part);
  double s = 0.0;
  for (int k = 0; k < nsplit; ++k) s += (double)p[(size_t)k * n + e];
  ((float*)(ws + u * ub + o_out))[e] = (float)s;
  ((double*)(ws + u * ub + o_out64))[e] = s;
}

// out[u][r][c] = fp16(in[u][r][c]) for r < rows, c < cols (row strides given).
__global__ void round_f16_kernel(char* ws, size_t ub, size_t o_in, int ld_in, size_t o_out,
                                 int ld_out, int rows, int cols, long long in_bs2,
                                 long long out_bs2, int nb2) {
  const int u = blockIdx.z / nb2, b2 = blockIdx.z % nb2;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)rows * cols) return;
  const int r = (int)(e / cols), c = (int)(e % cols);
  const float* in = (const float*)(ws + u * ub + o_in) + b2 * in_bs2;
  __half* out = (__half*)(ws + u * ub + o_out) + b2 * out_bs2;
  out[(long long)r * ld_out + c] = __float2half_rn(in[(long long)r * ld_in + c]);
}

// Deterministic start block for subspace iteration, uniform in [-1, 1).
__global__ void init_block_kernel(char* ws, size_t ub, size_t o_V, int n) {
  const int u = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  unsigned long long z = 0x9E3779B97F4A7C15ull * (unsigned long long)(e + 1) + 0x2545F4914F6CDD1Dull;
  z ^= z >> 31; z *= 0xBF58476D1CE4E5B9ull; z ^= z >> 27; z *= 0x94D049BB133111EBull; z ^= z >> 31;
  ((float*)(ws + u * ub + o_V))[e] = (float)((double)(z >> 11) * 0x1.0p-53 * 2.0 - 1.0);
}

// Rayleigh-Ritz convergence test and bookkeeping, one CTA per unit.
//   V2 = V W (Ritz vectors), Z2 = S V2, theta (descending Ritz values).
//   Converged when, for i < k, ||Z2_i - theta_i V2_i|| <= max(rel |theta_i|,
//   abs |theta_0|).  On convergence (or at the last iteration) the leading k
//   Ritz vectors go to U (T x k) and theta to ev.  Z2's columns are then
//   scaled by 1/||Z2_i|| (equilibration before CholeskyQR; the span is kept).
__global__ void ritz_check_kernel(char* ws, size_t ub, size_t o_V2, size_t o_Z2, size_t o_th,
                                  size_t o_U, size_t o_ev, size_t o_flag, size_t o_status,
                                  size_t o_V, int T, int Lw, int k, int last) {
  const int u = blockIdx.x;
  char* base = ws + u * ub;
  int* flag = (int*)(base + o_flag);
  if (*flag) return;
  const float* V2 = (const float*)(base + o_V2);
  float* Z2 = (float*)(base + o_Z2);
  const float* th = (const float*)(base + o_th);
  __shared__ float pr[512], pz[512];
  __shared__ float res[128], nz[128];
  __shared__ int ok, nonfinite;
  const int t = threadIdx.x;
  const int G = blockDim.x / Lw;          // row groups
  const int g = t / Lw, c = t % Lw;
  float r = 0.f, z = 0.f;
  if (g < G) {
    const float ti = th[c];
    for (int row = g; row < T; row += G) {
      const float zz = Z2[(long long)row * Lw + c];
      const float d = zz - ti * V2[(long long)row * Lw + c];
      r = fmaf(d, d, r);
      z = fmaf(zz, zz, z);
    }
  }
  pr[t] = r;
  pz[t] = z;
  __syncthreads();
  if (t < Lw) {
    float a = 0.f, b = 0.f;
    for (int q = 0; q < G; ++q) { a += pr[q * Lw + t]; b += pz[q * Lw + t]; }
    res[t] = sqrtf(a);
    nz[t] = sqrtf(b);
  }
  __syncthreads();
  if (t == 0) {
    int good = 1, nf = !isfinite(th[0]);
    const float a = RITZ_TOL_ABS * fabsf(th[0]);
    for (int i = 0; i < k; ++i) {
      const float lim = fmaxf(RITZ_TOL_REL * fabsf(th[i]), a);
      if (!(res[i] <= lim)) good = 0;
      if (!isfinite(res[i])) nf = 1;
    }
    ok = good;
    nonfinite = nf;
  }
  __syncthreads();
  if (nonfinite) {
    if (t == 0) {
      *flag = 1;
      atomicOr((int*)(base + o_status), ST_NONFINITE);
    }
    return;
  }
  if (ok || last) {
    float* U = (float*)(base + o_U);
    for (long long e = t; e < (long long)T * k; e += blockDim.x) {
      const int row = (int)(e / k), cc = (int)(e % k);
      U[e] = V2[(long long)row * Lw + cc];
    }
    // the orthonormal Ritz basis warm-starts the next feature rank
    float* V = (float*)(base + o_V);
    for (long long e = t; e < (long long)T * Lw; e += blockDim.x) V[e] = V2[e];
    float* ev = (float*)(base + o_ev);
    for (int i = t; i < k; i += blockDim.x) ev[i] = th[i];
    if (t == 0) {
      *flag = 1;
      if (!ok) atomicOr((int*)(base + o_status), ST_NOCONVERGE);
    }
    return;
  }
  // equilibrate the columns of Z2 before the next orthonormalisation
  for (long long e = t; e < (long long)T * Lw; e += blockDim.x) {
    const int cc = (int)(e % Lw);
    const float sc = nz[cc] > 0.f ? 1.f / nz[cc] : 0.f;
    Z2[e] *= sc;
  }
}

// out[u] = first k columns of in[u] (rows x ld_in) into rows x k.
__global__ void copy_cols_kernel(char* ws, size_t ub, size_t o_in, int ld_in, size_t o_out,
                                 int rows, int k) {
  const int u = blockIdx.y;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)rows * k) return;
  const int r = (int)(e / k), c = (int)(e % k);
  ((float*)(ws + u * ub + o_out))[e] = ((const float*)(ws + u * ub + o_in))[(long long)r * ld_in + c];
}

__global__ void set_int_kernel(char* ws, size_t ub, size_t o, int v) {
  if (threadIdx.x == 0) *(int*)(ws + blockIdx.x * ub + o) = v;
}

// Truncated problem p = u * ndt + id starts from the whole-feature problem's
// converged Ritz basis of unit u: V[p] = V[full u].
__global__ void warm_copy_kernel(char* pbase, size_t pb, size_t o_V, int ndt, const char* fbase,
                                 long long n) {
  const int p = blockIdx.y, u = p / ndt;
  const float* src = (const float*)(fbase + (size_t)u * pb + o_V);
  float* dst = (float*)(pbase + (size_t)p * pb + o_V);
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x)
    dst[e] = src[e];
}

// Token factors and eigenvalues of every problem into its unit's sections
// (U_T of rank id at o_UT + id * T * RT, eigenvalues at o_ev + id * RT), and
// the problem's status bits OR-ed into the unit's status.
__global__ void scatter_problems_kernel(char* ws, size_t ub, size_t o_UT, size_t o_ev,
                                        size_t o_status, const char* pbase, size_t pb,
                                        size_t p_UT, size_t p_ev, int ev_ld, size_t p_status,
                                        int U, int ndt, int T, int RT, size_t o_cap) {
  const int id = blockIdx.y, u = blockIdx.z;
  const int p = id < ndt ? u * ndt + id : U * ndt + u;
  const char* pr = pbase + (size_t)p * pb;
  char* un = ws + (size_t)u * ub;
  const float* src = (const float*)(pr + p_UT);
  float* dst = (float*)(un + o_UT) + (size_t)id * T * RT;
  const long long n = (long long)T * RT;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x)
    dst[e] = src[e];
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < RT; i += blockDim.x) {
      ((float*)(un + o_ev))[id * RT + i] = ((const float*)(pr + p_ev))[i * ev_ld];
      ((double*)(un + o_cap))[id * RT + i] = 0.0;   // the cores stage adds into it
    }
    if (threadIdx.x == 0) {
      const int sv = *(const int*)(pr + p_status);
      if (sv) atomicOr((int*)(un + o_status), sv);
    }
  }
}

// Captured energy of the unrounded cores, cap[id][j] = sum over h and i < r_d
// of G(r_d)[h][j][i]^2 in f64 (one warp per (rank, j)), from the fp32 cores
// G32[id][h][j][i] (row stride r_d).
struct RdList { int rd[JOLT_MAX_GRID]; };
__global__ void cap_g32_kernel(char* ws, size_t ub, size_t o_G32, size_t o_cap, int H, int RT,
                               int D, int nd, RdList rl) {
  const int u = blockIdx.y;
  char* un = ws + (size_t)u * ub;
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= nd * RT) return;
  const int id = w / RT, j = w % RT, rd = rl.rd[id];
  const float* G = (const float*)(un + o_G32) + (size_t)id * H * RT * D;
  double s = 0.0;
  for (int e = lane; e < H * rd; e += 32) {
    const int h = e / rd, i = e % rd;
    const double g = G[((size_t)h * RT + j) * rd + i];
    s += g * g;
  }
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) ((double*)(un + o_cap))[id * RT + j] = s;
}

// Cores G(r_d)[h] = U_T(r_d)^T B_h[:, :n] for a set of feature ranks that
// share the same B (Y for the truncated ranks, X for the whole-feature one),
// one CTA per (head, unit).  B's rows and every rank's U_T rows are copied
// to shared memory 32 tokens at a time by cp.async, two stages deep, and
// reused by all ranks of the set; each thread owns one 4 x 4 tile of one
// core (r0..r0+3 x c0..c0+3), so the products of all ranks cost one pass
// over B.  Global rows must be 16-byte aligned (checked by the caller).
constexpr int CO_THREADS = 256, CO_TK = 32;
struct CoreArgs {
  const void* B;            // unit u, head h at B + u * b_us + h * b_hs (elements), row stride ldb
  long long b_us, b_hs;
  int ldb;
  int nset;                 // ranks in the set
  int id[JOLT_MAX_GRID];    // their indices (U_T at o_UT + id * T * RT, core at o_G + id * H * RT * D)
  int n[JOLT_MAX_GRID];     // their column counts (r_d)
  int nmax;                 // max n, a multiple of 8
  int T, RT, H, D;
  char* ws;
  size_t ub, o_UT, o_G;
};

__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(sdst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gsrc),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <typename T16>
__device__ __forceinline__ void load4(const T16* p, float (&v)[4]) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  const T16* h = reinterpret_cast<const T16*>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = to_f32(h[i]);
}

template <typename TB>
__global__ void __launch_bounds__(CO_THREADS) cores_kernel(CoreArgs a) {
  extern __shared__ __align__(16) unsigned char co_sm[];
  const int h = blockIdx.x, u = blockIdx.y, t = threadIdx.x;
  const int RT = a.RT;
  const size_t b_bytes = (size_t)CO_TK * a.nmax * sizeof(TB);
  const size_t stage_bytes = b_bytes + (size_t)a.nset * CO_TK * RT * 4;
  // this thread's tile: walk the ranks' tile counts (RT/4 x n/4 each)
  int sel = -1, r0 = 0, c0 = 0, rem = t;
  for (int s = 0; s < a.nset; ++s) {
    const int tiles = (RT / 4) * (a.n[s] / 4);
    if (sel < 0 && rem < tiles) { sel = s; r0 = (rem / (a.n[s] / 4)) * 4; c0 = (rem % (a.n[s] / 4)) * 4; }
    else if (sel < 0) rem -= tiles;
  }
  char* base = a.ws + (size_t)u * a.ub;
  const TB* Bh = (const TB*)a.B + u * a.b_us + h * a.b_hs;
  auto issue = [&](int k0, int stg) {
    unsigned char* sb = co_sm + stg * stage_bytes;
    const int segs = (int)(a.nmax * sizeof(TB) / 16);   // 16-byte pieces per B row
    for (int e = t; e < CO_TK * segs; e += CO_THREADS) {
      const int k = e / segs, sg = e % segs;
      const bool ok = k0 + k < a.T;
      const TB* src = Bh + (long long)(ok ? k0 + k : 0) * a.ldb;
      cp_async16(sb + (size_t)k * a.nmax * sizeof(TB) + sg * 16,
                 reinterpret_cast<const unsigned char*>(src) + sg * 16, ok);
    }
    for (int s = 0; s < a.nset; ++s) {
      const float* Ug = (const float*)(base + a.o_UT) + (size_t)a.id[s] * a.T * RT;
      unsigned char* su = sb + b_bytes + (size_t)s * CO_TK * RT * 4;
      for (int e = t; e < CO_TK * RT / 4; e += CO_THREADS) {
        const int k = (4 * e) / RT;
        const bool ok = k0 + k < a.T;
        cp_async16(su + (size_t)e * 16, Ug + (ok ? (long long)k0 * RT + 4 * e : 0), ok);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  issue(0, 0);
  int stg = 0;
  for (int k0 = 0; k0 < a.T; k0 += CO_TK) {
    const bool more = k0 + CO_TK < a.T;
    if (more) {
      issue(k0 + CO_TK, stg ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    if (sel >= 0) {
      const unsigned char* sb = co_sm + stg * stage_bytes;
      const TB* bs = reinterpret_cast<const TB*>(sb);
      const float* us = reinterpret_cast<const float*>(sb + b_bytes) + sel * CO_TK * RT;
#pragma unroll 8
      for (int k = 0; k < CO_TK; ++k) {
        float ur[4], bc[4];
        load4(us + k * RT + r0, ur);
        load4(bs + k * a.nmax + c0, bc);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ur[i], bc[j], acc[i][j]);
      }
    }
    __syncthreads();   // this stage is refilled next
    stg ^= 1;
  }
  if (sel >= 0) {
    const int n = a.n[sel];
    float* G = (float*)(base + a.o_G) + (size_t)a.id[sel] * a.H * RT * a.D + (size_t)h * RT * n;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(G + (r0 + i) * n + c0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

// The batch of units of one call (unit u at ws + u * unit_bytes).
struct F {
  const Layout& L;
  char* ws;
  int U;
  cudaStream_t st;
  float* f(size_t o) const { return (float*)(ws + o); }
};

// A set of token problems: np problems at base + i * stride, offsets p_*.
struct PS {
  char* base;
  size_t stride;
  int np;
  long long s4() const { return (long long)stride / 4; }
  float* f(size_t o) const { return (float*)(base + o); }
  char* c(size_t o) const { return base + o; }
};

Opnd opnd(const void* p, int dt, long long s0, long long s1, long long sseg = 0, long long sb1 = 0,
          long long sb2 = 0) {
  Opnd o;
  o.p = p; o.dtype = dt; o.s0 = s0; o.s1 = s1; o.sseg = sseg; o.sb1 = sb1; o.sb2 = sb2;
  return o;
}

GemmDesc gd(int M, int N, int K, int nseg, int nb1, int nb2, Opnd A, Opnd B, float* C, long long cm,
            long long cn, long long cb1, long long cb2, float beta = 0.f, const int* skip = nullptr) {
  GemmDesc g;
  g.M = M; g.N = N; g.K = K; g.nseg = nseg; g.nb1 = nb1; g.nb2 = nb2;
  g.A = A; g.B = B; g.C = C; g.cm = cm; g.cn = cn; g.cb1 = cb1; g.cb2 = cb2;
  g.alpha = 1.f; g.beta = beta; g.skip = skip;
  return g;
}

#define TRY(x)                       \
  do {                               \
    jolt_status s_ = (x);            \
    if (s_ != JOLT_OK) return s_;    \
  } while (0)


// dst <- orth(src) by CholeskyQR through mid; T x Lw per problem.  passes =
// 2 is CholeskyQR2 (Fukaya et al. 2014); `shift` > 0 shifts the first pass
// (shifted CholeskyQR, Fukaya et al. 2020) for nearly dependent columns.
// Each pass: Gram split over L.ks row chunks (the partials are summed inside
// the Cholesky kernel), Cholesky R, then out = in R^{-1}.  With one pass the
// result goes straight to dst.  Problems whose flag is set are skipped when
// `use_flags`.
jolt_status cholqr(const Layout& L, const PS& P, int T, int Lw, size_t src, size_t mid, size_t dst,
                   bool use_flags, bool f64, int passes, float shift, cudaStream_t st,
                   bool* vs_written = nullptr) {
  const long long s4 = P.s4();
  const int ks = L.ks, kc = T / L.ks;
  const int* skip = use_flags ? (const int*)P.c(L.p_flag) : nullptr;
  int* status = (int*)P.c(L.p_status);
  if (vs_written) *vs_written = false;
  if (!f64 && cholqr_fused_supported(T, Lw, P.np)) {
    // the fused kernel also writes the power step's transposed operand
    const size_t vt = (dst == L.p_V && L.p_Vs != 0) ? L.p_Vs : 0;
    if (vs_written) *vs_written = vt != 0;
    return cholqr_fused(P.base, P.stride, P.np, src, dst, L.p_status, skip, s4, T, passes, shift,
                        st, vt);
  }
  const size_t ins[2] = {src, mid}, outs[2] = {passes == 1 ? dst : mid, dst};
  for (int pass = 0; pass < passes; ++pass) {
    GemmDesc g = gd(Lw, Lw, kc, 1, P.np, ks,
                    opnd(P.c(ins[pass]), JOLT_F32, 1, Lw, 0, s4, (long long)kc * Lw),
                    opnd(P.c(ins[pass]), JOLT_F32, Lw, 1, 0, s4, (long long)kc * Lw),
                    P.f(L.p_Gram), Lw, 1, s4, (long long)Lw * Lw, 0.f, skip);
    g.skip_stride = s4;
    TRY(launch_gemm(g, st));
    const float sh = pass == 0 ? shift : 0.f;
    if (!f64) {
      // out = in R^{-1} as a plain product (R^{-1} from the Cholesky kernel)
      TRY(launch_chol_inv(P.f(L.p_Gram), s4, Lw, ks, (long long)Lw * Lw, P.np, P.f(L.p_Rinv), s4,
                          status, s4, skip, s4, sh, st));
      GemmDesc m = gd(T, Lw, Lw, 1, P.np, 1, opnd(P.c(ins[pass]), JOLT_F32, Lw, 1, 0, s4),
                      opnd(P.c(L.p_Rinv), JOLT_F32, Lw, 1, 0, s4), P.f(outs[pass]), Lw, 1, s4, 0,
                      0.f, skip);
      m.skip_stride = s4;
      TRY(launch_gemm(m, st));
    } else {
      TRY(launch_chol(P.f(L.p_Gram), s4, Lw, ks, (long long)Lw * Lw, P.np, P.f(L.p_Rinv), s4,
                      status, s4, skip, s4, true, sh, st));
      TRY(launch_trsm_rows(P.f(ins[pass]), P.f(outs[pass]), s4, P.f(L.p_Rinv), s4, T, Lw, P.np,
                           skip, s4, st));
    }
  }
  return JOLT_OK;
}

jolt_status cholqr2(const Layout& L, const PS& P, int T, int Lw, size_t src, size_t mid,
                    size_t dst, bool use_flags, bool f64, cudaStream_t st,
                    bool* vs_written = nullptr) {
  return cholqr(L, P, T, Lw, src, mid, dst, use_flags, f64, 2, f64 ? 0.f : SUB_SHIFT, st,
                vs_written);
}

}  // namespace

jolt_status cholqr2_set(const Layout& L, char* base, size_t stride, int np, cudaStream_t st) {
  const PS P{base, stride, np};
  return cholqr2(L, P, L.T, L.ell, L.p_Z, L.p_V2, L.p_V, false, true, st);
}

namespace {

jolt_status read_flags_all(const Layout& L, const PS& P, cudaStream_t st, bool* all) {
  std::vector<int> h(P.np);
  JOLT_CUDA_TRY(cudaMemcpy2DAsync(h.data(), sizeof(int), P.c(L.p_flag), P.stride, sizeof(int),
                                  P.np, cudaMemcpyDeviceToHost, st));
  JOLT_CUDA_TRY(cudaStreamSynchronize(st));
  bool a = true;
  for (int v : h) a = a && (v != 0);
  *all = a;
  return JOLT_OK;
}

unsigned blocks_for(long long n, int tpb = 256) { return (unsigned)((n + tpb - 1) / tpb); }

// A non-blocking side stream per device for the feature stage, which runs
// alongside the whole-feature token problem (it needs only X).  Callers that
// share it serialise their feature stages on it; each joins through its own
// events.
//
// The whole-feature token solve, a chain of small latency-bound launches, runs
// on a second side stream of the highest priority, so that its blocks are
// scheduled ahead of the feature stage's wide launches.
jolt_status aux_stream(cudaStream_t* out, bool high = false) {
  static std::mutex mu;
  static cudaStream_t streams[2][64] = {};
  int dev = 0;
  JOLT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return JOLT_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  cudaStream_t& s = streams[high ? 1 : 0][dev];
  if (!s) {
    int least = 0, greatest = 0;
    JOLT_CUDA_TRY(cudaDeviceGetStreamPriorityRange(&least, &greatest));
    JOLT_CUDA_TRY(cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, high ? greatest : least));
  }
  *out = s;
  return JOLT_OK;
}

struct EventPair {
  cudaEvent_t a = nullptr, b = nullptr, c = nullptr;
  ~EventPair() {
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
    if (c) cudaEventDestroy(c);
  }
};

// On every exit (errors included) the caller's stream waits for all the
// side streams' work, so that the workspace is never released under it.
struct JoinGuard {
  cudaStream_t st = nullptr, fs = nullptr, ps = nullptr;
  cudaEvent_t ev = nullptr, ev2 = nullptr;
  ~JoinGuard() {
    if (ev && fs && fs != st && cudaEventRecord(ev, fs) == cudaSuccess) cudaStreamWaitEvent(st, ev, 0);
    if (ev2 && ps && ps != st && cudaEventRecord(ev2, ps) == cudaSuccess) cudaStreamWaitEvent(st, ev2, 0);
  }
};

// Exact token mode for a set of problems whose S_T (p_ST) is final: the
// leading RT eigenvectors into p_UT, eigenvalues into p_ev (direct Jacobi when
// T <= 128, else block subspace iteration with Rayleigh-Ritz).  `warm`: p_V
// already holds an orthonormal start block.
jolt_status token_exact(const Layout& L, const PS& P, bool warm, cudaStream_t st,
                        bool split_done = false) {
  const int T = L.T, RT = L.RT, Lw = L.L;
  const long long s4 = P.s4();
  int* status = (int*)P.c(L.p_status);
  if (T <= 128) {
    TRY(launch_jacobi(P.f(L.p_ST), s4, T, T, 1, 0, P.np, P.f(L.p_theta), s4, P.f(L.p_UT), s4, RT,
                      RT, status, s4, nullptr, 0, JAC_ABS_EXACT, st));
    copy_cols_kernel<<<dim3(blocks_for(RT), P.np), 256, 0, st>>>(P.base, P.stride, L.p_theta, T,
                                                                 L.p_ev, 1, RT);
    JOLT_LAUNCH_CHECK();
    return JOLT_OK;
  }
  bool vs_ready = false;   // p_Vs holds the current p_V's transpose and low part
  if (!warm) {
    init_block_kernel<<<dim3(blocks_for((long long)T * Lw), P.np), 256, 0, st>>>(
        P.base, P.stride, L.p_V, T * Lw);
    JOLT_LAUNCH_CHECK();
    TRY(cholqr2(L, P, T, Lw, L.p_V, L.p_V2, L.p_V, false, false, st, &vs_ready));
  }
  set_int_kernel<<<P.np, 32, 0, st>>>(P.base, P.stride, L.p_flag, 0);
  JOLT_LAUNCH_CHECK();
  const bool svtc = sv_tc_supported(L);
  if (svtc && !split_done) TRY(split_tok_gram(L, P.np, P.base, P.stride, st));
  const int* flags = (const int*)P.c(L.p_flag);
  // Z lives in one of two buffers: Rayleigh-Ritz writes Z2 = S V2 into the
  // other one, and the next block starts from it (its first power step is
  // already done), so the roles swap every block
  size_t zc = L.p_Z, zn = L.p_Z2;
  auto apply_S = [&]() -> jolt_status {  // Z = S V
    if (svtc) return sv_tc(L, P.np, P.base, P.stride, zc, st, vs_ready);
    GemmDesc gg = gd(T, Lw, T, 1, P.np, 1, opnd(P.c(L.p_ST), JOLT_F32, T, 1, 0, s4),
                     opnd(P.c(L.p_V), JOLT_F32, Lw, 1, 0, s4), P.f(zc), Lw, 1, s4, 0, 0.f,
                     flags);
    gg.skip_stride = s4;
    return launch_gemm(gg, st);
  };
  // blocks of SUB_STEPS power steps V <- orth(S V), then Rayleigh-Ritz and
  // the residual test; converged problems are skipped from then on
  for (int blk = 0; blk < g_sub_blocks; ++blk) {
    // one shifted CholeskyQR pass per power step; the last step of a block
    // takes two so that Rayleigh-Ritz sees an orthonormal basis
    for (int q = 0; q < SUB_STEPS; ++q) {
      if (q > 0 || blk == 0) TRY(apply_S());
      TRY(cholqr(L, P, T, Lw, zc, L.p_V2, L.p_V, true, false, q == SUB_STEPS - 1 ? 2 : 1,
                 SUB_SHIFT, st, &vs_ready));
    }
    TRY(apply_S());
    // H = V^T Z, split over row chunks; the eigensolver sums the partials
    const int kc = T / L.ks;
    GemmDesc g = gd(Lw, Lw, kc, 1, P.np, L.ks,
                    opnd(P.c(L.p_V), JOLT_F32, 1, Lw, 0, s4, (long long)kc * Lw),
                    opnd(P.c(zc), JOLT_F32, Lw, 1, 0, s4, (long long)kc * Lw), P.f(L.p_Hm),
                    Lw, 1, s4, (long long)Lw * Lw, 0.f, flags);
    g.skip_stride = s4;
    TRY(launch_gemm(g, st));
    {
      // Cholesky + one-sided Jacobi where Lw allows it; problems it leaves
      // unsolved (and every problem for another Lw) take the two-sided Jacobi
      int* done = status + 2;
      const jolt_status se = launch_sym_eig(P.c(L.p_Hm), false, s4, Lw, Lw, L.ks,
                                            (long long)Lw * Lw, P.np, P.f(L.p_theta), s4,
                                            P.f(L.p_Wm), s4, Lw, Lw, status, s4, done, s4, flags,
                                            s4, JAC_ABS_RR, st);
      if (se != JOLT_OK && se != JOLT_ERR_INVALID) return se;
      TRY(launch_jacobi(P.f(L.p_Hm), s4, Lw, Lw, L.ks, (long long)Lw * Lw, P.np, P.f(L.p_theta),
                        s4, P.f(L.p_Wm), s4, Lw, Lw, status, s4, se == JOLT_OK ? done : flags, s4,
                        JAC_ABS_RR, st));
    }
    // Ritz vectors V2 = V W and Z2 = Z W = S V2
    g = gd(T, Lw, Lw, 1, P.np, 1, opnd(P.c(L.p_V), JOLT_F32, Lw, 1, 0, s4),
           opnd(P.c(L.p_Wm), JOLT_F32, Lw, 1, 0, s4), P.f(L.p_V2), Lw, 1, s4, 0, 0.f, flags);
    g.skip_stride = s4;
    TRY(launch_gemm(g, st));
    g = gd(T, Lw, Lw, 1, P.np, 1, opnd(P.c(zc), JOLT_F32, Lw, 1, 0, s4),
           opnd(P.c(L.p_Wm), JOLT_F32, Lw, 1, 0, s4), P.f(zn), Lw, 1, s4, 0, 0.f, flags);
    g.skip_stride = s4;
    TRY(launch_gemm(g, st));
    const int last = (blk == g_sub_blocks - 1);
    ritz_check_kernel<<<P.np, 512, 0, st>>>(P.base, P.stride, L.p_V2, zn, L.p_theta, L.p_UT,
                                            L.p_ev, L.p_flag, L.p_status, L.p_V, T, Lw, RT, last);
    JOLT_LAUNCH_CHECK();
    if (last) break;
    // the next block starts from Z2 (equilibrated by the check)
    const size_t tmp = zc; zc = zn; zn = tmp;
    // a cold start takes two blocks at least: no host round trip before the
    // second (problems that converge earlier are skipped by their flags)
    if (!warm && blk == 0) continue;
    bool all = false;
    TRY(read_flags_all(L, P, st, &all));
    if (all) break;
  }
  return JOLT_OK;
}

// FlashJoLT randomized range finder for one feature rank over a set of U
// problems (one per unit): A_h = Y_h[:, :rdv] (or X_h for rdv = D), leading
// RT approximate eigenvectors of sum_h A_h A_h^T into p_UT, values into p_ev.
jolt_status token_randomized(const F& c, const PS& P, const void* Ab, int adt, long long as_t,
                             long long aseg, long long aub, int rdv, const float* sketch) {
  const Layout& L = c.L;
  const int T = L.T, H = L.H, D = L.D, RT = L.RT, ell = L.ell;
  const long long s4 = P.s4(), ub4 = (long long)L.unit_bytes / 4;
  cudaStream_t st = c.st;
  int* status = (int*)P.c(L.p_status);
  const long long sk_h = (long long)D * ell, sk_u = (long long)H * D * ell;
  // Q lives in V: Z = A Omega, Q = orth(Z); then q times Q = orth(A (A^T Q))
  TRY(launch_gemm(gd(T, ell, rdv, H, c.U, 1, opnd(Ab, adt, as_t, 1, aseg, aub),
                     opnd(sketch, JOLT_F32, ell, 1, sk_h, sk_u), P.f(L.p_Z), ell, 1, s4, 0),
                  st));
  TRY(cholqr2(L, P, T, ell, L.p_Z, L.p_V2, L.p_V, false, true, st));
  for (int q = 0; q <= L.power_iters; ++q) {
    // P_h = A_h^T Q  (rdv x ell per head)
    TRY(launch_gemm(gd(rdv, ell, T, 1, c.U, H, opnd(Ab, adt, 1, as_t, 0, aub, aseg),
                       opnd(P.c(L.p_V), JOLT_F32, ell, 1, 0, s4, 0), c.f(L.o_P), ell, 1, ub4,
                       (long long)rdv * ell),
                    st));
    if (q == L.power_iters) break;
    // Z = sum_h A_h P_h, re-orthonormalised
    TRY(launch_gemm(gd(T, ell, rdv, H, c.U, 1, opnd(Ab, adt, as_t, 1, aseg, aub),
                       opnd(c.ws + L.o_P, JOLT_F32, ell, 1, (long long)rdv * ell, ub4),
                       P.f(L.p_Z), ell, 1, s4, 0),
                    st));
    TRY(cholqr2(L, P, T, ell, L.p_Z, L.p_V2, L.p_V, false, true, st));
  }
  // Rayleigh-Ritz: B B^T with B = Q^T A, i.e. sum_h P_h^T P_h, split over
  // head groups; the Jacobi kernel sums the partials
  const int hs = L.hs, hper = H / L.hs;
  TRY(launch_gemm(gd(ell, ell, rdv, hper, c.U, hs,
                     opnd(c.ws + L.o_P, JOLT_F32, 1, ell, (long long)rdv * ell, ub4,
                          (long long)hper * rdv * ell),
                     opnd(c.ws + L.o_P, JOLT_F32, ell, 1, (long long)rdv * ell, ub4,
                          (long long)hper * rdv * ell),
                     P.f(L.p_Hm), ell, 1, s4, (long long)ell * ell),
                  st));
  TRY(launch_jacobi(P.f(L.p_Hm), s4, ell, ell, hs, (long long)ell * ell, c.U, P.f(L.p_theta), s4,
                    P.f(L.p_Wm), s4, ell, RT, status, s4, nullptr, 0, JAC_ABS_EXACT, st));
  TRY(launch_gemm(gd(T, RT, ell, 1, c.U, 1, opnd(P.c(L.p_V), JOLT_F32, ell, 1, 0, s4),
                     opnd(P.c(L.p_Wm), JOLT_F32, ell, 1, 0, s4), P.f(L.p_UT), RT, 1, s4, 0),
                  st));
  copy_cols_kernel<<<dim3(blocks_for(RT), c.U), 256, 0, st>>>(P.base, P.stride, L.p_theta, ell,
                                                              L.p_ev, 1, RT);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

// The end of a randomized solve for a set of problems whose p_Hm (the
// Rayleigh-Ritz matrix in L.hs partials) and p_V (the orthonormal Q) are final:
// eigenpairs of p_Hm, U_T = Q W, eigenvalues to p_ev.
jolt_status rand_finish(const Layout& L, const PS& P, cudaStream_t st) {
  const int T = L.T, RT = L.RT, ell = L.ell;
  const long long s4 = P.s4();
  int* status = (int*)P.c(L.p_status);
  TRY(launch_jacobi(P.f(L.p_Hm), s4, ell, ell, L.hs, (long long)ell * ell, P.np, P.f(L.p_theta),
                    s4, P.f(L.p_Wm), s4, ell, RT, status, s4, nullptr, 0, JAC_ABS_EXACT, st));
  TRY(launch_gemm(gd(T, RT, ell, 1, P.np, 1, opnd(P.c(L.p_V), JOLT_F32, ell, 1, 0, s4),
                     opnd(P.c(L.p_Wm), JOLT_F32, ell, 1, 0, s4), P.f(L.p_UT), RT, 1, s4, 0),
                  st));
  copy_cols_kernel<<<dim3(blocks_for(RT), P.np), 256, 0, st>>>(P.base, P.stride, L.p_theta, ell,
                                                              L.p_ev, 1, RT);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace

jolt_status factor_run(const Layout& L, int U, const void* X, const float* sketch, char* ws,
                       cudaStream_t st) {
  F c{L, ws, U, st};
  const size_t ub = L.unit_bytes;
  const long long ub4 = (long long)ub / 4;
  const int H = L.H, T = L.T, D = L.D, RD = L.RD, RT = L.RT;
  const int xdt = L.dtype;
  const long long xu = (long long)H * T * D;
  int* status = (int*)(ws + L.o_status);

  // measurement hook: stage-boundary events (see jolt_set_factor_events)
  auto mark = [&](int i, cudaStream_t s) -> jolt_status {
    if (g_factor_ev[i]) JOLT_CUDA_TRY(cudaEventRecord((cudaEvent_t)g_factor_ev[i], s));
    return JOLT_OK;
  };
  TRY(mark(0, st));
  set_int_kernel<<<U, 32, 0, st>>>(ws, ub, L.o_status, 0);
  JOLT_LAUNCH_CHECK();
  if (RT > 0) {
    // the token problems' status words, before any stream forks off
    set_int_kernel<<<U * L.nprob, 32, 0, st>>>(ws + (size_t)U * ub, L.prob_bytes, L.p_status, 0);
    JOLT_LAUNCH_CHECK();
  }

  const bool tc = gram_tc_supported(L);
  // The whole-feature token problem (r_d = D) reads only X: the feature
  // stage runs beside it on a side stream and the truncated ranks join it.
  const bool overlap = RT > 0 && L.hasFullD && RD > 0;
  cudaStream_t fs = st, ps = st;
  EventPair ev;
  if (overlap) {
    TRY(aux_stream(&fs));
    TRY(aux_stream(&ps, true));
    JOLT_CUDA_TRY(cudaEventCreateWithFlags(&ev.a, cudaEventDisableTiming));
    JOLT_CUDA_TRY(cudaEventCreateWithFlags(&ev.b, cudaEventDisableTiming));
    JOLT_CUDA_TRY(cudaEventCreateWithFlags(&ev.c, cudaEventDisableTiming));
    JOLT_CUDA_TRY(cudaEventRecord(ev.a, st));
    JOLT_CUDA_TRY(cudaStreamWaitEvent(fs, ev.a, 0));
    JOLT_CUDA_TRY(cudaStreamWaitEvent(ps, ev.a, 0));
  }
  JoinGuard join_guard;
  if (overlap) {
    join_guard.st = st; join_guard.fs = fs; join_guard.ev = ev.a;
    join_guard.ps = ps; join_guard.ev2 = ev.b;
  }
  // ---- feature mode: S_d, split over groups of hg heads, f64 reduction
  {
    const int hg = H / L.nsplit;
    if (tc && (hg * T) % 64 == 0) {
      TRY(gram_feat_tc(L, U, X, ws, fs));
    } else {
      TRY(launch_gemm(gd(D, D, T, hg, U, L.nsplit,
                         opnd(X, xdt, 1, D, (long long)T * D, xu, (long long)hg * T * D),
                         opnd(X, xdt, D, 1, (long long)T * D, xu, (long long)hg * T * D),
                         c.f(L.o_Sdp), D, 1, ub4, (long long)D * D),
                      fs));
    }
    reduce_splits_kernel<<<dim3(blocks_for(D * D), U), 256, 0, fs>>>(ws, ub, L.o_Sdp, L.o_Sd,
                                                                     L.o_Sd64, L.nsplit, D * D);
    JOLT_LAUNCH_CHECK();
    // Cholesky + one-sided Jacobi; units whose S_d is not definite (done
    // flag left clear) are solved by the two-sided Jacobi
    int* done = status + 2;
    TRY(launch_sym_eig(ws + L.o_Sd64, true, ub4 / 2, D, D, 1, 0, U, c.f(L.o_evd), ub4,
                       c.f(L.o_Vd), ub4, D, D, status, ub4, done, ub4, nullptr, 0, JAC_ABS_EXACT,
                       fs));
    TRY(launch_jacobi(c.f(L.o_Sd), ub4, D, D, 1, 0, U, c.f(L.o_evd), ub4, c.f(L.o_Vd), ub4, D, D,
                      status, ub4, done, ub4, JAC_ABS_EXACT, fs));
  }
  // projection Y = X U_d[:, :RD]: on the tensor cores for bf16 X (which also
  // writes U_d16, Y16 and the token-Gram relayout Yt), else the SIMT product
  bool yt_done = false;
  if (RD > 0 && proj_tc_supported(L)) {
    // Y in fp32 only for the consumers that read it: the randomized token
    // mode, the SIMT token Grams (T <= 128 or no tensor-core path) and the
    // SIMT cores
    const bool y_needed = L.token_mode == JOLT_TOKEN_RANDOMIZED || L.T <= 128 ||
                          !ygram_tc_supported(L) || !cores_tc_supported(L);
    TRY(proj_tc(L, U, X, ws, y_needed, fs));
    yt_done = L.o_Yt != 0;
  } else if (RD > 0) {
    round_f16_kernel<<<dim3(blocks_for(D * RD), 1, U), 256, 0, fs>>>(ws, ub, L.o_Vd, D, L.o_Ud16,
                                                                     RD, D, RD, 0, 0, 1);
    JOLT_LAUNCH_CHECK();
    TRY(launch_gemm(gd(H * T, RD, D, 1, U, 1, opnd(X, xdt, D, 1, 0, xu),
                       opnd(ws + L.o_Vd, JOLT_F32, D, 1, 0, ub4), c.f(L.o_Y), RD, 1, ub4, 0),
                    fs));
    round_f16_kernel<<<dim3(blocks_for((long long)H * T * RD), 1, U), 256, 0, fs>>>(
        ws, ub, L.o_Y, RD, L.o_Y16, RD, H * T, RD, 0, 0, 1);
    JOLT_LAUNCH_CHECK();
  }
  // The truncated ranks' token Grams need only Y: they follow the feature
  // stage on its stream, still beside the whole-feature token solve.
  const bool early_tr = RT > 0 && L.token_mode == JOLT_TOKEN_EXACT && L.ndt > 0 && L.T > 128;
  if (early_tr) {
    char* preg0 = ws + (size_t)U * ub;
    const size_t pb0 = L.prob_bytes;
    if (ygram_tc_supported(L)) {
      if (!yt_done) TRY(ytrans(L, U, ws, fs));
      TRY(ygram_tc(L, U, ws, preg0, pb0, fs));
    } else {
      for (int id = 0; id < L.ndt; ++id) {
        const long long ps4 = (long long)((size_t)L.ndt * pb0) / 4;
        const float* Y0 = (const float*)(ws + L.o_Y);
        const long long aseg = (long long)T * RD;
        TRY(launch_gemm(gd(T, T, L.rd[id], H, U, 1, opnd(Y0, JOLT_F32, RD, 1, aseg, ub4),
                           opnd(Y0, JOLT_F32, 1, RD, aseg, ub4),
                           (float*)(preg0 + (size_t)id * pb0 + L.p_ST), T, 1, ps4, 0),
                        fs));
      }
    }
    if (sv_tc_supported(L)) TRY(split_tok_gram(L, U * L.ndt, preg0, pb0, fs));
  }
  TRY(mark(1, fs));
  if (overlap) JOLT_CUDA_TRY(cudaEventRecord(ev.b, fs));
  if (RT == 0) {
    TRY(mark(2, st));
    TRY(mark(3, st));
    return mark(4, st);
  }

  // ---- token mode: one problem per (unit, feature rank)
  const bool exact = (L.token_mode == JOLT_TOKEN_EXACT);
  const int ndt = L.ndt;
  const size_t pb = L.prob_bytes;
  char* preg = ws + (size_t)U * ub;
  const PS all_tr{preg, pb, U * ndt};
  const PS full_ps{preg + (size_t)U * ndt * pb, pb, U};
  auto tr_id = [&](int id) { return PS{preg + (size_t)id * pb, (size_t)ndt * pb, U}; };
  bool joined = !overlap;
  // the caller's stream waits for the feature stage (event b) and for the
  // whole-feature solve on the high-priority stream (event c)
  auto join = [&]() -> jolt_status {
    if (!joined) {
      JOLT_CUDA_TRY(cudaStreamWaitEvent(st, ev.b, 0));
      JOLT_CUDA_TRY(cudaEventRecord(ev.c, ps));
      JOLT_CUDA_TRY(cudaStreamWaitEvent(st, ev.c, 0));
    }
    joined = true;
    return JOLT_OK;
  };
  if (exact) {
    // the whole-feature problem first: its Gram needs only X, so it runs
    // beside the feature stage
    if (L.hasFullD) {
      if (tc) {
        TRY(gram_tok_tc(L, U, X, full_ps.base, pb, ps));
      } else {
        TRY(launch_gemm(gd(T, T, D, H, U, 1, opnd(X, xdt, D, 1, (long long)T * D, xu),
                           opnd(X, xdt, 1, D, (long long)T * D, xu), full_ps.f(L.p_ST), T, 1,
                           full_ps.s4(), 0),
                        ps));
      }
      TRY(token_exact(L, full_ps, false, ps));
    }
    TRY(mark(2, ps));
    TRY(join());
    if (ndt > 0) {
      // every truncated rank's Gram (already queued after the feature stage
      // when T > 128), then one batched solve for all of them
      if (early_tr) {
      } else if (T > 128 && ygram_tc_supported(L)) {
        if (!yt_done) TRY(ytrans(L, U, ws, st));
        TRY(ygram_tc(L, U, ws, preg, pb, st));
      } else {
        for (int id = 0; id < ndt; ++id) {
          const PS P = tr_id(id);
          const float* Y0 = (const float*)(ws + L.o_Y);
          const long long aseg = (long long)T * RD;
          TRY(launch_gemm(gd(T, T, L.rd[id], H, U, 1, opnd(Y0, JOLT_F32, RD, 1, aseg, ub4),
                             opnd(Y0, JOLT_F32, 1, RD, aseg, ub4), P.f(L.p_ST), T, 1, P.s4(), 0),
                          st));
        }
      }
      const bool warm = L.hasFullD && T > 128;
      if (warm) {
        warm_copy_kernel<<<dim3(64, U * ndt), 256, 0, st>>>(preg, pb, L.p_V, ndt, full_ps.base,
                                                            (long long)T * L.L);
        JOLT_LAUNCH_CHECK();
      }
      TRY(token_exact(L, all_tr, warm, st, early_tr));
    }
  } else if (flash_tc_supported(L) && ndt <= 4 && ndt * L.ell <= 160) {
    // randomized on the tensor cores: the whole-feature rank first (beside
    // the feature stage: it needs only X), then every truncated rank in
    // lockstep (they need U_d)
    if (L.hasFullD) {
      const int rid[1] = {L.nd - 1}, pidx0[1] = {U * ndt};
      TRY(flash_tc_solve(L, U, X, sketch, ws, preg, 1, pidx0, rid, 1, st));
      TRY(rand_finish(L, full_ps, st));
    }
    TRY(mark(2, st));
    TRY(join());
    if (ndt > 0) {
      int rid[4], pidx0[4];
      for (int r = 0; r < ndt; ++r) rid[r] = pidx0[r] = r;
      TRY(flash_tc_solve(L, U, X, sketch, ws, preg, ndt, pidx0, rid, ndt, st));
      TRY(rand_finish(L, all_tr, st));
    }
  } else {
    bool marked = false;
    // randomized: the whole-feature rank first (beside the feature stage),
    // then the truncated ranks one at a time (their sketches differ in size)
    for (int oi = L.nd - 1; oi >= 0; --oi) {
      const int id = oi;
      const int rdv = L.rd[id];
      const bool full = (rdv == D);
      if (!full) {
        if (!marked) TRY(mark(2, st));
        marked = true;
        TRY(join());
      }
      if (full) {
        TRY(token_randomized(c, full_ps, X, xdt, D, (long long)T * D, xu, rdv, sketch));
      } else {
        TRY(token_randomized(c, tr_id(id), ws + L.o_Y, JOLT_F32, RD, (long long)T * RD, ub4, rdv,
                             sketch));
      }
    }
    if (!marked) TRY(mark(2, st));
  }
  TRY(join());
  TRY(mark(3, st));
  scatter_problems_kernel<<<dim3(64, L.nd, U), 256, 0, st>>>(
      ws, ub, L.o_UT32, L.o_tokev, L.o_status, preg, pb, L.p_UT, L.p_ev, 1, L.p_status, U, ndt, T,
      RT, L.o_cap);
  JOLT_LAUNCH_CHECK();
  // cores G(r_d)[h] = U_T^T A_h  (RT x rdv): on the tensor cores for bf16 X
  // (one pass over X for every rank, fp16 cores and U_T written directly)
  if (cores_tc_supported(L)) {
    TRY(cores_tc(L, U, X, ws, st));
    return mark(4, st);
  }
  // else the truncated ranks share one pass over Y, the whole-feature rank
  // reads X
  for (int pass = 0; pass < 2; ++pass) {
    CoreArgs ca;
    memset(&ca, 0, sizeof(ca));
    int tiles = 0;
    bool fits = (RT % 4) == 0;
    for (int id = 0; id < L.nd; ++id) {
      const bool full = (L.rd[id] == D);
      if (full != (pass == 1)) continue;
      ca.id[ca.nset] = id;
      ca.n[ca.nset] = L.rd[id];
      ca.nmax = ca.nmax > L.rd[id] ? ca.nmax : L.rd[id];
      fits = fits && (L.rd[id] % 4 == 0);
      tiles += (RT / 4) * (L.rd[id] / 4);
      ++ca.nset;
    }
    if (ca.nset == 0) continue;
    const size_t xel = pass == 1 ? (xdt == JOLT_F32 ? 4 : 2) : 4;
    fits = fits && tiles <= CO_THREADS && ca.nmax % 8 == 0 && RT % 4 == 0 &&
           (pass == 0 || ((uintptr_t)X % 16 == 0 && (D * xel) % 16 == 0));
    if (fits) {
      ca.T = T; ca.RT = RT; ca.H = H; ca.D = D;
      ca.ws = ws; ca.ub = ub; ca.o_UT = L.o_UT32; ca.o_G = L.o_G32;
      const size_t smem = 2 * ((size_t)CO_TK * ca.nmax * xel + (size_t)ca.nset * CO_TK * RT * 4);
      if (smem > 48 * 1024) fits = false;
    }
    if (fits) {
      const size_t smem = 2 * ((size_t)CO_TK * ca.nmax * xel + (size_t)ca.nset * CO_TK * RT * 4);
      const dim3 grid(H, U);
      if (pass == 0) {
        ca.B = ws + L.o_Y; ca.b_us = ub4; ca.b_hs = (long long)T * RD; ca.ldb = RD;
        cores_kernel<float><<<grid, CO_THREADS, smem, st>>>(ca);
      } else {
        ca.B = X; ca.b_us = xu; ca.b_hs = (long long)T * D; ca.ldb = D;
        if (xdt == JOLT_BF16) cores_kernel<__nv_bfloat16><<<grid, CO_THREADS, smem, st>>>(ca);
        else if (xdt == JOLT_F16) cores_kernel<__half><<<grid, CO_THREADS, smem, st>>>(ca);
        else cores_kernel<float><<<grid, CO_THREADS, smem, st>>>(ca);
      }
      JOLT_LAUNCH_CHECK();
    } else {
      for (int s = 0; s < ca.nset; ++s) {
        const int id = ca.id[s], rdv = L.rd[id];
        const bool full = (rdv == D);
        const void* Ab = full ? X : (const void*)(ws + L.o_Y);
        const int adt = full ? xdt : JOLT_F32;
        const long long as_t = full ? D : RD;
        const long long aseg = full ? (long long)T * D : (long long)T * RD;
        const long long aub = full ? xu : ub4;
        const size_t oUT = L.o_UT32 + (size_t)id * T * RT * 4;
        const size_t oG = L.o_G32 + (size_t)id * H * RT * D * 4;
        TRY(launch_gemm(gd(RT, rdv, T, 1, U, H, opnd(ws + oUT, JOLT_F32, 1, RT, 0, ub4),
                           opnd(Ab, adt, as_t, 1, 0, aub, aseg), c.f(oG), rdv, 1, ub4,
                           (long long)RT * rdv),
                        st));
      }
    }
  }
  {
    RdList rl;
    for (int i = 0; i < JOLT_MAX_GRID; ++i) rl.rd[i] = L.rd[i];
    cap_g32_kernel<<<dim3((L.nd * RT + 7) / 8, U), 256, 0, st>>>(ws, ub, L.o_G32, L.o_cap, H, RT,
                                                                D, L.nd, rl);
    JOLT_LAUNCH_CHECK();
  }
  for (int id = 0; id < L.nd; ++id) {
    const int rdv = L.rd[id];
    const size_t oG = L.o_G32 + (size_t)id * H * RT * D * 4;
    round_f16_kernel<<<dim3(blocks_for((long long)H * RT * rdv), 1, U), 256, 0, st>>>(
        ws, ub, oG, rdv, L.o_G16 + (size_t)id * H * RT * D * 2, rdv, H * RT, rdv, 0, 0, 1);
    JOLT_LAUNCH_CHECK();
  }
  round_f16_kernel<<<dim3(blocks_for((long long)L.nd * T * RT), 1, U), 256, 0, st>>>(
      ws, ub, L.o_UT32, RT, L.o_UT16, RT, L.nd * T, RT, 0, 0, 1);
  JOLT_LAUNCH_CHECK();
  return mark(4, st);
}

void set_subspace_blocks(int n) { g_sub_blocks = n > 0 ? n : SUB_MAX_BLOCKS; }

}  // namespace jolt
