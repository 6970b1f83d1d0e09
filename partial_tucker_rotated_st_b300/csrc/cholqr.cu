// CholeskyQR of the subspace-iteration blocks in one launch per call.
//
// ["Technical Summary: A JOLT for the KV Cache", Methodology 1 and 4: the
//  token-mode factor from the leading eigenvectors of the token Gram; the
//  block orthonormalisation is CholeskyQR / CholeskyQR2 (Fukaya et al. 2014),
//  with a diagonal shift on the first pass (shifted CholeskyQR, Fukaya et al.
//  2020).]
//
// The unfused path takes three launches per pass (the Gram, the Cholesky
// factor and its inverse, the product Z R^{-1}), each a few tens of
// microseconds of latency for a T x 64 block.  Here a cluster of CQ_NC CTAs
// (8, or 4 or 2 when 8 per problem would not all be resident at once: a
// problem holds its SMs for the whole call) owns one problem: each CTA keeps
// T / CQ_NC rows of the block in shared
// memory for every pass, forms their partial 64 x 64 Gram, and the partials
// are summed through distributed shared memory into CTA 0, which factors and
// inverts the equilibrated Gram (the same blocked Cholesky as the unfused
// kernel) and hands R^{-1} back the same way; every CTA then multiplies its
// rows in place.  Global memory is read once and written once per call.
#include "jolt_internal.cuh"
#include "chol_smem.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace jolt {

namespace {

constexpr int CQ_N = 64;          // block width
constexpr int CQ_THREADS = 256;
constexpr int CQ_ZLD = CQ_N + 4;  // staged row stride (floats): consecutive rows 4 banks apart
constexpr int CQ_MAXROWS = 512;   // rows per CTA
constexpr int CQ_GLD = CQ_N + 1;  // row stride of the Cholesky work arrays

struct CqArgs {
  char* base;
  size_t stride;        // problem p at base + p * stride
  size_t src, dst;      // T x 64 input and output blocks (may coincide)
  size_t vt;            // 64 x T transpose of the output and its tf32 low part (0: none)
  size_t o_status;
  const int* skip;      // optional per-problem flag (ints, stride sk_s): set -> skipped
  long long sk_s;
  int T, passes;
  float shift;          // added to the equilibrated Gram's diagonal on the first pass
};

size_t cq_smem(int rows) {
  return ((size_t)rows * CQ_ZLD + 2 * CQ_N * CQ_N + 2 * CQ_N * CQ_GLD + 2 * CQ_N) * 4 + 16;
}

// CQ_NC CTAs per problem (one cluster); the staged rows at the front of the
// dynamic shared memory, rows_per = ceil(T / CQ_NC) of them
template <int CQ_NC>
__global__ void __launch_bounds__(CQ_THREADS, 1)
cholqr_cluster_kernel(CqArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  const int p = blockIdx.y;
  if (a.skip && a.skip[p * a.sk_s]) return;   // uniform over the cluster
  const int rank = (int)cl.block_rank();
  extern __shared__ __align__(16) float cq_sm[];
  float* Z = cq_sm;                                 // [rows][CQ_ZLD]
  const int rows_per = (a.T + CQ_NC - 1) / CQ_NC;
  float* Gp = Z + rows_per * CQ_ZLD;                // this CTA's partial Gram [64][64]
  float* Rs = Gp + CQ_N * CQ_N;                     // R^{-1} [k][r]
  float* S = Rs + CQ_N * CQ_N;                      // CTA 0: equilibrated Gram, then L'
  float* X = S + CQ_N * CQ_GLD;                     // CTA 0: the summed Gram, then L'^{-1}
  float* rds = X + CQ_N * CQ_GLD;
  float* rpiv = rds + CQ_N;
  int* bad = reinterpret_cast<int*>(rpiv + CQ_N);
  const int t = threadIdx.x;
  const int r0 = rank * rows_per;
  const int nr = max(0, min(rows_per, a.T - r0));
  char* pb = a.base + (size_t)p * a.stride;

  // this CTA's rows (zero past T)
  const float* src = reinterpret_cast<const float*>(pb + a.src);
  for (int e = t; e < rows_per * (CQ_N / 4); e += CQ_THREADS) {
    const int r = e / (CQ_N / 4), c4 = e % (CQ_N / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nr) v = *reinterpret_cast<const float4*>(src + (size_t)(r0 + r) * CQ_N + 4 * c4);
    *reinterpret_cast<float4*>(Z + r * CQ_ZLD + 4 * c4) = v;
  }
  if (t == 0) *bad = 0;
  __syncthreads();

  for (int pass = 0; pass < a.passes; ++pass) {
    // ---- partial Gram of this CTA's rows: thread (bi, bj) owns a 4 x 4 block
    {
      const int bi = t >> 4, bj = t & 15;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
      for (int r = 0; r < rows_per; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(Z + r * CQ_ZLD + 4 * bi);
        const float4 y = *reinterpret_cast<const float4*>(Z + r * CQ_ZLD + 4 * bj);
        const float xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], yv[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(Gp + (4 * bi + i) * CQ_N + 4 * bj) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
    cl.sync();
    // ---- CTA c sums rows [8c, 8c + 8) of every partial into CTA 0's X
    {
      constexpr int RB = CQ_N / CQ_NC;
      float* X0 = cl.map_shared_rank(X, 0);
      for (int e = t; e < RB * CQ_N; e += CQ_THREADS) {
        const int i = rank * RB + e / CQ_N, j = e % CQ_N;
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < CQ_NC; ++c) s += cl.map_shared_rank(Gp, c)[i * CQ_N + j];
        X0[i * CQ_GLD + j] = s;
      }
    }
    cl.sync();
    // ---- CTA 0: R^{-1} of the (shifted) equilibrated Gram
    if (rank == 0) {
      chol_inv_smem<CQ_N>(S, X, rds, rpiv, bad, pass == 0 ? a.shift : 0.f);
      for (int e = t; e < CQ_N * CQ_N; e += CQ_THREADS) {
        const int k = e / CQ_N, r = e % CQ_N;
        Rs[e] = k <= r ? X[r * CQ_GLD + k] * rds[k] : 0.f;
      }
    }
    cl.sync();
    if (rank != 0) {
      const float4* R0 = reinterpret_cast<const float4*>(cl.map_shared_rank(Rs, 0));
      for (int e = t; e < CQ_N * CQ_N / 4; e += CQ_THREADS) reinterpret_cast<float4*>(Rs)[e] = R0[e];
    }
    // CTA 0's arrays change only after every copy (and, on the last pass,
    // CTA 0 exits only after them)
    cl.sync();
    // ---- Z <- Z R^{-1}, 128 rows at a time: thread (rg, cg) owns rows
    // rb + rg + 32 i (i < 4) and columns 8 cg .. 8 cg + 7
    {
      const int rg = t >> 3, cgi = t & 7;
      for (int rb = 0; rb < rows_per; rb += 128) {
        float acc[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 4
        for (int k = 0; k < CQ_N; ++k) {
          const float4 ra = *reinterpret_cast<const float4*>(Rs + k * CQ_N + 8 * cgi);
          const float4 rb4 = *reinterpret_cast<const float4*>(Rs + k * CQ_N + 8 * cgi + 4);
          const float rv[8] = {ra.x, ra.y, ra.z, ra.w, rb4.x, rb4.y, rb4.z, rb4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = rb + rg + 32 * i;
            const float z = r < rows_per ? Z[r * CQ_ZLD + k] : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(z, rv[j], acc[i][j]);
          }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rb + rg + 32 * i;
          if (r < rows_per) {
            *reinterpret_cast<float4*>(Z + r * CQ_ZLD + 8 * cgi) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            *reinterpret_cast<float4*>(Z + r * CQ_ZLD + 8 * cgi + 4) =
                make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
          }
        }
        __syncthreads();
      }
    }
  }
  // ---- the orthonormal rows out
  float* dst = reinterpret_cast<float*>(pb + a.dst);
  for (int e = t; e < nr * (CQ_N / 4); e += CQ_THREADS) {
    const int r = e / (CQ_N / 4), c4 = e % (CQ_N / 4);
    *reinterpret_cast<float4*>(dst + (size_t)(r0 + r) * CQ_N + 4 * c4) =
        *reinterpret_cast<const float4*>(Z + r * CQ_ZLD + 4 * c4);
  }
  // the power step's operand: V^T (64 x T) and its tf32 low part
  if (a.vt) {
    float* vh = reinterpret_cast<float*>(pb + a.vt);
    float* vl = vh + (size_t)a.T * CQ_N;
    for (int e = t; e < CQ_N * nr; e += CQ_THREADS) {
      const int n = e / nr, r = e % nr;
      const float v = Z[r * CQ_ZLD + n];
      vh[(size_t)n * a.T + r0 + r] = v;
      vl[(size_t)n * a.T + r0 + r] = v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
    }
  }
  if (rank == 0 && t == 0 && *bad) atomicOr(reinterpret_cast<int*>(pb + a.o_status), ST_NOTPD);
}

}  // namespace

namespace {

template <int NC>
jolt_status launch_cq(const CqArgs& a, int np, cudaStream_t st) {
  const int rows = (a.T + NC - 1) / NC;
  const size_t smem = cq_smem(rows);
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(cholqr_cluster_kernel<NC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)cq_smem(CQ_MAXROWS)));
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NC, np);
  cfg.blockDim = dim3(CQ_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = NC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  JOLT_CUDA_TRY(cudaLaunchKernelEx(&cfg, cholqr_cluster_kernel<NC>, a));
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

int sm_count_cq() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 1;
  }
  return n;
}

// the cluster width for np problems: every problem's cluster resident at
// once (a problem holds its SMs for the whole call), else 0 (unfused path)
int cq_width(int T, int np) {
  const int sms = sm_count_cq();
  if ((T + 7) / 8 <= CQ_MAXROWS && np * 8 <= sms) return 8;
  if ((T + 3) / 4 <= CQ_MAXROWS && np * 4 <= sms) return 4;
  if ((T + 1) / 2 <= CQ_MAXROWS && np * 2 <= sms) return 2;
  return 0;
}

}  // namespace

bool cholqr_fused_supported(int T, int Lw, int np) {
  return Lw == CQ_N && T > 0 && np > 0 && cq_width(T, np) > 0;
}

jolt_status cholqr_fused(char* base, size_t stride, int np, size_t src, size_t dst,
                         size_t o_status, const int* skip, long long sk_s, int T, int passes,
                         float shift, cudaStream_t st, size_t vt) {
  if (np <= 0) return JOLT_OK;
  const int nc = cq_width(T, np);
  if (nc == 0 || passes < 1 || np > 65535) return JOLT_ERR_INVALID;
  CqArgs a;
  a.base = base; a.stride = stride; a.src = src; a.dst = dst; a.vt = vt; a.o_status = o_status;
  a.skip = skip; a.sk_s = sk_s; a.T = T; a.passes = passes; a.shift = shift;
  if (nc == 8) return launch_cq<8>(a, np, st);
  if (nc == 4) return launch_cq<4>(a, np, st);
  return launch_cq<2>(a, np, st);
}

}  // namespace jolt
