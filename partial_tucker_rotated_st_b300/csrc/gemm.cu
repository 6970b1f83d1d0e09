// Strided, batched, segment-summed fp32 GEMM on CUDA cores.
//
// Used for the small and oddly-strided contractions of the factor step
// (projections, cores, Rayleigh-Ritz products).  Operands may be fp32, bf16 or
// fp16 (converted exactly to fp32 on load); accumulation is fp32.
#include "jolt_internal.cuh"

namespace jolt {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename TA, typename TB>
__global__ void __launch_bounds__(NT) gemm_kernel(GemmDesc g) {
  const int b = blockIdx.z;
  const int b1 = b / g.nb2, b2 = b % g.nb2;
  if (g.skip && g.skip[b1 * g.skip_stride]) return;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const TA* A = (const TA*)g.A.p + b1 * g.A.sb1 + b2 * g.A.sb2;
  const TB* B = (const TB*)g.B.p + b1 * g.B.sb1 + b2 * g.B.sb2;

  // two stages: the next tile's global loads are in flight (in registers)
  // while the current tile is multiplied
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];

  const int t = threadIdx.x;
  const int tx = t % 16, ty = t / 16;
  const bool a_kfast = (g.A.s1 == 1);
  const bool b_nfast = (g.B.s1 == 1);

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  const int ktiles = (g.K + BK - 1) / BK;
  const int total = ktiles * g.nseg;
  float ra[4], rb[4];
  auto load = [&](int it) {
    const int s = it / ktiles;
    const int k0 = (it % ktiles) * BK;
    const TA* As_g = A + s * g.A.sseg;
    const TB* Bs_g = B + s * g.B.sseg;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = t + i * NT;
      int m, k;
      if (a_kfast) { m = e / BK; k = e % BK; } else { m = e % BM; k = e / BM; }
      const int gm = m0 + m, gk = k0 + k;
      ra[i] = (gm < g.M && gk < g.K) ? to_f32(As_g[gm * g.A.s0 + gk * g.A.s1]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = t + i * NT;
      int k, n;
      if (b_nfast) { k = e / BN; n = e % BN; } else { n = e / BK; k = e % BK; }
      const int gk = k0 + k, gn = n0 + n;
      rb[i] = (gk < g.K && gn < g.N) ? to_f32(Bs_g[gk * g.B.s0 + gn * g.B.s1]) : 0.f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = t + i * NT;
      int m, k;
      if (a_kfast) { m = e / BK; k = e % BK; } else { m = e % BM; k = e / BM; }
      As[buf][k][m] = ra[i];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = t + i * NT;
      int k, n;
      if (b_nfast) { k = e / BN; n = e % BN; } else { n = e / BK; k = e % BK; }
      Bs[buf][k][n] = rb[i];
    }
  };
  load(0);
  store(0);
  __syncthreads();
  for (int it = 0; it < total; ++it) {
    const int buf = it & 1;
    if (it + 1 < total) load(it + 1);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
      const float4 bb = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (it + 1 < total) store(buf ^ 1);
    __syncthreads();
  }

  float* C = g.C + b1 * g.cb1 + b2 * g.cb2;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= g.N) continue;
      float* c = C + gm * g.cm + gn * g.cn;
      float v = g.alpha * acc[i][j];
      if (g.beta != 0.f) v = fmaf(g.beta, *c, v);
      *c = v;
    }
  }
}

template <typename TA>
jolt_status launch_b(const GemmDesc& g, dim3 grid, cudaStream_t st) {
  switch (g.B.dtype) {
    case JOLT_F32: gemm_kernel<TA, float><<<grid, NT, 0, st>>>(g); break;
    case JOLT_BF16: gemm_kernel<TA, __nv_bfloat16><<<grid, NT, 0, st>>>(g); break;
    case JOLT_F16: gemm_kernel<TA, __half><<<grid, NT, 0, st>>>(g); break;
    default: return JOLT_ERR_INVALID;
  }
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace

jolt_status launch_gemm(const GemmDesc& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.nseg <= 0 || g.nb1 <= 0 || g.nb2 <= 0)
    return JOLT_OK;
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, g.nb1 * g.nb2);
  if (grid.z > 65535 || grid.y > 65535) return JOLT_ERR_INVALID;
  switch (g.A.dtype) {
    case JOLT_F32: return launch_b<float>(g, grid, st);
    case JOLT_BF16: return launch_b<__nv_bfloat16>(g, grid, st);
    case JOLT_F16: return launch_b<__half>(g, grid, st);
    default: return JOLT_ERR_INVALID;
  }
}

}  // namespace jolt
