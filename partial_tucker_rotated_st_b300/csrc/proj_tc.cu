// Feature-mode projection Y = X U_d[:, :RD] on the 5th-generation tensor
// cores, for bf16 X with D = 128.
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
// One CTA covers one 128-token tile of HB heads of one unit; X tiles and the
// split factor arrive by TMA (128-byte swizzle).  The epilogue (one thread per
// token row) writes, per head, Y16 = fp16(Y) [H][T][RD] and, when asked, Y in
// fp32 [H][T][RD]; and the token-Gram relayout Yt[t][j H + h] with its tf32
// low part, HB consecutive heads per store, staged through shared memory.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

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
__global__ void __launch_bounds__(PJ_THREADS, 1)
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
  // ---- Yt[t][j H + h0 .. h0 + HB - 1] and its tf32 low part
  if (a.o_Yt && in) {
    const size_t K = (size_t)RD * a.H;
    float* yt = (float*)(wu + a.o_Yt) + (size_t)row * K + h0;
    float* ytl = yt + (size_t)a.T * K;
#pragma unroll 4
    for (int j = 0; j < RD; ++j) {
      float v[HB], l[HB];
#pragma unroll
      for (int i = 0; i < HB; ++i) {
        v[i] = stg[j * HB + i];
        l[i] = v[i] - __uint_as_float(__float_as_uint(v[i]) & 0xFFFFE000u);
      }
      if (HB == 4) {
        *reinterpret_cast<float4*>(yt + (size_t)j * a.H) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(ytl + (size_t)j * a.H) = make_float4(l[0], l[1], l[2], l[3]);
      } else if (HB == 2) {
        *reinterpret_cast<float2*>(yt + (size_t)j * a.H) = make_float2(v[0], v[1]);
        *reinterpret_cast<float2*>(ytl + (size_t)j * a.H) = make_float2(l[0], l[1]);
      } else {
        yt[(size_t)j * a.H] = v[0];
        ytl[(size_t)j * a.H] = l[0];
      }
    }
  }
  if (!ok) atomicOr((int*)(wu + a.o_status), ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
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
  const int tiles = (L.T + PJ_ROWS - 1) / PJ_ROWS;
  if (L.H % 4 == 0) return launch_proj<4>(dim3(tiles, L.H / 4, U), tX, tB, a, st);
  if (L.H % 2 == 0) return launch_proj<2>(dim3(tiles, L.H / 2, U), tX, tB, a, st);
  return launch_proj<1>(dim3(tiles, L.H, U), tX, tB, a, st);
}

}  // namespace jolt
