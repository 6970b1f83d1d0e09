// Decoder on the tensor cores (D = 128): X^ = X~ + Q^T (s * codes) for one
// 128-token tile of one head per CTA.
//
// ["Rotated Tucker residual for outlier-resistant KV quantization",
//  Implementation notes: decode by multiplying the codes by s, applying the
//  inverse orthogonal transform and adding X~.  "Joint Tucker-rank and
//  residual-bit KV allocator", Formulas: X~ = G x_2 U_T x_3 U_d.]
//
// Both parts are matrix products on tcgen05 with TMEM accumulators:
//   residual   R = codes (128 x 128, fp16, exact small integers)
//                  x (H diag(sigma))^T (fp16, exact +-1)      kind::f16
//              -> exact integer sums in fp32; x^ gets s_t R / sqrt(D);
//   low rank   r_T < T, r_d < D:  Z = U_T G_h (tf32, fp16 values exact),
//                                 X~ = (Z_hi + Z_lo) U_d^T (tf32 split)
//              r_T < T, r_d = D:  X~ = U_T G_h
//              r_T = T, r_d < D:  X~ = G_h[t] U_d^T
//              r_T = T, r_d = D:  X~ = G_h[t] (fp16(X)), no product.
// The codes are unpacked by placing each b-bit code in the mantissa of the
// fp16 1024 (0x6400 | u = 1024 + u) and subtracting 1024 + 2^(b-1) in
// half2 arithmetic; a 32-bit word of codes is split into its byte lanes, so
// within a word the codes reach the K index in an order that depends on b,
// and the rows of H diag(sigma) are built in the same order.  The epilogue
// (one thread per token row) reads both accumulators from TMEM, adds them
// and stages the tile in shared memory for coalesced stores.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

#include <string.h>

namespace jolt {

namespace {

constexpr int DT_ROWS = 128, DT_THREADS = 256, DT_D = 128;
constexpr int DT_ATOM = 128 * 128;          // 128 rows x 128 bytes, one swizzle block
constexpr int DT_MAX_UNITS = 32;

struct DecTcUnit {
  int rT, rd, b, pad;
  unsigned long long off_UT, off_Ud, off_G, off_scale, off_codes;
};
struct DecTcArgs {
  int H, T, out_dtype, u0;
  const char* blob;
  unsigned long long stride;
  void* xhat;
  DecTcUnit un[DT_MAX_UNITS];
};

__device__ __forceinline__ uint32_t sw128(int r, int byte) {
  return (uint32_t)(r * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15)));
}

// 16 fp32 TMEM columns of this thread's lane, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns of this thread's TMEM lane, issued without waiting.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}
// Wait for this thread's TMEM loads, tied to the registers they fill.
__device__ __forceinline__ void tmem_ld_wait2(uint32_t (&r)[16], uint32_t (&q)[16]) {
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

// tf32 operand element (row, k): K-major rows of KW fp32, 32 per swizzle atom.
__device__ __forceinline__ float* tf32_at(unsigned char* op, int row, int k) {
  return reinterpret_cast<float*>(op + (k >> 5) * DT_ATOM + sw128(row, (k & 31) * 4));
}

// A row of KW values v[k] = src[k * step] (k < n, else 0), every load issued
// before any is used; then stored as tf32 row `row` of an operand.
template <int KW>
__device__ __forceinline__ void load_row(__half (&v)[KW], const __half* src, long long step, int n,
                                         bool valid) {
#pragma unroll
  for (int k = 0; k < KW; ++k) v[k] = (valid && k < n) ? src[k * step] : __float2half(0.f);
}
template <int KW>
__device__ __forceinline__ void store_row(unsigned char* op, int row, const __half (&v)[KW]) {
#pragma unroll
  for (int k = 0; k < KW; k += 4)
    *reinterpret_cast<float4*>(tf32_at(op, row, k)) =
        make_float4(__half2float(v[k]), __half2float(v[k + 1]), __half2float(v[k + 2]),
                    __half2float(v[k + 3]));
}
template <int KW>
__device__ __forceinline__ void gather_row(unsigned char* op, int row, const __half* src,
                                           long long step, int n, bool valid) {
  __half v[KW];
  load_row<KW>(v, src, step, n, valid);
  store_row<KW>(op, row, v);
}

__host__ __device__ constexpr uint32_t idesc_f16h(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);   // fp16 A, B
}
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Residual operands of one row for K positions [64 half, 64 half + 64):
// codes (A, fp16) of token row `row` and row d = r of H diag(sigma) (B), in
// the K order of the unpacked words (position p of a word of 32 / B codes
// holds code (p % 4) (8 / B) + p / 4 of that word).  sgn: the 16-entry
// table of four fp16 +-1 values for each 4-bit sign pattern.
template <int B>
__device__ __forceinline__ void build_residual(unsigned char* sC, unsigned char* sH, int r,
                                               int half, const uint4 (&cq)[4], bool in,
                                               const unsigned char* sb, const uint2* sgn) {
  constexpr int PER = 32 / B, M = 8 / B, NW = 64 * B / 32;   // words in 64 codes
  constexpr uint32_t MASK = B == 8 ? 0xFFFFFFFFu : (B == 4 ? 0x0F0F0F0Fu : 0x03030303u);
  constexpr uint32_t BIAS = 0x64006400u | (1u << (B - 1)) | (1u << (B - 1 + 16));
  const uint32_t bias = BIAS;
  const __half2 off2 = *reinterpret_cast<const __half2*>(&bias);
  uint32_t w[NW];
#pragma unroll
  for (int q = 0; q < NW / 4; ++q) {
    w[4 * q] = cq[q].x; w[4 * q + 1] = cq[q].y; w[4 * q + 2] = cq[q].z; w[4 * q + 3] = cq[q].w;
  }
#pragma unroll
  for (int wi = 0; wi < NW; ++wi)
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const uint32_t x = (w[wi] >> (i * B)) & MASK;
      uint32_t lo = __byte_perm(x, 0x64646464u, 0x5140);   // halves 0x64|lane0, 0x64|lane1
      uint32_t hi = __byte_perm(x, 0x64646464u, 0x7362);
      const __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), off2);
      const __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), off2);
      const int k = 64 * half + wi * PER + 4 * i;
      uint2 v;
      v.x = in ? *reinterpret_cast<const uint32_t*>(&l2) : 0u;
      v.y = in ? *reinterpret_cast<const uint32_t*>(&h2) : 0u;
      *reinterpret_cast<uint2*>(sC + (k >> 6) * DT_ATOM + sw128(r, (k & 63) * 2)) = v;
    }
  // H diag(sigma), row d = r: neg(k) = parity(d & c(k)) ^ sigma_d; c(k) =
  // word base + local code, and the parity splits over the two
  const int d = r;
  const uint32_t sneg = (sb[d >> 3] >> (d & 7)) & 1u;
  uint32_t loc = 0;                               // parity(d & local code) per position
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int c = (p & 3) * M + (p >> 2);
    loc |= (uint32_t)(__popc(d & c) & 1) << p;
  }
#pragma unroll
  for (int wi = 0; wi < 64 / PER; ++wi) {
    const int k0 = 64 * half + wi * PER;        // word base = k0 (codes k0 .. k0 + PER - 1)
    const uint32_t flip = ((__popc(d & k0) & 1) ^ sneg) ? 0xFFFFFFFFu : 0u;
    const uint32_t neg = loc ^ flip;
#pragma unroll
    for (int p = 0; p < PER; p += 4) {
      const int k = k0 + p;
      const uint2 v = sgn[(neg >> p) & 15u];
      *reinterpret_cast<uint2*>(sH + (k >> 6) * DT_ATOM + sw128(d, (k & 63) * 2)) = v;
    }
  }
}

template <int KW>
__global__ void __launch_bounds__(DT_THREADS, KW == 32 ? 2 : 1) decode_tc_kernel(const __grid_constant__ DecTcArgs a) {
  constexpr int NCH = KW / 32;                 // swizzle atoms per tf32 row
  extern __shared__ __align__(1024) unsigned char dtc_raw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)dtc_raw + 1023) & ~(uintptr_t)1023);
  // region R: the residual operands (codes, H diag(sigma)); once the
  // residual product is done, Z hi / Z lo / U_d of the second stage (mode 0)
  // and at the end the output staging
  unsigned char* sC = base;                    // codes, fp16 [128 rows][128], 2 atoms
  unsigned char* sH = sC + 2 * DT_ATOM;        // H diag(sigma), fp16 [128 d][128], 2 atoms
  unsigned char* sA = sH + 2 * DT_ATOM;        // tf32 A of the first product [128 rows][KW]
  unsigned char* sX = sA + NCH * DT_ATOM;      // tf32 B of the first product
  unsigned char* sZh = sC;                     // mode 0, second stage: Z hi, Z lo, U_d rows
  unsigned char* sZl = sC + NCH * DT_ATOM;
  unsigned char* sU = sC + 2 * NCH * DT_ATOM;
  struct Bars { uint64_t mma; uint32_t tmem; uint2 sgn[16]; };
  Bars* S = reinterpret_cast<Bars*>(sX + NCH * DT_ATOM);
  const int tile = blockIdx.x, h = blockIdx.y, uz = blockIdx.z;
  const int u = a.u0 + uz;
  const DecTcUnit du = a.un[uz];
  // two threads per token row: r = the row (and the TMEM lane), half = which
  // half of the K range / the output columns
  const int t = threadIdx.x, warp = t >> 5, r = t & (DT_ROWS - 1), half = t >> 7;
  const int T = a.T, H = a.H;
  const int t0 = tile * DT_ROWS, row = t0 + r;
  const bool in = row < T;
  const char* blob = a.blob + (unsigned long long)u * a.stride;
  const int rT = du.rT, rd = du.rd, b = du.b;
  const bool fullT = (rT == T), fullD = (rd == DT_D);
  // 0: Z = U_T G_h then Z U_d^T; 1: U_T G_h; 2: G rows U_d^T; 3: G rows as X~
  const int mode = fullT ? (fullD ? 3 : 2) : (fullD ? 1 : 0);
  const int kz = fullT ? rd : rT;              // K of the product into X~ (modes 1, 2)
  const int k8 = (kz + 7) & ~7;
  const int rT8 = (rT + 7) & ~7, rd8 = (rd + 7) & ~7, rd16 = (rd + 15) & ~15;

  // ---- every global read of the CTA issued first: this thread's half row of
  // codes, its scale, the rows it gathers for the low-rank operands
  const __half* UT = reinterpret_cast<const __half*>(blob + du.off_UT);
  const __half* Ud = reinterpret_cast<const __half*>(blob + du.off_Ud);
  const __half* G = reinterpret_cast<const __half*>(blob + du.off_G);
  const __half* Gh = G + (size_t)h * rT * rd;
  uint4 cq[4];                                 // up to 64 bytes of codes
  {
    const uint4* cw = reinterpret_cast<const uint4*>(
        blob + du.off_codes + ((unsigned long long)h * T + (in ? row : 0)) * (DT_D * b / 8) +
        half * (8 * b));
#pragma unroll
    for (int q = 0; q < 4; ++q)
      cq[q] = (b > 0 && in && q < b / 2) ? cw[q] : make_uint4(0, 0, 0, 0);
  }
  const float s = (b > 0 && in) ? __half2float(reinterpret_cast<const __half*>(blob + du.off_scale)
                                                   [(size_t)h * T + row]) * rsqrtf((float)DT_D)
                                : 0.f;
  __half g1[KW], g2[KW];   // first-product operand row; mode 0: the U_d row of the second
  if (mode == 0 || mode == 1) {
    if (half == 0) load_row<KW>(g1, UT + (size_t)(in ? row : 0) * rT, 1, rT, in);
    else if (mode == 0) load_row<KW>(g1, Gh + (r < rd ? r : 0), rd, rT, r < rd);
    else load_row<KW>(g1, Gh + r, DT_D, rT, true);
  } else if (mode == 2) {
    if (half == 0) load_row<KW>(g1, G + ((size_t)h * T + (in ? row : 0)) * rd, 1, rd, in);
    else load_row<KW>(g1, Ud + (size_t)r * rd, 1, rd, true);
  }
  if (mode == 0 && half == 1) load_row<KW>(g2, Ud + (size_t)r * rd, 1, rd, true);

  if (t == 0) {
    tc::mbar_init(tc::smem_u32(&S->mma), 1);
    tc::fence_barrier_init();
  }
  if (t < 16) {
    uint32_t v[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      v[j] = (0x3C00u | (((uint32_t)t >> (2 * j)) & 1u) << 15) |
             ((0x3C00u | (((uint32_t)t >> (2 * j + 1)) & 1u) << 15) << 16);
    S->sgn[t] = make_uint2(v[0], v[1]);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&S->tmem), 256);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  bool ok = true;
  uint32_t phase = 0;
  auto mma_wait = [&]() {
    if (!tc::mbar_wait(tc::smem_u32(&S->mma), phase & 1)) ok = false;
    ++phase;
    tc::tc_fence_after();
  };

  // ---- residual operands: codes (A) and H diag(sigma) (B), fp16
  if (b > 0) {
    const unsigned char* sb = reinterpret_cast<const unsigned char*>(blob) + 88;
    if (b == 2) build_residual<2>(sC, sH, r, half, cq, in, sb, S->sgn);
    else if (b == 4) build_residual<4>(sC, sH, r, half, cq, in, sb, S->sgn);
    else build_residual<8>(sC, sH, r, half, cq, in, sb, S->sgn);
  }

  // ---- low-rank operands of the first product: A = sA (half 0), B = sX (half 1)
  if (mode == 0) {
    if (half == 0) store_row<KW>(sA, r, g1);
    else if (r < rd16) store_row<KW>(sX, r, g1);   // B rows j < rd16: G_h[k][j]
  } else if (mode == 1 || mode == 2) {
    store_row<KW>(half == 0 ? sA : sX, r, g1);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();

  // ---- residual into TMEM [0, 128); the first low-rank product into
  // [128, ...): X~ itself (modes 1, 2) or Z = U_T G_h (mode 0)
  const bool any = (b > 0) || mode != 3;
  if (t == 0 && any) {
    tc::tc_fence_after();
    if (b > 0) {
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sC + kc * DT_ATOM) + 32 * k, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sH + kc * DT_ATOM) + 32 * k, 16, 1024);
          tc::mma_f16(tmem, ad, bd, idesc_f16h(128, 128), (kc | k) != 0);
        }
    }
    if (mode != 3) {
      const int kk_n = (mode == 0 ? rT8 : k8) / 8;
      const uint32_t id = idesc_tf32(128, mode == 0 ? rd16 : 128);
      for (int kk = 0; kk < kk_n; ++kk) {
        const uint32_t off = (kk >> 2) * DT_ATOM;
        const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + off) + 32 * (kk & 3), 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sX + off) + 32 * (kk & 3), 16, 1024);
        tc::mma_tf32(tmem + 128, ad, bd, id, kk != 0);
      }
    }
    tc::mma_commit(tc::smem_u32(&S->mma));
  }
  if (any) mma_wait();

  // ---- mode 0, second stage: X~ = (Z hi + Z lo) U_d^T into [128, 256)
  if (mode == 0) {
    // half 0: the Z row -> tf32 hi and lo (K = r_d); half 1: U_d row d = r;
    // both over the residual's operands (its product is done)
    if (half == 0) {
      for (int c = 0; c < rd16; c += 16) {
        float z[16];
        tmem_ld16(trow + 128 + c, z);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          float4 hi, lo;
          float* ph = reinterpret_cast<float*>(&hi);
          float* pl = reinterpret_cast<float*>(&lo);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = (c + i + e < rd) ? z[i + e] : 0.f;
            const float vh = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
            ph[e] = vh;
            pl[e] = v - vh;
          }
          if (c + i < rd8) {
            *reinterpret_cast<float4*>(tf32_at(sZh, r, c + i)) = hi;
            *reinterpret_cast<float4*>(tf32_at(sZl, r, c + i)) = lo;
          }
        }
      }
    } else {
      store_row<KW>(sU, r, g2);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc::tc_fence_after();
      for (int kk = 0; kk < rd8 / 8; ++kk) {
        const uint32_t off = (kk >> 2) * DT_ATOM;
        const uint64_t ah = tc::sdesc_sw128(tc::smem_u32(sZh + off) + 32 * (kk & 3), 16, 1024);
        const uint64_t al = tc::sdesc_sw128(tc::smem_u32(sZl + off) + 32 * (kk & 3), 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sU + off) + 32 * (kk & 3), 16, 1024);
        tc::mma_tf32(tmem + 128, ah, bd, idesc_tf32(128, 128), kk != 0);
        tc::mma_tf32(tmem + 128, al, bd, idesc_tf32(128, 128), 1);
      }
      tc::mma_commit(tc::smem_u32(&S->mma));
    }
    mma_wait();
  }

  // ---- epilogue: x^ = X~ + s R / sqrt(D) for columns [64 half, 64 half + 64)
  // of row r, staged row-major (padded rows)
  const bool f32 = (a.out_dtype == JOLT_F32);
  const int rowb = f32 ? DT_D * 4 + 16 : DT_D * 2 + 16;   // staging row stride (bytes)
  unsigned char* stg = sC;                                 // no operand is read any more
  const __half* Grow = G + ((size_t)h * T + (in ? row : 0)) * DT_D;
  for (int c = 64 * half; c < 64 * half + 64; c += 16) {
    uint32_t lu[16], ru[16];
    if (mode != 3) tmem_ld16_issue(trow + 128 + c, lu);
    if (b > 0) tmem_ld16_issue(trow + c, ru);
    if (mode != 3 || b > 0) tmem_ld_wait2(lu, ru);
    float lr[16], rr[16];
    if (mode != 3) {
#pragma unroll
      for (int i = 0; i < 16; ++i) lr[i] = __uint_as_float(lu[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; i += 8) {
        const uint4 raw = in ? *reinterpret_cast<const uint4*>(Grow + c + i) : make_uint4(0, 0, 0, 0);
        const __half* hv = reinterpret_cast<const __half*>(&raw);
#pragma unroll
        for (int e = 0; e < 8; ++e) lr[i + e] = __half2float(hv[e]);
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) rr[i] = __uint_as_float(ru[i]);
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (b > 0) ? fmaf(s, rr[i], lr[i]) : lr[i];
    if (!ok) {
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __int_as_float(0x7fc00000);   // a timed-out tile reads NaN
    }
    if (f32) {
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(stg + r * rowb + (c + i) * 4) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
    } else {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        pk[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
      *reinterpret_cast<uint4*>(stg + r * rowb + c * 2) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(stg + r * rowb + c * 2 + 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
  // coalesced copy-out of the tile's rows < T
  const int rowbytes = f32 ? DT_D * 4 : DT_D * 2;
  const int per_row = rowbytes / 16;
  const int nrows = min(DT_ROWS, T - t0);
  char* out = reinterpret_cast<char*>(a.xhat) +
              (((size_t)u * H + h) * T + t0) * (size_t)rowbytes;
  for (int i = t; i < nrows * per_row; i += DT_THREADS) {
    const int rr = i / per_row, c16 = i % per_row;
    *reinterpret_cast<uint4*>(out + (size_t)rr * rowbytes + c16 * 16) =
        *reinterpret_cast<const uint4*>(stg + rr * rowb + c16 * 16);
  }
}

template <int KW>
jolt_status launch_dtc(dim3 grid, const DecTcArgs& a, cudaStream_t st) {
  constexpr int NCH = KW / 32;
  const size_t smem = 1024 + 4 * DT_ATOM + 2 * NCH * DT_ATOM + 256;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(decode_tc_kernel<KW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  decode_tc_kernel<KW><<<grid, DT_THREADS, smem, st>>>(a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace

bool decode_tc_supported(int D) { return D == DT_D; }

jolt_status decode_tc_run(int U, const jolt_blob_desc* desc, const char* blob, size_t stride,
                          void* xhat, int out_dtype, cudaStream_t st) {
  const int H = desc[0].H, T = desc[0].T;
  for (int u0 = 0; u0 < U; u0 += DT_MAX_UNITS) {
    const int nu = (U - u0) < DT_MAX_UNITS ? (U - u0) : DT_MAX_UNITS;
    DecTcArgs a;
    memset(&a, 0, sizeof(a));
    a.H = H; a.T = T; a.out_dtype = out_dtype; a.u0 = u0; a.blob = blob; a.stride = stride;
    a.xhat = xhat;
    int kmax = 0;
    for (int i = 0; i < nu; ++i) {
      const jolt_blob_desc& d = desc[u0 + i];
      a.un[i].rT = d.rT; a.un[i].rd = d.rd; a.un[i].b = d.b;
      a.un[i].off_UT = d.off_UT; a.un[i].off_Ud = d.off_Ud; a.un[i].off_G = d.off_G;
      a.un[i].off_scale = d.off_scale; a.un[i].off_codes = d.off_codes;
      if (d.rT < T) kmax = kmax > d.rT ? kmax : d.rT;
      if (d.rd < DT_D) kmax = kmax > d.rd ? kmax : d.rd;
    }
    const dim3 grid((T + DT_ROWS - 1) / DT_ROWS, H, nu);
    const jolt_status s = kmax <= 32 ? launch_dtc<32>(grid, a, st) : launch_dtc<64>(grid, a, st);
    if (s != JOLT_OK) return s;
  }
  return JOLT_OK;
}

}  // namespace jolt
