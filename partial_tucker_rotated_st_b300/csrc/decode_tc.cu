// Decoder on the tensor cores (D = 128): X^ = X~ + Q^T (s * codes), every
// 128-token tile of every head of a batch of units.
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
//   low rank   r_T < T, r_d < D:  X~ = U_T W_h, W_h = G_h U_d^T (fp32 sums
//                                 of exact fp16 products, split tf32 hi + lo)
//              r_T < T, r_d = D:  X~ = U_T G_h (fp16 values, exact in tf32)
//              r_T = T, r_d < D:  X~ = G_h[t] U_d^T
//              r_T = T, r_d = D:  X~ = G_h[t] (fp16(X)), no product.
// The codes are unpacked by placing each b-bit code in the mantissa of the
// fp16 1024 (0x6400 | u = 1024 + u) and subtracting 1024 + 2^(b-1) in
// half2 arithmetic; a 32-bit word of codes is split into its byte lanes, so
// within a word the codes reach the K index in an order that depends on b,
// and the rows of H diag(sigma) are built in the same order.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

#include <string.h>

namespace jolt {

namespace {

constexpr int DT_ROWS = 128, DT_D = 128;
constexpr int DT_ATOM = 128 * 128;          // 128 rows x 128 bytes, one swizzle block
constexpr int DT_MAX_UNITS = 32;

struct DecTcUnit {
  int rT, rd, b, pad;
  unsigned long long off_UT, off_Ud, off_G, off_scale, off_codes;
};
struct DecTcArgs {
  int H, T, out_dtype, u0, nu;
  const char* blob;
  unsigned long long stride;
  void* xhat;
  DecTcUnit un[DT_MAX_UNITS];
};

__device__ __forceinline__ uint32_t sw128(int r, int byte) {
  return (uint32_t)(r * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15)));
}

// 32 columns of this thread's TMEM lane, issued without waiting.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t addr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(addr));
}
// Wait for this thread's TMEM loads, tied to the 32 registers of one load.
__device__ __forceinline__ void tmem_ld_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
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
                                               const unsigned char* sb, const uint2* sgn,
                                               bool codes = true, bool signs = true) {
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
  if (codes)
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
  if (!signs) return;
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


// ------------------------------------------------------------------ kernel
// One persistent CTA per SM walks a contiguous range of 128-token tiles
// (unit-major, then head, then token tile), two tiles in flight:
//   warps 0-7  (two threads per tile row) stage tile n's operands in shared
//              memory stage n % 2: the row's codes unpacked to fp16, its
//              low-rank row (a U_T row, or a G row for r_T = T) as tf32; and,
//              when the unit or head changes, the B operands: H diag(sigma)
//              (per unit and bit width) and the low-rank factor (per head:
//              W_h = G_h U_d^T split tf32 hi + lo; G_h; or U_d);
//   warp 8     issues tile n's products into TMEM buffer n % 2 (residual,
//              256 columns per buffer: [0, 128) the codes times H diag(sigma),
//              [128, 256) the low-rank rebuild);
//   warps 9-16 read buffer n % 2 (two threads per row, 64 columns each), form
//              x^ = X~ + (s_t / sqrt(D)) R and write the row.
// Hand-offs by mbarriers: full (stage written), empty (the stage's products
// done), tfull (buffer written), tempty (buffer read).  Every wait is
// bounded; a wait that gives up sets the decoder's status word and the
// tile's output reads NaN.
constexpr int DP_THREADS = 544;

__device__ int g_decode_status;   // ST_* bits of decoder waits that gave up

struct DpBars {
  uint64_t full[2], empty[2], tfull[2], tempty[2];
  uint32_t tmem;
  uint2 sgn[16];
};

template <int KW>
struct DpLayout {
  static constexpr int NCH = KW / 32;                     // swizzle atoms per tf32 row
  static constexpr int STAGE = 2 * DT_ATOM + NCH * DT_ATOM;   // codes fp16, low-rank A
  static constexpr int O_HS = 2 * STAGE;                   // H diag(sigma), 2 atoms
  static constexpr int O_LBH = O_HS + 2 * DT_ATOM;         // low-rank B hi
  static constexpr int O_LBL = O_LBH + NCH * DT_ATOM;      // low-rank B lo
  static constexpr int O_BARS = O_LBL + NCH * DT_ATOM;
  // bf16 output staging for the TMA stores, two tiles (KW = 32 only: the
  // 64-wide operands leave no room, and that variant stores directly)
  static constexpr bool STAGED = KW == 32;
  static constexpr int O_OUT = O_BARS + 1024;
  static constexpr int BYTES = O_OUT + (STAGED ? 2 * 2 * DT_ATOM : 0) + 1024;
};

__device__ __forceinline__ int dp_mode(int rT, int rd, int T) {
  // 0: U_T W_h (both truncated); 1: U_T G_h (r_d = D); 2: G rows U_d^T
  // (r_T = T); 3: G rows themselves
  return rT == T ? (rd == DT_D ? 3 : 2) : (rd == DT_D ? 1 : 0);
}

template <int KW>
__global__ void __launch_bounds__(DP_THREADS, 1)
decode_tc_kernel(const __grid_constant__ DecTcArgs a, const __grid_constant__ CUtensorMap tO) {
  using LY = DpLayout<KW>;
  extern __shared__ __align__(1024) unsigned char dtc_raw[];
  unsigned char* base = dtc_raw + ((1024u - (tc::smem_u32(dtc_raw) & 1023u)) & 1023u);
  DpBars* S = reinterpret_cast<DpBars*>(base + LY::O_BARS);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int T = a.T, H = a.H;
  const int tiles_t = (T + DT_ROWS - 1) / DT_ROWS;
  const int ntot = a.nu * H * tiles_t;
  const int chunk = (ntot + gridDim.x - 1) / gridDim.x;
  const int i0 = blockIdx.x * chunk, i1 = min(ntot, i0 + chunk);
  const int nt = i1 > i0 ? i1 - i0 : 0;
  if (t == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(tc::smem_u32(&S->full[s]), 8);
      tc::mbar_init(tc::smem_u32(&S->empty[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->tfull[s]), 1);
      tc::mbar_init(tc::smem_u32(&S->tempty[s]), 8);
    }
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
  if (warp == 8) tc::tmem_alloc(tc::smem_u32(&S->tmem), 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem;
  bool ok = true;
  const float rsD = rsqrtf((float)DT_D);
  auto tile_at = [&](int n, int& u, int& h, int& tt) {
    const int i = i0 + n;
    u = i / (H * tiles_t);
    h = (i / tiles_t) % H;
    tt = i % tiles_t;
  };

  if (warp < 8) {
    // ---------------- operand staging: two threads per tile row, thread
    // (r, hf) owns half hf of the row's K range; the next tile's global
    // reads are issued before the current tile's operands are written
    const int r = t & (DT_ROWS - 1), hf = t >> 7;
    int hs_key = -1, lb_key = -1;          // what the B operands hold
    // this thread's reads of tile n: its half of the codes, its half of the
    // low-rank A row (raw fp16)
    uint4 pc[4], pa[KW / 16];
    auto fetch = [&](int n) {
      int u, h, tt;
      tile_at(n, u, h, tt);
      const DecTcUnit du = a.un[u];
      const int mode = dp_mode(du.rT, du.rd, T), b = du.b;
      const char* blob = a.blob + (unsigned long long)(a.u0 + u) * a.stride;
      const int row = tt * DT_ROWS + r;
      const bool in = row < T;
      const uint4* cw = reinterpret_cast<const uint4*>(
          blob + du.off_codes + ((unsigned long long)h * T + (in ? row : 0)) * (DT_D * b / 8));
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        pc[qq] = (b > 0 && in && qq < b / 2) ? cw[hf * (b / 2) + qq] : make_uint4(0, 0, 0, 0);
      const int K = mode == 2 ? du.rd : du.rT;
      const __half* src = mode == 2 ? reinterpret_cast<const __half*>(blob + du.off_G) +
                                          ((size_t)h * T + (in ? row : 0)) * du.rd
                                    : reinterpret_cast<const __half*>(blob + du.off_UT) +
                                          (size_t)(in ? row : 0) * du.rT;
      const int k0 = hf * (KW / 2);
      // rows start on 16-, 8- or 4-byte boundaries as K is a multiple of 8,
      // 4 or 2; the widest aligned loads land in pa without being combined,
      // so nothing waits for them until the next tile is staged
#pragma unroll
      for (int i = 0; i < KW / 16; ++i) {
        const int k = k0 + 8 * i;
        if (mode == 3 || !in || k >= K) {
          pa[i] = make_uint4(0, 0, 0, 0);
        } else if ((K & 7) == 0) {
          pa[i] = *reinterpret_cast<const uint4*>(src + k);
        } else if ((K & 3) == 0) {
          const uint2 lo = *reinterpret_cast<const uint2*>(src + k);
          const uint2 hi = k + 4 < K ? *reinterpret_cast<const uint2*>(src + k + 4) : make_uint2(0, 0);
          pa[i] = make_uint4(lo.x, lo.y, hi.x, hi.y);
        } else if ((K & 1) == 0) {
          const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src + k);
          pa[i] = make_uint4(s32[0], k + 2 < K ? s32[1] : 0u, k + 4 < K ? s32[2] : 0u,
                             k + 6 < K ? s32[3] : 0u);
        } else {
          uint32_t hw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const unsigned short lo = k + 2 * e < K ? __half_as_ushort(src[k + 2 * e]) : 0;
            const unsigned short hi = k + 2 * e + 1 < K ? __half_as_ushort(src[k + 2 * e + 1]) : 0;
            hw[e] = (uint32_t)lo | ((uint32_t)hi << 16);
          }
          pa[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
      }
    };
    if (nt > 0) fetch(0);
    for (int n = 0; n < nt; ++n) {
      int u, h, tt;
      tile_at(n, u, h, tt);
      const DecTcUnit du = a.un[u];
      const int rT = du.rT, rd = du.rd, b = du.b;
      const int mode = dp_mode(rT, rd, T);
      const char* blob = a.blob + (unsigned long long)(a.u0 + u) * a.stride;
      const int s = n & 1;
      unsigned char* sC = base + s * LY::STAGE;
      unsigned char* sA = sC + 2 * DT_ATOM;
      const int hk = b > 0 ? u * 16 + b : -1;
      const int lk = mode == 0 || mode == 1 ? u * H + h : (mode == 2 ? (1 << 30) + u : -1);
      const bool need_hs = b > 0 && hk != hs_key;
      const bool need_lb = lk >= 0 && lk != lb_key;
      // the B operands are rewritten only once every product of earlier
      // tiles is done; the stage once tile n - 2's products are
      if (n >= 1 && (need_hs || need_lb)) {
        if (!tc::mbar_wait(tc::smem_u32(&S->empty[(n - 1) & 1]), ((n - 1) >> 1) & 1)) ok = false;
      }
      if (n >= 2 && !tc::mbar_wait(tc::smem_u32(&S->empty[s]), ((n - 2) >> 1) & 1)) ok = false;
      const int row = tt * DT_ROWS + r;
      const bool in = row < T;
      const __half* Ud = reinterpret_cast<const __half*>(blob + du.off_Ud);
      const __half* G = reinterpret_cast<const __half*>(blob + du.off_G);
      const __half* Gh = G + (size_t)h * rT * rd;
      if (need_lb) {
        // low-rank B^T, K-major [n = d][k], column d = r, this thread's half
        // of k; zero past K
        unsigned char* sBh = base + LY::O_LBH;
        unsigned char* sBl = base + LY::O_LBL;
        const int d = r, kb = hf * (KW / 2);
        if (mode == 0) {
          // W_h[k][d] = sum_j G_h[k][j] U_d[d][j], split tf32 hi + lo; G_h
          // (r_T x r_d) and U_d (D x r_d) are first staged, in fp32, in this
          // stage's operand area (free: its codes and A rows come after)
          // (every global read issued before the first is used)
          constexpr int UQ = DT_D * KW / 512, GQ = KW * KW / 256;   // per-thread bounds
          __half2 ur[UQ];
          __half gr[GQ];
          const __half2* Ud2 = reinterpret_cast<const __half2*>(Ud);
#pragma unroll
          for (int i = 0; i < UQ; ++i) {
            const int e = t + 256 * i;
            ur[i] = e < DT_D * rd / 2 ? Ud2[e] : __floats2half2_rn(0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < GQ; ++i) {
            const int e = t + 256 * i;
            gr[i] = e < rT * rd ? Gh[e] : __float2half(0.f);
          }
          float* gs = reinterpret_cast<float*>(sC);
          // U_d, staged beside G_h (fp32); row d is read back as a broadcast
          float* us = gs + rT * rd;
#pragma unroll
          for (int i = 0; i < GQ; ++i)
            if (t + 256 * i < rT * rd) gs[t + 256 * i] = __half2float(gr[i]);
#pragma unroll
          for (int i = 0; i < UQ; ++i)
            if (t + 256 * i < DT_D * rd / 2) {
              const float2 f = __half22float2(ur[i]);
              us[2 * (t + 256 * i)] = f.x;
              us[2 * (t + 256 * i) + 1] = f.y;
            }
          asm volatile("bar.sync 1, 256;" ::: "memory");
          const float* udr = us + (size_t)d * rd;
          // the 4-row groups of column d alternate between the row's two
          // threads; groups past r_T are zero.  With r_d a multiple of 4 the
          // rows of G_h and U_d start on 16-byte boundaries: 4 values a load
          const bool v4 = (rd & 3) == 0;
          for (int k = 4 * hf; k < KW; k += 8) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (k < rT && v4) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (k + e < rT) {
                  const float* gr = gs + (k + e) * rd;
                  float acc = 0.f;
#pragma unroll 1
                  for (int j = 0; j < rd; j += 4) {
                    const float4 u4 = *reinterpret_cast<const float4*>(udr + j);
                    const float4 g4 = *reinterpret_cast<const float4*>(gr + j);
                    acc = fmaf(g4.x, u4.x, acc);
                    acc = fmaf(g4.y, u4.y, acc);
                    acc = fmaf(g4.z, u4.z, acc);
                    acc = fmaf(g4.w, u4.w, acc);
                  }
                  v[e] = acc;
                }
              }
            } else if (k < rT) {
              for (int j = 0; j < rd; ++j) {
                const float uj = udr[j];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (k + e < rT) v[e] = fmaf(gs[(k + e) * rd + j], uj, v[e]);
              }
            }
            float hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              hi[e] = __uint_as_float(__float_as_uint(v[e]) & 0xFFFFE000u);
              lo[e] = v[e] - hi[e];
            }
            *reinterpret_cast<float4*>(tf32_at(sBh, d, k)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<float4*>(tf32_at(sBl, d, k)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");   // the area is overwritten next
        } else {
          // exact fp16 values: G_h[k][d] (mode 1) or U_d[d][k] (mode 2)
          const int K = mode == 1 ? rT : rd;
          for (int k = kb; k < kb + KW / 2; k += 4) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int kk = k + e;
              v[e] = kk >= K ? 0.f
                             : __half2float(mode == 1 ? Gh[(size_t)kk * DT_D + d] : Ud[(size_t)d * rd + kk]);
            }
            *reinterpret_cast<float4*>(tf32_at(sBh, d, k)) = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
        lb_key = lk;
      }
      // this thread's half of the row's codes and, when the unit or bit
      // width changed, of row d = r of H diag(sigma)
      if (b > 0) {
        const unsigned char* sb = reinterpret_cast<const unsigned char*>(blob) + 88;
        unsigned char* sH = base + LY::O_HS;
        if (b == 2) build_residual<2>(sC, sH, r, hf, pc, in, sb, S->sgn, true, need_hs);
        else if (b == 4) build_residual<4>(sC, sH, r, hf, pc, in, sb, S->sgn, true, need_hs);
        else build_residual<8>(sC, sH, r, hf, pc, in, sb, S->sgn, true, need_hs);
        if (need_hs) hs_key = hk;
      }
      // this thread's half of the low-rank A row, fp16 -> tf32
      if (mode != 3) {
#pragma unroll
        for (int i = 0; i < KW / 16; ++i) {
          const __half2* hv = reinterpret_cast<const __half2*>(&pa[i]);
          const int k = hf * (KW / 2) + 8 * i;
          const float2 f0 = __half22float2(hv[0]), f1 = __half22float2(hv[1]);
          const float2 f2 = __half22float2(hv[2]), f3 = __half22float2(hv[3]);
          *reinterpret_cast<float4*>(tf32_at(sA, r, k)) = make_float4(f0.x, f0.y, f1.x, f1.y);
          *reinterpret_cast<float4*>(tf32_at(sA, r, k + 4)) = make_float4(f2.x, f2.y, f3.x, f3.y);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(&S->full[s]))
                     : "memory");
      if (n + 1 < nt) fetch(n + 1);
    }
  } else if (warp == 8) {
    // ---------------- products
    for (int n = 0; n < nt; ++n) {
      int u, h, tt;
      tile_at(n, u, h, tt);
      const DecTcUnit du = a.un[u];
      const int mode = dp_mode(du.rT, du.rd, T), b = du.b;
      const int s = n & 1;
      bool okw = tc::mbar_wait(tc::smem_u32(&S->full[s]), (n >> 1) & 1);
      if (n >= 2) okw = tc::mbar_wait(tc::smem_u32(&S->tempty[s]), ((n - 2) >> 1) & 1) && okw;
      if (!okw) ok = false;
      tc::tc_fence_after();
      if (lane == 0) {
        const uint32_t d0 = tmem + 256u * (uint32_t)s;
        const uint32_t sC = tc::smem_u32(base + s * LY::STAGE), sA = sC + 2 * DT_ATOM;
        const uint32_t sH = tc::smem_u32(base + LY::O_HS);
        const uint32_t sBh = tc::smem_u32(base + LY::O_LBH), sBl = tc::smem_u32(base + LY::O_LBL);
        if (b > 0) {
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = tc::sdesc_sw128(sC + kc * DT_ATOM + 32 * k, 16, 1024);
              const uint64_t bd = tc::sdesc_sw128(sH + kc * DT_ATOM + 32 * k, 16, 1024);
              tc::mma_f16(d0, ad, bd, idesc_f16h(128, 128), (kc | k) != 0);
            }
        }
        if (mode != 3) {
          const int K = (mode == 2) ? du.rd : du.rT;
          const int ks = (K + 7) >> 3;
          for (int kk = 0; kk < ks; ++kk) {
            const uint32_t off = (kk >> 2) * DT_ATOM + 32 * (kk & 3);
            const uint64_t ad = tc::sdesc_sw128(sA + off, 16, 1024);
            const uint64_t bh = tc::sdesc_sw128(sBh + off, 16, 1024);
            tc::mma_tf32(d0 + 128, ad, bh, idesc_tf32(128, 128), kk != 0);
            if (mode == 0) {
              const uint64_t bl = tc::sdesc_sw128(sBl + off, 16, 1024);
              tc::mma_tf32(d0 + 128, ad, bl, idesc_tf32(128, 128), 1);
            }
          }
        }
        tc::mma_commit(tc::smem_u32(&S->tfull[s]));
        tc::mma_commit(tc::smem_u32(&S->empty[s]));
      }
      __syncwarp();
    }
  } else {
    // ---------------- epilogue, thread = row 32 q + lane (TMEM lane quarter
    // q), columns [64 hf, 64 hf + 64)
    const int q = warp & 3, r = 32 * q + lane, hf = (warp - 9) >> 2;
    const bool f32 = (a.out_dtype == JOLT_F32);
    // bf16 tiles go out through shared memory by TMA stores (the 128-byte
    // swizzled layout: conflict-free row writes), fp32 ones directly
    const bool staged = LY::STAGED && !f32;
    const bool lead = (warp == 9 && lane == 0);
    // this row's scale of tile n (raw fp16), read one tile ahead
    auto scale_of = [&](int n) -> unsigned short {
      int u, h, tt;
      tile_at(n, u, h, tt);
      const DecTcUnit du = a.un[u];
      const int row = tt * DT_ROWS + r;
      if (du.b == 0 || row >= T) return 0;
      const char* blob = a.blob + (unsigned long long)(a.u0 + u) * a.stride;
      return reinterpret_cast<const unsigned short*>(blob + du.off_scale)[(size_t)h * T + row];
    };
    unsigned short sc_next = nt > 0 ? scale_of(0) : 0;
    for (int n = 0; n < nt; ++n) {
      int u, h, tt;
      tile_at(n, u, h, tt);
      const DecTcUnit du = a.un[u];
      const int mode = dp_mode(du.rT, du.rd, T), b = du.b;
      const int s = n & 1;
      const float sc = __half2float(__ushort_as_half(sc_next)) * rsD;
      if (n + 1 < nt) sc_next = scale_of(n + 1);
      const bool okw = tc::mbar_wait(tc::smem_u32(&S->tfull[s]), (n >> 1) & 1);
      if (!okw) ok = false;
      tc::tc_fence_after();
      const int row = tt * DT_ROWS + r;
      const bool in = row < T;
      const char* blob = a.blob + (unsigned long long)(a.u0 + u) * a.stride;
      const __half* Grow = reinterpret_cast<const __half*>(blob + du.off_G) +
                           ((size_t)h * T + (in ? row : 0)) * DT_D;
      const uint32_t tl = tmem + 256u * (uint32_t)s + ((uint32_t)(32 * q) << 16);
      const size_t obase = (((size_t)(a.u0 + u) * H + h) * T + (in ? row : 0)) * DT_D;
      unsigned char* stg = base + LY::O_OUT + (n & 1) * 2 * DT_ATOM;
      if (staged) {
        // the TMA store that last read this buffer (tile n - 2) is done
        if (lead && n >= 2) tc::bulk_wait_read1();
        asm volatile("bar.sync 2, 256;" ::: "memory");
      }
      const int cb = 64 * hf;
      // 32 columns of both accumulators per TMEM load (two waits a tile)
#pragma unroll 1
      for (int c0 = cb; c0 < cb + 64; c0 += 32) {
        uint32_t rr[32], rl[32];
        if (b > 0) tmem_ld32_issue(tl + c0, rr);
        if (mode != 3) {
          tmem_ld32_issue(tl + 128 + c0, rl);
        } else {
          // r_T = T, r_d = D: the row of G itself, read while the residual loads
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            const uint4 raw = in ? *reinterpret_cast<const uint4*>(Grow + c0 + i) : make_uint4(0, 0, 0, 0);
            const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(hv[e]);
              rl[i + 2 * e] = __float_as_uint(f.x);
              rl[i + 2 * e + 1] = __float_as_uint(f.y);
            }
          }
        }
        if (b > 0) tmem_ld_wait32(rr);
        if (mode != 3) tmem_ld_wait32(rl);
#pragma unroll
        for (int c = c0; c < c0 + 32; c += 16) {
          const int o16 = c - c0;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float xl = __uint_as_float(rl[o16 + i]);
            x[i] = b > 0 ? fmaf(sc, __uint_as_float(rr[o16 + i]), xl) : xl;
            if (!okw) x[i] = __int_as_float(0x7fc00000);   // a tile whose wait gave up reads NaN
          }
          if (f32) {
            if (in) {
              float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.xhat) + obase + c);
#pragma unroll
              for (int i = 0; i < 16; i += 4) o[i / 4] = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
            }
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const __nv_bfloat162 pv = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
              pk[e] = *reinterpret_cast<const uint32_t*>(&pv);
            }
            if (staged) {
              unsigned char* at = stg + (c >> 6) * DT_ATOM;
              *reinterpret_cast<uint4*>(at + sw128(r, (c & 63) * 2)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              *reinterpret_cast<uint4*>(at + sw128(r, (c & 63) * 2 + 16)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else if (in) {
              uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.xhat) + obase + c);
              o[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              o[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(&S->tempty[s]))
                     : "memory");
      if (staged) {
        // the tile's rows below T go out in two 64-column boxes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync 2, 256;" ::: "memory");
        if (lead) {
          const int rb = (a.u0 + u) * H + h;
          tc::tma_store_3d(&tO, tc::smem_u32(stg), 0, tt * DT_ROWS, rb);
          tc::tma_store_3d(&tO, tc::smem_u32(stg + DT_ATOM), 64, tt * DT_ROWS, rb);
          tc::bulk_commit();
        }
      }
    }
    if (lead) tc::bulk_wait_all();
  }
  if (!ok) atomicOr(&g_decode_status, ST_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 8) tc::tmem_dealloc(tmem, 512);
}

int dp_sm_count() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    n[dev] = v;
  }
  return n[dev];
}

template <int KW>
jolt_status launch_dtc(int ntiles, const DecTcArgs& a, const CUtensorMap& tO, cudaStream_t st) {
  const size_t smem = DpLayout<KW>::BYTES;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(decode_tc_kernel<KW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  const int grid = ntiles < dp_sm_count() ? ntiles : dp_sm_count();
  decode_tc_kernel<KW><<<grid, DP_THREADS, smem, st>>>(a, tO);
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
    a.xhat = xhat; a.nu = nu;
    int kmax = 0;
    for (int i = 0; i < nu; ++i) {
      const jolt_blob_desc& d = desc[u0 + i];
      a.un[i].rT = d.rT; a.un[i].rd = d.rd; a.un[i].b = d.b;
      a.un[i].off_UT = d.off_UT; a.un[i].off_Ud = d.off_Ud; a.un[i].off_G = d.off_G;
      a.un[i].off_scale = d.off_scale; a.un[i].off_codes = d.off_codes;
      if (d.rT < T) kmax = kmax > d.rT ? kmax : d.rT;
      if (d.rd < DT_D) kmax = kmax > d.rd ? kmax : d.rd;
    }
    const int ntiles = nu * H * ((T + DT_ROWS - 1) / DT_ROWS);
    // bf16 output by TMA stores: a map over every unit's rows
    CUtensorMap tO;
    memset(&tO, 0, sizeof(tO));
    if (out_dtype == JOLT_BF16 && kmax <= 32) {
      const cuuint64_t dO[3] = {DT_D, (cuuint64_t)T, (cuuint64_t)U * H};
      const cuuint64_t sO[2] = {DT_D * 2, (cuuint64_t)T * DT_D * 2};
      const cuuint32_t bO[3] = {64, DT_ROWS, 1};
      if (!tc::make_map(&tO, xhat, 3, dO, sO, bO)) return JOLT_ERR_CUDA;
    }
    const jolt_status s =
        kmax <= 32 ? launch_dtc<32>(ntiles, a, tO, st) : launch_dtc<64>(ntiles, a, tO, st);
    if (s != JOLT_OK) return s;
  }
  return JOLT_OK;
}

// The decoder's status word: ST_* bits of bounded waits that gave up since
// the last read (which clears it).
jolt_status decode_tc_status(int* out, cudaStream_t st) {
  JOLT_CUDA_TRY(cudaStreamSynchronize(st));
  int v = 0;
  JOLT_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(int)));
  if (v) {
    const int zero = 0;
    JOLT_CUDA_TRY(cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(int)));
  }
  *out = v;
  return JOLT_OK;
}

}  // namespace jolt
