// The fused candidate sweep on the tensor cores, for bf16 X with D = 128 and
// truncated ranks <= 32.
//
// ["Joint Tucker-rank and residual-bit KV allocator", Formulas: the normalized
//  distortion of every (r_T, r_d, b) candidate; "Rotated Tucker residual for
//  outlier-resistant KV quantization", Key formulas and Implementation notes:
//  the residual rotated by Q = H diag(sigma) / sqrt(D), per-row absmax scale
//  stored in fp16, codes round(y / s).]
//
// The rotated residual of a candidate is formed in the rotated domain,
//   y' = sqrt(D) y = X diag(sigma) H  -  K[:, :r] (sqrt(D) W)[:r, :],
// with K the chain coefficients of the candidate's chain (the fp16 U_T rows
// of one feature rank, or the fp16 rows of Y for the whole token mode) and W
// the rotated factor rows (G (Q U_d)^T, or (Q U_d)^T).  One tensor-core job per
// candidate builds y' directly in a TMEM accumulator: X diag(sigma) H by
// kind::f16 MMAs (bf16 X and the +-1 matrix are exact, fp32 sums), then the
// chain accumulated on top by kind::tf32 MMAs (K is fp16, exact in tf32;
// -sqrt(D) W split into tf32 hi + lo).  Two accumulators alternate, so the
// job of the next candidate runs on the tensor cores while the current one is
// scored.
//
// One persistent CTA of 512 threads per SM walks 128-token tiles of one head.
// Four threads share a token row (32 columns each; warps w, w + 4, w + 8 and
// w + 12 read the same TMEM lane quarter) and meet on the row maximum through
// shared memory and a 128-thread named barrier.  A thread reads its 32 values
// of y' once and keeps them in registers for both passes:
//   pass 1  m = max |y'|, e0 += y'^2;
//   scales  s_b = fp16(m / (sqrt(D) qmax_b)), the stored scale of y, and
//           s'_b = sqrt(D) s_b, its value for y';
//   pass 2  b = 2: the nearest of the levels {-s', 0, s'} lies at distance
//           min(|y'|, ||y'| - s'|) (|y'| / s' <= 1 + 2^-11, the clip never
//           binds); b > 2: q = rint(y' / s') by the 1.5 * 2^23 constant,
//           d = y' - s' q; e_b += d^2.
// A cell gets e / D (the error of y = y' / sqrt(D)), summed per tile in shared
// memory and written to the tile's partials; ||x||^2 of the tile goes to the
// last slot.  Every wait is bounded; a timeout sets the unit's status and
// ends the CTA's work.
#include "jolt_internal.cuh"
#include "tc_common.cuh"

#include <string.h>

namespace jolt {

namespace {

constexpr int STC_ROWS = 128, STC_THREADS = 512, STC_GT = 256;   // two groups of 256
constexpr int STC_XBYTES = STC_ROWS * 256;       // 128 rows x 128 bf16, two 64-column atoms
constexpr int STC_KBYTES = STC_ROWS * 128;       // 128 rows x 32 fp32, one atom
constexpr int STC_KRAW = STC_ROWS * 64;          // 128 rows x 32 fp16: a chain's K as stored
constexpr int STC_GBYTES = STC_XBYTES + 3 * STC_KBYTES + STC_KRAW;   // a group's X, K, W hi / lo, raw K
constexpr int STC_MAX_JOBS = JOLT_MAX_GRID * JOLT_MAX_GRID + JOLT_MAX_GRID + 1;
constexpr int STC_MAX_CELLS = 260;
constexpr float STC_SQRTD = 11.313708498984761f;   // sqrt(128)
constexpr float STC_INVD = 1.f / 128.f;             // exact

struct SweepTcArgs {
  int H, T, nT, nd, nb, nTt, ndt, RT, RD, hasFullT, hasFullD;
  int rT[JOLT_MAX_GRID], rd[JOLT_MAX_GRID], b[4];
  float sq[4];         // 1 / (sqrt(D) qmax_b): max |y'| -> the fp16 scale of y
  int ncand, tiles_t;
  int npu, npairs;     // tile pairs per unit, in all
  char* ws;
  size_t ub, o_UT16, o_W, o_Y16, o_QUd, o_status;
  float* part;
  long long part_us;
};

// One candidate's accumulator.  kind 0: the U_T chain of feature rank `id`;
// 1: the Y chain (whole token mode); 2: the whole-modes residual x - fp16(x).
// r: columns of K used; cell: the candidate's first cell (b index 0).
struct Job {
  int8_t kind, id;
  int16_t r, cell;
};

struct Smem {
  uint64_t hs, tma[2], mma[2][2], ops[2];
  uint32_t tmem;
  int njobs;
  Job job[STC_MAX_JOBS];
};

// Byte offset of (row r, byte b) in a K-major operand with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int r, int byte) {
  return (uint32_t)(r * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15)));
}

// 16 fp32 columns of this thread's TMEM lane into registers, not waited for.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}
// Wait for this thread's TMEM loads, tied to the registers they fill (so that
// no use of them is scheduled before it).
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// One pass over this thread's 64 columns of an accumulator, 16 at a time with
// the next 16 in flight: f(y0, y1) on consecutive pairs.
template <typename F>
__device__ __forceinline__ void stc_pass(uint32_t taddr, F&& f) {
  uint32_t ra[16], rb[16];
  tmem_ld16_issue(taddr, ra);
  tmem_ld_wait(ra);
#pragma unroll
  for (int c = 0; c < 64; c += 32) {
    tmem_ld16_issue(taddr + c + 16, rb);
#pragma unroll
    for (int i = 0; i < 16; i += 2) f(__uint_as_float(ra[i]), __uint_as_float(ra[i + 1]));
    tmem_ld_wait(rb);
    if (c + 32 < 64) tmem_ld16_issue(taddr + c + 32, ra);
#pragma unroll
    for (int i = 0; i < 16; i += 2) f(__uint_as_float(rb[i]), __uint_as_float(rb[i + 1]));
    if (c + 32 < 64) tmem_ld_wait(ra);
  }
}

// Scores one candidate from its accumulator (this thread's 64 columns at
// taddr): the row maximum with the partner thread (rm: the two halves' slots,
// pbar: the pair's 64-thread barrier), the fp16 scales, and the squared
// errors of b = 0 (v0), of b = 2 when present (v2) and of the NQ widths above
// 2 (vq, scale factors sqq).  The widths are template parameters so that the
// per-element loops carry no branch.
template <bool HAS2, int NQ>
__device__ __forceinline__ void score_t(uint32_t taddr, float* rm, int hf, int lr, int pbar,
                                        float sq2, const float (&sqq)[2], float& v0, float& v2,
                                        float (&vq)[2]) {
  float m0 = 0.f, m1 = 0.f;
  float2 e0 = make_float2(0.f, 0.f);
  stc_pass(taddr, [&](float y0, float y1) {
    m0 = fmaxf(m0, fabsf(y0));
    m1 = fmaxf(m1, fabsf(y1));
    const float2 yy = make_float2(y0, y1);
    e0 = __ffma2_rn(yy, yy, e0);
  });
  rm[hf * STC_ROWS + lr] = fmaxf(m0, m1);
  asm volatile("bar.sync %0, 64;" ::"r"(pbar) : "memory");
  const float m = fmaxf(rm[lr], rm[STC_ROWS + lr]);
  v0 = e0.x + e0.y;
  const float s2 = HAS2 ? round_f16(m * sq2) * STC_SQRTD : 0.f;
  float sq[2], inv[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    sq[k] = 0.f;
    inv[k] = 0.f;
    if (k < NQ) {
      sq[k] = round_f16(m * sqq[k]) * STC_SQRTD;
      float r;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(sq[k]));
      inv[k] = sq[k] > 0.f ? r : 0.f;
    }
  }
  const float2 M2 = make_float2(12582912.0f, 12582912.0f);
  const float2 nM2 = make_float2(-12582912.0f, -12582912.0f);
  float2 e2 = make_float2(0.f, 0.f);
  float2 eq[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if (HAS2 || NQ > 0) {
    stc_pass(taddr, [&](float y0, float y1) {
      if (HAS2) {
        // distance to the nearest of {-s, 0, s}
        const float a0 = fabsf(y0), a1 = fabsf(y1);
        const float d0 = fminf(a0, fabsf(a0 - s2)), d1 = fminf(a1, fabsf(a1 - s2));
        e2.x = fmaf(d0, d0, e2.x);
        e2.y = fmaf(d1, d1, e2.y);
      }
#pragma unroll
      for (int k = 0; k < NQ; ++k) {
        const float2 yy = make_float2(y0, y1);
        const float2 qq = __fadd2_rn(__ffma2_rn(yy, make_float2(inv[k], inv[k]), M2), nM2);
        const float2 dd = __ffma2_rn(make_float2(-sq[k], -sq[k]), qq, yy);
        eq[k] = __ffma2_rn(dd, dd, eq[k]);
      }
    });
  }
  v2 = e2.x + e2.y;
#pragma unroll
  for (int k = 0; k < 2; ++k) vq[k] = eq[k].x + eq[k].y;
}

// The global reads of a chain's operands for this thread: K row lr, columns
// [16 hf, 16 hf + 16) as raw fp16, and W[k][lr] for the same k.
struct Pre {
  uint4 k[2];
  float w[16];
};

template <bool HAS2, int NQ>
__global__ void __launch_bounds__(STC_THREADS, 1)
sweep_tc_kernel(const __grid_constant__ CUtensorMap tX, const __grid_constant__ CUtensorMap tHs,
                SweepTcArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  // 1024-byte aligned, derived from the shared array itself (so that every
  // pointer below stays a shared-window address)
  unsigned char* base = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int g = t >> 8, gt = t & (STC_GT - 1);                // group, thread in group
  const int q = warp & 3, hf = (gt >> 5) >> 2;                // lane quarter, column half
  const int lr = 32 * q + lane;                               // token row within the tile
  const int k0 = 16 * hf;                                     // this thread's K columns
  unsigned char* sH = base;                                   // diag(sigma) H (B^T, bf16), shared
  unsigned char* sX = base + STC_XBYTES + g * STC_GBYTES;     // this group's X tile
  unsigned char* sK = sX + STC_XBYTES;                        // chain coefficients (tf32)
  unsigned char* sBh = sK + STC_KBYTES;                       // -sqrt(D) W^T, tf32 hi
  unsigned char* sBl = sBh + STC_KBYTES;                      // and lo
  uint4* sKraw = reinterpret_cast<uint4*>(sBl + STC_KBYTES);  // the chain's K, fp16 [128][32]
  float* cells_all = reinterpret_cast<float*>(base + STC_XBYTES + 2 * STC_GBYTES);
  float* cells = cells_all + g * STC_MAX_CELLS;               // [ncand + 1]
  float* rmax_all = cells_all + 2 * STC_MAX_CELLS;            // [group][2 jobs][2 halves][128]
  float* rmax = rmax_all + g * 2 * 2 * STC_ROWS;
  Smem* S = reinterpret_cast<Smem*>(rmax_all + 2 * 2 * 2 * STC_ROWS);
  const int gbar = 1 + g;                                     // the group's named barrier
  const int pbar = 3 + 4 * g + q;                             // the row pair's (64 threads)

  if (t == 0) {
    int n = 0;
    if (a.nTt > 0)
      for (int id = 0; id < a.nd; ++id)
        for (int i = 0; i < a.nTt; ++i) {
          Job j; j.kind = 0; j.id = (int8_t)id; j.r = (int16_t)a.rT[i];
          j.cell = (int16_t)((i * a.nd + id) * a.nb);
          S->job[n++] = j;
        }
    if (a.hasFullT && a.ndt > 0)
      for (int i = 0; i < a.ndt; ++i) {
        Job j; j.kind = 1; j.id = 0; j.r = (int16_t)a.rd[i];
        j.cell = (int16_t)(((a.nT - 1) * a.nd + i) * a.nb);
        S->job[n++] = j;
      }
    if (a.hasFullT && a.hasFullD) {
      Job j; j.kind = 2; j.id = 0; j.r = 0;
      j.cell = (int16_t)(((a.nT - 1) * a.nd + a.nd - 1) * a.nb);
      S->job[n++] = j;
    }
    S->njobs = n;
    tc::mbar_init(tc::smem_u32(&S->hs), 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(tc::smem_u32(&S->tma[i]), 1);
      tc::mbar_init(tc::smem_u32(&S->mma[i][0]), 1);
      tc::mbar_init(tc::smem_u32(&S->mma[i][1]), 1);
      tc::mbar_init(tc::smem_u32(&S->ops[i]), 8);
    }
    tc::fence_barrier_init();
  }
  for (int i = t; i < 2 * STC_MAX_CELLS; i += STC_THREADS) cells_all[i] = 0.f;
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&S->tmem), 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S->tmem + 256u * (uint32_t)g;         // this group's two accumulators
  const int J = S->njobs;
  // the bit widths' slots: b = 0, b = 2 and the (NQ) widths above 2
  int i0 = -1, i2 = -1, iq0 = -1, iq1 = -1;
  float sq2 = 0.f, sqq[2] = {0.f, 0.f};
  for (int ib = 0; ib < a.nb; ++ib) {
    if (a.b[ib] == 0) {
      i0 = ib;
    } else if (a.b[ib] == 2) {
      i2 = ib;
      sq2 = a.sq[ib];
    } else if (iq0 < 0) {
      iq0 = ib;
      sqq[0] = a.sq[ib];
    } else {
      iq1 = ib;
      sqq[1] = a.sq[ib];
    }
  }

  constexpr uint32_t idesc16 = tc::idesc_bf16(128, 128, 0, 0);
  constexpr uint32_t idesc32 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(128 >> 3) << 17) |
                               ((uint32_t)(128 >> 4) << 24);
  const bool leader = (gt == 0);
  const int tiles_u = a.tiles_t * a.H;                        // tiles per unit
  bool ok = true;
  // commits issued and waited for, per barrier (the same counts across a group)
  uint32_t hs_issued = 0, hs_waited = 0;
  uint32_t tma_issued = 0, tma_waited = 0;
  // jobs of this group issued / waited for, counted over the whole kernel:
  // job n uses accumulator n & 1, and is phase n >> 1 of that buffer's barrier
  uint32_t jobs_issued = 0, jobs_waited = 0;
  uint32_t ops_phase = 0;
  int loaded_unit = -1, fail_unit = 0;
  // this group's tile of pair p (unit, head, token tile), or false
  auto tile_of = [&](int p, int& u, int& h, int& tt) {
    u = p / a.npu;
    const int i = 2 * (p % a.npu) + g;
    h = i / a.tiles_t;
    tt = i % a.tiles_t;
    return i < tiles_u;
  };
  auto issue_x = [&](int u, int h, int tt) {
    if (leader) {
      const uint32_t fb = tc::smem_u32(&S->tma[g]);
      tc::mbar_expect_tx(fb, STC_XBYTES);
      tc::tma_load_3d(tc::smem_u32(sX), &tX, 0, tt * STC_ROWS, u * a.H + h, fb);
      tc::tma_load_3d(tc::smem_u32(sX + STC_XBYTES / 2), &tX, 64, tt * STC_ROWS, u * a.H + h, fb);
    }
    ++tma_issued;
  };
  bool x_ready = false;   // this group's X of the next pair is already on its way
  bool stop = false;
#pragma unroll 1
  for (int p = blockIdx.x; p < a.npairs; p += gridDim.x) {
    int u, h, tt;
    const bool valid = tile_of(p, u, h, tt);
    // every product of the previous pair is done (each group waited for its
    // last one): the sign matrix may change
    if (__syncthreads_or(!ok)) { stop = true; break; }
    if (u != loaded_unit) {
      if (t == 0) {
        const uint32_t fb = tc::smem_u32(&S->hs);
        tc::mbar_expect_tx(fb, STC_XBYTES);
        tc::tma_load_3d(tc::smem_u32(sH), &tHs, 0, 0, u, fb);
        tc::tma_load_3d(tc::smem_u32(sH + STC_XBYTES / 2), &tHs, 64, 0, u, fb);
      }
      ++hs_issued;
      loaded_unit = u;
    }
    if (valid && !x_ready) issue_x(u, h, tt);
    x_ready = false;
    if (hs_waited < hs_issued) {
      if (!tc::mbar_wait(tc::smem_u32(&S->hs), hs_waited & 1)) ok = false;
      ++hs_waited;
    }
    if (!valid) continue;
    fail_unit = u;
    const int row = tt * STC_ROWS + lr;
    const bool in = row < a.T;
    char* wu = a.ws + (size_t)u * a.ub;
    if (!tc::mbar_wait(tc::smem_u32(&S->tma[g]), tma_waited & 1)) ok = false;
    ++tma_waited;
    // ---- ||x||^2 of the tile, this thread's 64 columns
    {
      float xn = 0.f;
      const unsigned char* px = sX + hf * (STC_XBYTES / 2);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(px + sw128(lr, 16 * i));
        const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(e[k]);
          xn = fmaf(f.x, f.x, fmaf(f.y, f.y, xn));
        }
      }
      xn = warp_sum(xn);
      if (lane == 0) atomicAdd(&cells[a.ncand], xn);
    }
    // operand reads of job jb's chain (kinds 0 and 1)
    auto fetch = [&](const Job& jb, Pre& pr) {
      const __half* Kg;
      int kn;
      const float* Bg;
      if (jb.kind == 0) {
        Kg = (const __half*)(wu + a.o_UT16) + (long long)jb.id * a.T * a.RT;
        kn = a.RT;
        Bg = (const float*)(wu + a.o_W) + ((long long)jb.id * a.H + h) * a.RT * 128;
      } else {
        Kg = (const __half*)(wu + a.o_Y16) + (long long)h * a.T * a.RD;
        kn = a.RD;
        Bg = (const float*)(wu + a.o_QUd);
      }
      if (kn == 32) {
        const uint4* src = reinterpret_cast<const uint4*>(Kg + (long long)row * 32 + k0);
        pr.k[0] = in ? src[0] : make_uint4(0, 0, 0, 0);
        pr.k[1] = in ? src[1] : make_uint4(0, 0, 0, 0);
      } else {
        uint32_t hw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ka = k0 + 2 * i, kb = ka + 1;
          const unsigned short lo =
              (in && ka < kn) ? __half_as_ushort(Kg[(long long)row * kn + ka]) : (unsigned short)0;
          const unsigned short hi =
              (in && kb < kn) ? __half_as_ushort(Kg[(long long)row * kn + kb]) : (unsigned short)0;
          hw[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        pr.k[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        pr.k[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) pr.w[i] = (k0 + i < kn) ? Bg[(long long)(k0 + i) * 128 + lr] : 0.f;
    };
    // the chain's K (raw fp16, kept for the masks) and -sqrt(D) W^T hi / lo
    auto store = [&](const Pre& pr) {
      sKraw[lr * 4 + 2 * hf] = pr.k[0];
      sKraw[lr * 4 + 2 * hf + 1] = pr.k[1];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        float bh[4], bl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float b = -STC_SQRTD * pr.w[i + e];
          bh[e] = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
          bl[e] = b - bh[e];
        }
        *reinterpret_cast<float4*>(sBh + sw128(lr, (k0 + i) * 4)) = make_float4(bh[0], bh[1], bh[2], bh[3]);
        *reinterpret_cast<float4*>(sBl + sw128(lr, (k0 + i) * 4)) = make_float4(bl[0], bl[1], bl[2], bl[3]);
      }
    };
    // this thread's K columns for a job of chain length r, with columns
    // [r, 8 ceil(r / 8)) zero (the MMA runs whole k-steps of 8)
    auto set_mask = [&](int r) {
      const int hi = (r + 7) & ~7;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 raw = sKraw[lr * 4 + 2 * hf + c];
        const __half2* hv = reinterpret_cast<const __half2*>(&raw);
        float kv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(hv[i]);
          kv[2 * i] = f.x;
          kv[2 * i + 1] = f.y;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int k = k0 + 8 * c + i;
          if (k >= r && k < hi) kv[i] = 0.f;
        }
        *reinterpret_cast<float4*>(sK + sw128(lr, (k0 + 8 * c) * 4)) = make_float4(kv[0], kv[1], kv[2], kv[3]);
        *reinterpret_cast<float4*>(sK + sw128(lr, (k0 + 8 * c + 4) * 4)) = make_float4(kv[4], kv[5], kv[6], kv[7]);
      }
    };
    // x - fp16(x) over this thread's half of the X tile, in place (bf16-exact)
    auto residual_x = [&]() {
      unsigned char* px = sX + hf * (STC_XBYTES / 2);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint4* pv = reinterpret_cast<uint4*>(px + sw128(lr, 16 * i));
        uint4 v = *pv;
        __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&v);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float x = __bfloat162float(e[k]);
          e[k] = __float2bfloat16_rn(x - round_f16(x));
        }
        *pv = v;
      }
    };
    auto same_chain = [](const Job& x, const Job& y) { return x.kind == y.kind && x.id == y.id; };
    // job jb into the next accumulator (the group's leader issues)
    auto issue_mma = [&](const Job& jb) {
      const int buf = (int)(jobs_issued & 1);
      ++jobs_issued;
      if (!leader) return;
      tc::tc_fence_after();
      const uint32_t d = tmem + 128u * (uint32_t)buf;
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sX + kc * (STC_XBYTES / 2)) + 32 * k, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sH + kc * (STC_XBYTES / 2)) + 32 * k, 16, 1024);
          tc::mma_f16(d, ad, bd, idesc16, (kc | k) != 0);
        }
      if (jb.kind != 2) {
        const int ks = (jb.r + 7) >> 3;
        for (int k = 0; k < ks; ++k) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sK) + 32 * k, 16, 1024);
          const uint64_t bh = tc::sdesc_sw128(tc::smem_u32(sBh) + 32 * k, 16, 1024);
          const uint64_t bl = tc::sdesc_sw128(tc::smem_u32(sBl) + 32 * k, 16, 1024);
          tc::mma_tf32(d, ad, bh, idesc32, 1);
          tc::mma_tf32(d, ad, bl, idesc32, 1);
        }
      }
      tc::mma_commit(tc::smem_u32(&S->mma[g][buf]));
    };
    auto wait_mma = [&]() {
      const int buf = (int)(jobs_waited & 1);
      if (!tc::mbar_wait(tc::smem_u32(&S->mma[g][buf]), (jobs_waited >> 1) & 1,
                         ok ? tc::WAIT_LIMIT : 1024))
        ok = false;
      ++jobs_waited;
      tc::tc_fence_after();
    };

    // every warp of the group has written its share of the next job's
    // operands (and is done with the accumulator that job overwrites): one
    // arrival per warp; the leader, which issues the job, waits for all eight
    auto ops_ready = [&]() {
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(&S->ops[g]))
                     : "memory");
      if (leader && !tc::mbar_wait(tc::smem_u32(&S->ops[g]), ops_phase & 1, ok ? tc::WAIT_LIMIT : 1024))
        ok = false;
      ++ops_phase;
    };
    // ---- job 0
    Pre pre;
    {
      const Job j0 = S->job[0];
      if (j0.kind == 2) {
        residual_x();
      } else {
        fetch(j0, pre);
        store(pre);
        set_mask(j0.r);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc::tc_fence_before();
      ops_ready();
      issue_mma(j0);
    }
    for (int j = 0; j < J; ++j) {
      const Job jb = S->job[j];
      const int buf = (int)(jobs_waited & 1);   // job j's accumulator
      wait_mma();
      // the next job's operands (the chain's, or K's mask) and its product
      // into the other accumulator, which job j - 1 no longer reads
      if (j + 1 < J) {
        const Job jn = S->job[j + 1];
        if (jn.kind == 2) {
          residual_x();
        } else {
          if (!same_chain(jn, jb)) {
            fetch(jn, pre);
            store(pre);
          }
          set_mask(jn.r);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::tc_fence_before();
        ops_ready();
        issue_mma(jn);
      } else if (p + (int)gridDim.x < a.npairs) {
        // every product of this tile is done: the next X may land
        int u2, h2, tt2;
        if (tile_of(p + (int)gridDim.x, u2, h2, tt2)) {
          issue_x(u2, h2, tt2);
          x_ready = true;
        }
      }
      // ---- score job j from accumulator buf
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + 128u * (uint32_t)buf + 64u * (uint32_t)hf;
      float* rm = rmax + (size_t)buf * 2 * STC_ROWS;
      float v0, v2, vq[2];
      score_t<HAS2, NQ>(taddr, rm, hf, lr, pbar, sq2, sqq, v0, v2, vq);
      v0 = warp_sum(v0) * STC_INVD;
      v2 = warp_sum(v2) * STC_INVD;
#pragma unroll
      for (int k = 0; k < 2; ++k) vq[k] = warp_sum(vq[k]) * STC_INVD;
      if (lane == 0) {
        if (i0 >= 0) atomicAdd(&cells[jb.cell + i0], v0);
        if (i2 >= 0) atomicAdd(&cells[jb.cell + i2], v2);
        if (iq0 >= 0) atomicAdd(&cells[jb.cell + iq0], vq[0]);
        if (iq1 >= 0) atomicAdd(&cells[jb.cell + iq1], vq[1]);
      }
    }
    // ---- the tile's partials
    asm volatile("bar.sync %0, 256;" ::"r"(gbar) : "memory");
    float* part = a.part + u * a.part_us + ((long long)h * a.tiles_t + tt) * (a.ncand + 1);
    for (int i = gt; i <= a.ncand; i += STC_GT) {
      part[i] = cells[i];
      cells[i] = 0.f;
    }
  }
  if (!ok || stop) {
    atomicOr((int*)(a.ws + (size_t)fail_unit * a.ub + a.o_status), ST_TIMEOUT);
    // let the copies and products still in flight finish (bounded) before
    // the accumulators are freed
    if (leader) {
      while (tma_waited < tma_issued) {
        tc::mbar_wait(tc::smem_u32(&S->tma[g]), tma_waited & 1);
        ++tma_waited;
      }
      while (jobs_waited < jobs_issued) {
        tc::mbar_wait(tc::smem_u32(&S->mma[g][jobs_waited & 1]), (jobs_waited >> 1) & 1);
        ++jobs_waited;
      }
    }
    if (t == 0)
      while (hs_waited < hs_issued) {
        tc::mbar_wait(tc::smem_u32(&S->hs), hs_waited & 1);
        ++hs_waited;
      }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(S->tmem, 512);
}

size_t sweep_smem() {
  return 1024 + (size_t)STC_XBYTES + 2 * (size_t)STC_GBYTES + 2 * STC_MAX_CELLS * 4 +
         2 * 2 * 2 * STC_ROWS * 4 + sizeof(Smem) + 64;
}

template <bool HAS2, int NQ>
jolt_status launch_sweep(int grid, const CUtensorMap& tX, const CUtensorMap& tH,
                         const SweepTcArgs& a, cudaStream_t st) {
  const size_t smem = sweep_smem();
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(sweep_tc_kernel<HAS2, NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  sweep_tc_kernel<HAS2, NQ><<<grid, STC_THREADS, smem, st>>>(tX, tH, a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

int sm_count() {
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

}  // namespace

bool sweep_tc_supported(const Layout& L) {
  return L.dtype == JOLT_BF16 && L.D == 128 && L.RT <= 32 && L.RD <= 32 && L.o_Hs != 0 &&
         tc::encode_fn() != nullptr && L.ncand + 1 <= STC_MAX_CELLS && L.nb <= 4;
}

// Tiles per head: 128 tokens each.
int sweep_tc_tiles(const Layout& L) { return (L.T + STC_ROWS - 1) / STC_ROWS; }

jolt_status sweep_tc_run(const Layout& L, int U, const void* X, char* ws, float* part,
                         long long part_us, int* tiles_t_out, cudaStream_t st) {
  CUtensorMap tX;
  const cuuint64_t dX[3] = {128, (cuuint64_t)L.T, (cuuint64_t)U * L.H};
  const cuuint64_t sX[2] = {256, (cuuint64_t)L.T * 256};
  const cuuint32_t bX[3] = {64, 128, 1};
  if (!tc::make_map(&tX, X, 3, dX, sX, bX)) return JOLT_ERR_CUDA;
  // the sign matrices sit one per unit region: a 3-D map (128 cols, 128 rows, unit)
  CUtensorMap tH3;
  const cuuint64_t dH3[3] = {128, 128, (cuuint64_t)U};
  const cuuint64_t sH3[2] = {256, (cuuint64_t)L.unit_bytes};
  const cuuint32_t bH3[3] = {64, 128, 1};
  if (!tc::make_map(&tH3, ws + L.o_Hs, 3, dH3, sH3, bH3)) return JOLT_ERR_CUDA;
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
    a.sq[i] = L.b[i] > 0 ? (float)(1.0 / (11.313708498984761 * ((1 << (L.b[i] - 1)) - 1))) : 0.f;
  }
  a.ncand = L.ncand;
  a.tiles_t = sweep_tc_tiles(L);
  a.npu = (a.tiles_t * L.H + 1) / 2;
  a.npairs = a.npu * U;
  a.ws = ws; a.ub = L.unit_bytes;
  a.o_UT16 = L.o_UT16; a.o_W = L.o_W; a.o_Y16 = L.o_Y16; a.o_QUd = L.o_QUd; a.o_status = L.o_status;
  a.part = part; a.part_us = part_us;
  bool has2 = false;
  int nq = 0;
  for (int i = 0; i < L.nb; ++i) {
    if (L.b[i] == 2) has2 = true;
    if (L.b[i] > 2) ++nq;
  }
  const int grid = a.npairs < sm_count() ? a.npairs : sm_count();
  jolt_status s;
  if (has2) {
    s = nq == 0 ? launch_sweep<true, 0>(grid, tX, tH3, a, st)
                : (nq == 1 ? launch_sweep<true, 1>(grid, tX, tH3, a, st)
                           : launch_sweep<true, 2>(grid, tX, tH3, a, st));
  } else {
    s = nq == 0 ? launch_sweep<false, 0>(grid, tX, tH3, a, st)
                : (nq == 1 ? launch_sweep<false, 1>(grid, tX, tH3, a, st)
                           : launch_sweep<false, 2>(grid, tX, tH3, a, st));
  }
  if (s != JOLT_OK) return s;
  *tiles_t_out = a.tiles_t;
  return JOLT_OK;
}

}  // namespace jolt
