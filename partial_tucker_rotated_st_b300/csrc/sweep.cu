// Distortion of every (r_T, r_d, b) candidate of every unit, in one pass over X.
//
// ["Joint Tucker-rank and residual-bit KV allocator", Formulas: R = X - X~,
//  X^ = X~ + Q^T Q_b(Q R), D = ||X - X^||^2 / ||X||^2; "Rotated Tucker
//  residual for outlier-resistant KV quantization", Key formulas and
//  Implementation notes: Q_b(Y) = s clip(round(Y/s), -2^(b-1), 2^(b-1)-1),
//  s = max|Y_i| / (2^(b-1) - 1) per block, Q a normalized Hadamard transform.]
//
// The kernel evaluates the same quantities through identities that are exact
// in real arithmetic:
//   * Q is orthogonal, so ||X - X^|| = ||Q R - Q_b(Q R)||: no inverse
//     transform is needed to score a candidate.
//   * Q R = Q X - X~ Q^T, and X~ Q^T = U_T (G (Q U_d)^T): X is rotated once
//     per tile (a warp-level fast Walsh-Hadamard transform) and the small
//     factor matrices are rotated instead of every residual row.
//   * Truncated ranks are nested: the reconstruction for r_T = 4, 8, 16, 32
//     is a running prefix sum over the rank index, so every token rank of
//     one r_d costs one chain of RT multiply-adds per element, and likewise
//     for the feature ranks of the r_T = T column.
//   * One quantization block is one (h, t) row of D values; the clip of the
//     quantizer never binds (|y/s| <= qmax (1 + 2^-11) < qmax + 1/2), and
//     y - s round(y/s) is scored for every b of the grid from one residual.
// X is read from HBM once per tile; each tile keeps its rotated rows in
// registers across all candidates.
#include "jolt_internal.cuh"

namespace jolt {

void* g_sweep_ev[2] = {nullptr, nullptr};

namespace {

constexpr int SW_WARPS = 8;
constexpr int SW_THREADS = SW_WARPS * 32;
constexpr int SW_EPT = 16;   // features per lane
constexpr int SW_RPT = 2;    // rows per thread

struct SweepArgs {
  const void* X;
  const int8_t* signs;
  char* ws;
  size_t ub;
  int H, T, D, dtype;
  int nT, nd, nb, nTt, ndt, RT, RD, hasFullT, hasFullD;
  int rT[JOLT_MAX_GRID], rd[JOLT_MAX_GRID], b[4];
  float rq[4];         // 1 / (2^(b-1) - 1) for b > 0
  int ncand, tiles_t;
  size_t o_UT16, o_W, o_Y16, o_QUd;
  float* part;          // per-tile partial sums, unit u at part + u * part_us
  long long part_us;
};

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

// Fast Walsh-Hadamard transform (Sylvester order) of a row held by LPR lanes,
// 16 consecutive features each: element index = (lane % LPR) * 16 + i.
template <int LPR>
__device__ __forceinline__ void fwht16(float (&v)[SW_EPT], int lane) {
#pragma unroll
  for (int h = 1; h < SW_EPT; h <<= 1)
#pragma unroll
    for (int e = 0; e < SW_EPT; ++e)
      if (!(e & h)) {
        const float a = v[e], b = v[e + h];
        v[e] = a + b;
        v[e + h] = a - b;
      }
#pragma unroll
  for (int m = 1; m < LPR; m <<= 1)
#pragma unroll
    for (int e = 0; e < SW_EPT; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = (lane & m) ? (o - v[e]) : (v[e] + o);
    }
}

// Sum v[0..3] over the 32 lanes of the warp (reduce-scatter butterfly);
// lane 8*i (i < 4) ends with the total of v[i].
__device__ __forceinline__ float reduce4(const float (&v)[4], int lane) {
  const bool h16 = lane & 16;
  float a0 = h16 ? v[2] : v[0], a1 = h16 ? v[3] : v[1];
  const float s0 = h16 ? v[0] : v[2], s1 = h16 ? v[1] : v[3];
  a0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  a1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  const bool h8 = lane & 8;
  float c = h8 ? a1 : a0;
  const float d = h8 ? a0 : a1;
  c += __shfl_xor_sync(0xffffffffu, d, 8);
  c += __shfl_xor_sync(0xffffffffu, c, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// Score one candidate.  acc holds the rotated residual Q R of this thread's
// two rows, 16 features each, as packed pairs.  Per row: m = max|y| over the
// row's LPR lanes; per b > 0: s = fp16(m / qmax), z = y / s (a reciprocal
// multiply), q = round-half-even(z), error y - s q; b = 0 scores y itself.
template <int LPR>
__device__ __forceinline__ void score(const float2 (&acc)[SW_RPT][SW_EPT / 2],
                                      const SweepArgs& a, float* cells, int cell0, int lane) {
  // independent accumulators per row and per half of the row keep the
  // dependency chains short
  float m[SW_RPT];
  float2 e0[SW_RPT];
#pragma unroll
  for (int r = 0; r < SW_RPT; ++r) {
    float ma = 0.f, mb = 0.f;
    float2 ea = make_float2(0.f, 0.f), eb = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < SW_EPT / 2; i += 2) {
      ma = fmaxf(ma, fmaxf(fabsf(acc[r][i].x), fabsf(acc[r][i].y)));
      mb = fmaxf(mb, fmaxf(fabsf(acc[r][i + 1].x), fabsf(acc[r][i + 1].y)));
      ea = __ffma2_rn(acc[r][i], acc[r][i], ea);
      eb = __ffma2_rn(acc[r][i + 1], acc[r][i + 1], eb);
    }
    float mm = fmaxf(ma, mb);
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    m[r] = mm;
    e0[r] = __fadd2_rn(ea, eb);
  }
  // round-half-even to an integer by adding and removing 1.5 * 2^23; the
  // product y / s and the addition are fused, so q is the integer nearest
  // to the exact y * (1/s)
  const float2 M2 = f2(12582912.0f), nM2 = f2(-12582912.0f);
  float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ib = 0; ib < 4; ++ib) {
    if (ib >= a.nb) break;
    if (a.b[ib] == 0) {
      const float2 e = __fadd2_rn(e0[0], e0[1]);
      v[ib] = e.x + e.y;
      continue;
    }
    float2 ebr[SW_RPT];
#pragma unroll
    for (int r = 0; r < SW_RPT; ++r) {
      const float s = round_f16(m[r] * a.rq[ib]);
      float inv;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(s));
      if (!(s > 0.f)) inv = 0.f;
      const float2 inv2 = f2(inv), ns2 = f2(-s);
      float2 ea = make_float2(0.f, 0.f), eb = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < SW_EPT / 2; i += 2) {
        const float2 qa = __fadd2_rn(__ffma2_rn(acc[r][i], inv2, M2), nM2);
        const float2 qb = __fadd2_rn(__ffma2_rn(acc[r][i + 1], inv2, M2), nM2);
        const float2 da = __ffma2_rn(ns2, qa, acc[r][i]);
        const float2 db = __ffma2_rn(ns2, qb, acc[r][i + 1]);
        ea = __ffma2_rn(da, da, ea);
        eb = __ffma2_rn(db, db, eb);
      }
      ebr[r] = __fadd2_rn(ea, eb);
    }
    const float2 e = __fadd2_rn(ebr[0], ebr[1]);
    v[ib] = e.x + e.y;
  }
  const float t = reduce4(v, lane);
  if ((lane & 7) == 0) {
    const int ib = lane >> 3;
    if (ib < a.nb) atomicAdd(&cells[cell0 + ib], t);
  }
}

// acc -= K[k][rows] * B[k][:] for k in [k0, k1), then score at each nested rank.
template <int LPR>
__device__ __forceinline__ void chain_step(float2 (&acc)[SW_RPT][SW_EPT / 2], const float* Ks,
                                           const float* Bs, int tile, int bld, int k, int row0,
                                           int l) {
  const float2 kr = *reinterpret_cast<const float2*>(Ks + k * tile + row0);
  const float4* bp = reinterpret_cast<const float4*>(Bs + k * bld + l * 20);
  float2 bv[SW_EPT / 2];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 t4 = bp[q];
    bv[2 * q] = make_float2(t4.x, t4.y);
    bv[2 * q + 1] = make_float2(t4.z, t4.w);
  }
  const float2 n0 = f2(-kr.x), n1 = f2(-kr.y);
#pragma unroll
  for (int i = 0; i < SW_EPT / 2; ++i) {
    acc[0][i] = __ffma2_rn(n0, bv[i], acc[0][i]);
    acc[1][i] = __ffma2_rn(n1, bv[i], acc[1][i]);
  }
}

template <typename TX, int LPR>
__global__ void __launch_bounds__(SW_THREADS, 2) sweep_kernel(SweepArgs a) {
  constexpr int D = SW_EPT * LPR;
  constexpr int GPW = 32 / LPR;              // row groups per warp
  constexpr int TILE = SW_WARPS * GPW * SW_RPT;
  constexpr int BLD = LPR * 20;              // factor row, 16 floats + 4 pad per lane block
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;                          // [64][TILE] chain coefficients
  float* Bs = Ks + 64 * TILE;                // [64][BLD]  rotated factor rows
  float* cells = Bs + 64 * BLD;              // [ncand + 1]

  const int u = blockIdx.z, h = blockIdx.y, tt = blockIdx.x;
  const int t0 = tt * TILE;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int l = lane % LPR, g = lane / LPR;
  const int row0 = w * GPW * SW_RPT + g * SW_RPT;   // this thread's first tile row
  char* base = a.ws + u * a.ub;
  for (int i = threadIdx.x; i <= a.ncand; i += SW_THREADS) cells[i] = 0.f;

  // ---- X rows, rotated once: qx = H (sigma .* x) / sqrt(D)
  const TX* Xu = (const TX*)a.X + ((long long)u * a.H + h) * a.T * D;
  float sg[SW_EPT];
#pragma unroll
  for (int i = 0; i < SW_EPT; ++i) sg[i] = (float)a.signs[(long long)u * D + l * SW_EPT + i];
  const float rs = rsqrtf((float)D);
  float2 qx[SW_RPT][SW_EPT / 2], acc[SW_RPT][SW_EPT / 2];
  float xn = 0.f;
  const bool fullTD = a.hasFullT && a.hasFullD;
#pragma unroll
  for (int r = 0; r < SW_RPT; ++r) {
    const int t = t0 + row0 + r;
    float x[SW_EPT], v[SW_EPT];
#pragma unroll
    for (int i = 0; i < SW_EPT; ++i)
      x[i] = (t < a.T) ? to_f32(Xu[(long long)t * D + l * SW_EPT + i]) : 0.f;
#pragma unroll
    for (int i = 0; i < SW_EPT; ++i) {
      xn = fmaf(x[i], x[i], xn);
      v[i] = x[i] * sg[i];
    }
    fwht16<LPR>(v, lane);
#pragma unroll
    for (int i = 0; i < SW_EPT / 2; ++i) qx[r][i] = make_float2(v[2 * i] * rs, v[2 * i + 1] * rs);
    if (fullTD) {
      // (r_T, r_d) = (T, D): the stored core is fp16(X) itself
#pragma unroll
      for (int i = 0; i < SW_EPT; ++i) v[i] = (x[i] - round_f16(x[i])) * sg[i];
      fwht16<LPR>(v, lane);
#pragma unroll
      for (int i = 0; i < SW_EPT / 2; ++i) acc[r][i] = make_float2(v[2 * i] * rs, v[2 * i + 1] * rs);
    }
  }
  __syncthreads();  // cells cleared
  xn = warp_sum(xn);
  if (lane == 0) atomicAdd(&cells[a.ncand], xn);
  const int iTfull = a.nT - 1, idfull = a.nd - 1;
  if (fullTD) score<LPR>(acc, a, cells, (iTfull * a.nd + idfull) * a.nb, lane);

  // ---- r_T = T, truncated r_d: X~ Q^T = Y16 (Q U_d)^T, prefix over r_d
  if (a.hasFullT && a.ndt > 0) {
    const __half* Yh = (const __half*)(base + a.o_Y16) + (long long)h * a.T * a.RD;
    // consecutive threads take consecutive rows: conflict-free stores
    for (int i = threadIdx.x; i < TILE * a.RD; i += SW_THREADS) {
      const int row = i % TILE, j = i / TILE, t = t0 + row;
      Ks[j * TILE + row] = (t < a.T) ? __half2float(Yh[(long long)t * a.RD + j]) : 0.f;
    }
    const float* QU = (const float*)(base + a.o_QUd);
    for (int i = threadIdx.x; i < a.RD * D; i += SW_THREADS) {
      const int j = i / D, e = i % D;
      Bs[j * BLD + (e >> 4) * 20 + (e & 15)] = QU[i];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < SW_RPT; ++r)
#pragma unroll
      for (int i = 0; i < SW_EPT / 2; ++i) acc[r][i] = qx[r][i];
    int next = 0;
    for (int j = 0; j < a.RD; ++j) {
      chain_step<LPR>(acc, Ks, Bs, TILE, BLD, j, row0, l);
      if (next < a.ndt && j + 1 == a.rd[next]) {
        score<LPR>(acc, a, cells, (iTfull * a.nd + next) * a.nb, lane);
        ++next;
      }
    }
    __syncthreads();
  }

  // ---- truncated r_T, every r_d: X~ Q^T = U_T W_h, W_h = G_h (Q U_d)^T
  if (a.nTt > 0) {
    for (int id = 0; id < a.nd; ++id) {
      const __half* Ug = (const __half*)(base + a.o_UT16) + (long long)id * a.T * a.RT;
      for (int i = threadIdx.x; i < TILE * a.RT; i += SW_THREADS) {
        const int row = i % TILE, k = i / TILE, t = t0 + row;
        Ks[k * TILE + row] = (t < a.T) ? __half2float(Ug[(long long)t * a.RT + k]) : 0.f;
      }
      const float* Wg = (const float*)(base + a.o_W) + ((long long)id * a.H + h) * a.RT * D;
      for (int i = threadIdx.x; i < a.RT * D; i += SW_THREADS) {
        const int k = i / D, e = i % D;
        Bs[k * BLD + (e >> 4) * 20 + (e & 15)] = Wg[i];
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < SW_RPT; ++r)
#pragma unroll
        for (int i = 0; i < SW_EPT / 2; ++i) acc[r][i] = qx[r][i];
      int next = 0;
      for (int k = 0; k < a.RT; ++k) {
        chain_step<LPR>(acc, Ks, Bs, TILE, BLD, k, row0, l);
        if (next < a.nTt && k + 1 == a.rT[next]) {
          score<LPR>(acc, a, cells, (next * a.nd + id) * a.nb, lane);
          ++next;
        }
      }
      __syncthreads();
    }
  }

  __syncthreads();
  float* part = a.part + u * a.part_us + ((long long)h * a.tiles_t + tt) * (a.ncand + 1);
  for (int i = threadIdx.x; i <= a.ncand; i += SW_THREADS) part[i] = cells[i];
}

// QUd[j][:] = Q Ud16[:, j] (one warp per column j).
template <int EPT>
__global__ void rotate_ud_kernel(char* ws, size_t ub, const int8_t* signs, size_t o_Ud16, int RD,
                                 size_t o_QUd) {
  constexpr int D = 32 * EPT;
  const int u = blockIdx.y;
  const int j = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (j >= RD) return;
  const __half* Ud = (const __half*)(ws + u * ub + o_Ud16);
  float v[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = lane * EPT + e;
    v[e] = __half2float(Ud[(long long)i * RD + j]) * (float)signs[(long long)u * D + i];
  }
  fwht_row<EPT>(v, lane);
  const float rs = rsqrtf((float)D);
  float* out = (float*)(ws + u * ub + o_QUd) + (long long)j * D;
#pragma unroll
  for (int e = 0; e < EPT; ++e) out[lane * EPT + e] = v[e] * rs;
}

// Hs[u][j][d] = sigma_d (-1)^popcount(d & j): B^T of the rotation X diag(sigma) H
// (Sylvester order, unnormalised) for the tensor-core sweep, bf16 (exact).
__global__ void sign_hadamard_kernel(char* ws, size_t ub, const int8_t* signs, size_t o_Hs, int D) {
  const int u = blockIdx.y;
  __nv_bfloat16* Hs = (__nv_bfloat16*)(ws + u * ub + o_Hs);
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < D * D; e += gridDim.x * blockDim.x) {
    const int j = e / D, d = e % D;
    const int sgn = (__popc(d & j) & 1) ? -1 : 1;
    Hs[e] = __float2bfloat16_rn((float)(sgn * (int)signs[(long long)u * D + d]));
  }
}

// W[id][h][k][:] = sum_j G16[id][h][k][j] QUd[j][:]  (r_d < D), or
//                = Q G16[id][h][k][:]                  (r_d = D).
// One launch for every feature rank: block (id, h, u).
struct RdList {
  int rd[JOLT_MAX_GRID];
};
template <int EPT>
__global__ void build_w_kernel(char* ws, size_t ub, const int8_t* signs, size_t o_G16,
                               size_t o_QUd, size_t o_W, int H, int RT, RdList rl, int RD,
                               int staged) {
  constexpr int D = 32 * EPT;
  const int id = blockIdx.x, u = blockIdx.z, h = blockIdx.y;
  const int rdv = rl.rd[id];
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32, nw = blockDim.x / 32;
  char* base = ws + u * ub;
  const __half* G = (const __half*)(base + o_G16) + ((long long)id * H * RT * D) +
                    (long long)h * RT * rdv;
  float* W = (float*)(base + o_W) + ((long long)id * H + h) * RT * D;
  const float rs = rsqrtf((float)D);
  // a truncated rank's rows W[k] = G[k] (Q U_d)^T: Q U_d (r_d x D) and this
  // head's core (RT x r_d) staged in shared memory first
  extern __shared__ float bw_sm[];
  float* qsm = bw_sm;                  // [r_d][D]
  float* gsm = bw_sm + RD * D;         // [RT][r_d]
  const float* QUg = (const float*)(base + o_QUd);
  if (staged && rdv < D) {
    for (int e = threadIdx.x; e < rdv * D; e += blockDim.x) qsm[e] = QUg[e];
    for (int e = threadIdx.x; e < RT * rdv; e += blockDim.x) gsm[e] = __half2float(G[e]);
    __syncthreads();
  }
  for (int k = w; k < RT; k += nw) {
    float v[EPT];
    if (rdv == D) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const int i = lane * EPT + e;
        v[e] = __half2float(G[(long long)k * D + i]) * (float)signs[(long long)u * D + i];
      }
      fwht_row<EPT>(v, lane);
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] *= rs;
    } else {
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = 0.f;
      if (staged) {
        for (int j = 0; j < rdv; ++j) {
          const float g = gsm[k * rdv + j];
#pragma unroll
          for (int e = 0; e < EPT; ++e) v[e] = fmaf(g, qsm[j * D + lane * EPT + e], v[e]);
        }
      } else {
        for (int j = 0; j < rdv; ++j) {
          const float g = __half2float(G[(long long)k * rdv + j]);
#pragma unroll
          for (int e = 0; e < EPT; ++e) v[e] = fmaf(g, QUg[(long long)j * D + lane * EPT + e], v[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) W[(long long)k * D + lane * EPT + e] = v[e];
  }
}

// dist[u][c] = sum_tiles e / sum_tiles ||x||^2 (f64), 0 for an all-zero unit.
// Block (u, group of 32 candidates), 256 threads: warp w sums tiles w, w + 8,
// ... of its lane's candidate, the eight partial sums are then added in warp
// order; every block reduces the ||x||^2 column (slot ncand) in the same
// fixed order.
constexpr int SR_THREADS = 256, SR_WARPS = SR_THREADS / 32;
__global__ void __launch_bounds__(SR_THREADS)
sweep_reduce_kernel(char* ws, size_t ub, const float* part_base, long long part_us,
                    size_t o_status, int ntiles, int ncand, double* dist) {
  const int u = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.y * 32 + lane;
  const float* part = part_base + u * part_us;
  const long long ld = ncand + 1;
  __shared__ double px[SR_WARPS], pc[SR_WARPS][32];
  double sx = 0.0;
  for (int i = threadIdx.x; i < ntiles; i += SR_THREADS) sx += (double)part[(long long)i * ld + ncand];
  for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
  if (lane == 0) px[w] = sx;
  double s = 0.0;
  if (c < ncand)
    for (int i = w; i < ntiles; i += SR_WARPS) s += (double)part[(long long)i * ld + c];
  pc[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < ncand) {
    double xn = 0.0, e = 0.0;
    for (int k = 0; k < SR_WARPS; ++k) {
      xn += px[k];
      e += pc[k][lane];
    }
    const double d = (xn > 0.0) ? e / xn : 0.0;
    if (!isfinite(d) || !isfinite(xn)) atomicOr((int*)(ws + u * ub + o_status), ST_NONFINITE);
    dist[(long long)u * ncand + c] = d;
  }
}

struct CostArgs {
  int H, T, D, nT, nd, nb, block, align, model, ncand;
  int rT[JOLT_MAX_GRID], rd[JOLT_MAX_GRID], b[4];
};

__device__ __forceinline__ long long al(long long x, long long a) { return (x + a - 1) / a * a; }

__global__ void cost_kernel(CostArgs a, int n_units, int64_t* cost) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_units * a.ncand) return;
  const int c = i % a.ncand;
  const int ib = c % a.nb, id = (c / a.nb) % a.nd, iT = c / (a.nb * a.nd);
  const long long H = a.H, T = a.T, D = a.D, rT = a.rT[iT], rd = a.rd[id], b = a.b[ib];
  const long long n = H * T * D;
  long long v;
  if (a.model == JOLT_COST_FORMULA) {
    v = al(2 * H * (rT * T + rd * rT + rd * D), a.align);
    if (b > 0) v += al(b * n / 8, a.align) + al(2 * n / a.block, a.align);
    v += JOLT_HEADER_BYTES;
  } else {
    long long off = JOLT_HEADER_BYTES;
    const long long secs[5] = {rT == T ? 0 : 2 * T * rT, rd == D ? 0 : 2 * D * rd, 2 * H * rT * rd,
                               b == 0 ? 0 : 2 * (n / a.block), b == 0 ? 0 : n * b / 8};
    for (int s = 0; s < 5; ++s) {
      off = al(off, a.align);
      off += secs[s];
    }
    v = al(off, a.align);
  }
  cost[i] = v;
}

template <int LPR>
jolt_status launch_sweep_t(const SweepArgs& a, int U, cudaStream_t st) {
  constexpr int D = SW_EPT * LPR, TILE = SW_WARPS * (32 / LPR) * SW_RPT, BLD = LPR * 20;
  dim3 grid(a.tiles_t, a.H, U);
  const size_t smem = (size_t)(64 * TILE + 64 * BLD + a.ncand + 1) * sizeof(float);
  (void)D;
  if (a.dtype == JOLT_BF16) {
    static bool s1 = false;
    if (!s1) {
      JOLT_CUDA_TRY(cudaFuncSetAttribute(sweep_kernel<__nv_bfloat16, LPR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
      s1 = true;
    }
    sweep_kernel<__nv_bfloat16, LPR><<<grid, SW_THREADS, smem, st>>>(a);
  } else {
    static bool s2 = false;
    if (!s2) {
      JOLT_CUDA_TRY(cudaFuncSetAttribute(sweep_kernel<float, LPR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
      s2 = true;
    }
    sweep_kernel<float, LPR><<<grid, SW_THREADS, smem, st>>>(a);
  }
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace

jolt_status sweep_prep(const Layout& L, int U, const int8_t* signs, char* ws, cudaStream_t st) {
  const size_t ub = L.unit_bytes;
  const int EPT = L.D / 32;
  // rotated factors
  if (L.RD > 0) {
    dim3 g((L.RD + 7) / 8, U);
    if (EPT == 4) rotate_ud_kernel<4><<<g, 256, 0, st>>>(ws, ub, signs, L.o_Ud16, L.RD, L.o_QUd);
    else if (EPT == 2) rotate_ud_kernel<2><<<g, 256, 0, st>>>(ws, ub, signs, L.o_Ud16, L.RD, L.o_QUd);
    else rotate_ud_kernel<1><<<g, 256, 0, st>>>(ws, ub, signs, L.o_Ud16, L.RD, L.o_QUd);
    JOLT_LAUNCH_CHECK();
  }
  if (L.o_Hs != 0) {
    sign_hadamard_kernel<<<dim3(16, U), 256, 0, st>>>(ws, ub, signs, L.o_Hs, L.D);
    JOLT_LAUNCH_CHECK();
  }
  if (L.RT > 0) {
    RdList rl;
    for (int id = 0; id < JOLT_MAX_GRID; ++id) rl.rd[id] = id < L.nd ? L.rd[id] : 0;
    dim3 g(L.nd, L.H, U);
    // Q U_d (RD x D) and one head's core (RT x RD) in shared memory when
    // they fit the default 48 KB, else read from global memory
    const size_t need = ((size_t)L.RD * L.D + (size_t)L.RT * L.RD) * 4;
    const int staged = need <= 48 * 1024 ? 1 : 0;
    const size_t smem = staged ? need : 0;
    if (EPT == 4) build_w_kernel<4><<<g, 256, smem, st>>>(ws, ub, signs, L.o_G16, L.o_QUd, L.o_W, L.H, L.RT, rl, L.RD, staged);
    else if (EPT == 2) build_w_kernel<2><<<g, 256, smem, st>>>(ws, ub, signs, L.o_G16, L.o_QUd, L.o_W, L.H, L.RT, rl, L.RD, staged);
    else build_w_kernel<1><<<g, 256, smem, st>>>(ws, ub, signs, L.o_G16, L.o_QUd, L.o_W, L.H, L.RT, rl, L.RD, staged);
    JOLT_LAUNCH_CHECK();
  }
  return JOLT_OK;
}

jolt_status sweep_run(const Layout& L, int U, const void* X, const int8_t* signs, char* ws,
                      double* dist, int64_t* cost, cudaStream_t st, float* part_override) {
  const size_t ub = L.unit_bytes;
  const int D = L.D;
  {
    jolt_status s0 = sweep_prep(L, U, signs, ws, st);
    if (s0 != JOLT_OK) return s0;
  }
  SweepArgs a;
  a.X = X; a.signs = signs; a.ws = ws; a.ub = ub;
  a.H = L.H; a.T = L.T; a.D = D; a.dtype = L.dtype;
  a.nT = L.nT; a.nd = L.nd; a.nb = L.nb; a.nTt = L.nTt; a.ndt = L.ndt; a.RT = L.RT; a.RD = L.RD;
  a.hasFullT = L.hasFullT; a.hasFullD = L.hasFullD;
  for (int i = 0; i < JOLT_MAX_GRID; ++i) {
    a.rT[i] = i < L.nTt ? L.rT[i] : -1;
    a.rd[i] = i < L.ndt ? L.rd[i] : -1;
  }
  for (int i = 0; i < 4; ++i) a.b[i] = L.b[i];
  a.ncand = L.ncand;
  a.tiles_t = (L.T + L.tile_rows - 1) / L.tile_rows;
  for (int i = 0; i < 4; ++i) a.rq[i] = L.b[i] > 0 ? 1.f / (float)((1 << (L.b[i] - 1)) - 1) : 0.f;
  a.o_UT16 = L.o_UT16; a.o_W = L.o_W; a.o_Y16 = L.o_Y16; a.o_QUd = L.o_QUd;
  if (part_override) {
    a.part = part_override;
    a.part_us = (long long)L.ntiles * (L.ncand + 1);
  } else {
    a.part = (float*)(ws + L.o_part);
    a.part_us = (long long)ub / 4;
  }
  jolt_status s;
  int ntiles = L.ntiles;
  // optional timing events around the fused kernel alone (measurement hook)
  if (g_sweep_ev[0]) JOLT_CUDA_TRY(cudaEventRecord((cudaEvent_t)g_sweep_ev[0], st));
  if (sweep_tc_supported(L)) {
    int tiles_t = 0;
    s = sweep_tc_run(L, U, X, ws, a.part, a.part_us, &tiles_t, st);
    ntiles = L.H * tiles_t;
  } else if (D == 128) {
    s = launch_sweep_t<8>(a, U, st);
  } else if (D == 64) {
    s = launch_sweep_t<4>(a, U, st);
  } else {
    s = launch_sweep_t<2>(a, U, st);
  }
  if (g_sweep_ev[1]) JOLT_CUDA_TRY(cudaEventRecord((cudaEvent_t)g_sweep_ev[1], st));
  if (s != JOLT_OK) return s;
  sweep_reduce_kernel<<<dim3(U, (L.ncand + 31) / 32), SR_THREADS, 0, st>>>(
      ws, ub, a.part, a.part_us, L.o_status, ntiles, L.ncand, dist);
  JOLT_LAUNCH_CHECK();
  CostArgs ca;
  ca.H = L.H; ca.T = L.T; ca.D = D; ca.nT = L.nT; ca.nd = L.nd; ca.nb = L.nb;
  ca.block = L.block; ca.align = L.align; ca.model = L.cost_model; ca.ncand = L.ncand;
  for (int i = 0; i < JOLT_MAX_GRID; ++i) { ca.rT[i] = L.rT[i]; ca.rd[i] = L.rd[i]; }
  for (int i = 0; i < 4; ++i) ca.b[i] = L.b[i];
  cost_kernel<<<(U * L.ncand + 255) / 256, 256, 0, st>>>(ca, U, cost);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace jolt
