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

namespace {

constexpr int SW_WARPS = 8;
constexpr int SW_ROWS = 8;                       // rows per warp
constexpr int SW_TILE = SW_WARPS * SW_ROWS;      // 64 rows per CTA
constexpr int SW_THREADS = SW_WARPS * 32;

struct SweepArgs {
  const void* X;
  const int8_t* signs;
  char* ws;
  size_t ub;
  int H, T, D, dtype;
  int nT, nd, nb, nTt, ndt, RT, RD, hasFullT, hasFullD;
  int rT[JOLT_MAX_GRID], rd[JOLT_MAX_GRID], b[4];
  int ncand, tiles_t;
  size_t o_UT16, o_W, o_Y16, o_QUd, o_part;
};

template <typename TX, int EPT>
__device__ __forceinline__ void load_row(const TX* row, int lane, float (&v)[EPT]) {
#pragma unroll
  for (int e = 0; e < EPT; ++e) v[e] = to_f32(row[lane * EPT + e]);
}

// Score one candidate: acc holds Q R for the warp's rows.
template <int EPT>
__device__ __forceinline__ void score(const float (&acc)[SW_ROWS][EPT], const SweepArgs& a,
                                      float* cells, int cell0, int lane) {
  float m[SW_ROWS];
  float e0 = 0.f;
#pragma unroll
  for (int r = 0; r < SW_ROWS; ++r) {
    float mm = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      mm = fmaxf(mm, fabsf(acc[r][e]));
      e0 = fmaf(acc[r][e], acc[r][e], e0);
    }
    m[r] = mm;
  }
#pragma unroll
  for (int r = 0; r < SW_ROWS; ++r) m[r] = warp_max(m[r]);
  for (int ib = 0; ib < a.nb; ++ib) {
    const int b = a.b[ib];
    float eb;
    if (b == 0) {
      eb = e0;
    } else {
      const float qmax = (float)((1 << (b - 1)) - 1);
      eb = 0.f;
#pragma unroll
      for (int r = 0; r < SW_ROWS; ++r) {
        const float s = round_f16(__fdiv_rn(m[r], qmax));
        const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          const float q = rint_magic(acc[r][e] * inv);
          const float d = fmaf(-s, q, acc[r][e]);
          eb = fmaf(d, d, eb);
        }
      }
    }
    eb = warp_sum(eb);
    if (lane == 0) atomicAdd(&cells[cell0 + ib], eb);
  }
}

template <typename TX, int EPT>
__global__ void __launch_bounds__(SW_THREADS) sweep_kernel(SweepArgs a) {
  constexpr int D = 32 * EPT;
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;                     // [64][SW_TILE]  chain coefficients, k-major
  float* Bs = Ks + 64 * SW_TILE;        // [64][D]        rotated factor rows
  float* cells = Bs + 64 * D;           // [ncand + 1]

  const int u = blockIdx.z, h = blockIdx.y, tt = blockIdx.x;
  const int t0 = tt * SW_TILE;
  const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
  char* base = a.ws + u * a.ub;
  for (int i = threadIdx.x; i <= a.ncand; i += SW_THREADS) cells[i] = 0.f;

  // ---- load X rows, rotate once: qx = H (sigma .* x) / sqrt(D)
  const TX* Xu = (const TX*)a.X + ((long long)u * a.H + h) * a.T * D;
  float sg[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) sg[e] = (float)a.signs[(long long)u * D + lane * EPT + e];
  const float rs = rsqrtf((float)D);
  float x[SW_ROWS][EPT], qx[SW_ROWS][EPT];
  float xn = 0.f;
#pragma unroll
  for (int r = 0; r < SW_ROWS; ++r) {
    const int t = t0 + w * SW_ROWS + r;
    if (t < a.T) {
      load_row<TX, EPT>(Xu + (long long)t * D, lane, x[r]);
    } else {
#pragma unroll
      for (int e = 0; e < EPT; ++e) x[r][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      xn = fmaf(x[r][e], x[r][e], xn);
      qx[r][e] = x[r][e] * sg[e];
    }
    fwht_row<EPT>(qx[r], lane);
#pragma unroll
    for (int e = 0; e < EPT; ++e) qx[r][e] *= rs;
  }
  __syncthreads();  // cells cleared
  xn = warp_sum(xn);
  if (lane == 0) atomicAdd(&cells[a.ncand], xn);

  float acc[SW_ROWS][EPT];
  const int iTfull = a.nT - 1, idfull = a.nd - 1;

  // ---- (r_T, r_d) = (T, D): the stored core is fp16(X) itself
  if (a.hasFullT && a.hasFullD) {
#pragma unroll
    for (int r = 0; r < SW_ROWS; ++r) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[r][e] = (x[r][e] - round_f16(x[r][e])) * sg[e];
      fwht_row<EPT>(acc[r], lane);
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[r][e] *= rs;
    }
    score<EPT>(acc, a, cells, (iTfull * a.nd + idfull) * a.nb, lane);
  }

  // ---- r_T = T, truncated r_d: X~ Q^T = Y16 (Q U_d)^T, prefix over r_d
  if (a.hasFullT && a.ndt > 0) {
    const __half* Yh = (const __half*)(base + a.o_Y16) + (long long)h * a.T * a.RD;
    for (int i = threadIdx.x; i < SW_TILE * a.RD; i += SW_THREADS) {
      const int row = i / a.RD, j = i % a.RD;
      const int t = t0 + row;
      Ks[j * SW_TILE + row] = (t < a.T) ? __half2float(Yh[(long long)t * a.RD + j]) : 0.f;
    }
    const float* QU = (const float*)(base + a.o_QUd);
    for (int i = threadIdx.x; i < a.RD * D; i += SW_THREADS) Bs[i] = QU[i];
    __syncthreads();
#pragma unroll
    for (int r = 0; r < SW_ROWS; ++r)
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[r][e] = qx[r][e];
    int next = 0;
    for (int j = 0; j < a.RD; ++j) {
      const float* kk = Ks + j * SW_TILE + w * SW_ROWS;
      const float* bb = Bs + j * D + lane * EPT;
      float bv[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) bv[e] = bb[e];
#pragma unroll
      for (int r = 0; r < SW_ROWS; ++r) {
        const float kr = kk[r];
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[r][e] = fmaf(-kr, bv[e], acc[r][e]);
      }
      if (next < a.ndt && j + 1 == a.rd[next]) {
        score<EPT>(acc, a, cells, (iTfull * a.nd + next) * a.nb, lane);
        ++next;
      }
    }
    __syncthreads();
  }

  // ---- truncated r_T, every r_d: X~ Q^T = U_T W_h, W_h = G_h (Q U_d)^T
  if (a.nTt > 0) {
    for (int id = 0; id < a.nd; ++id) {
      const __half* Ug = (const __half*)(base + a.o_UT16) + (long long)id * a.T * a.RT;
      for (int i = threadIdx.x; i < SW_TILE * a.RT; i += SW_THREADS) {
        const int row = i / a.RT, k = i % a.RT;
        const int t = t0 + row;
        Ks[k * SW_TILE + row] = (t < a.T) ? __half2float(Ug[(long long)t * a.RT + k]) : 0.f;
      }
      const float* Wg = (const float*)(base + a.o_W) + ((long long)id * a.H + h) * a.RT * D;
      for (int i = threadIdx.x; i < a.RT * D; i += SW_THREADS) Bs[i] = Wg[i];
      __syncthreads();
#pragma unroll
      for (int r = 0; r < SW_ROWS; ++r)
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[r][e] = qx[r][e];
      int next = 0;
      for (int k = 0; k < a.RT; ++k) {
        const float* kk = Ks + k * SW_TILE + w * SW_ROWS;
        const float* bb = Bs + k * D + lane * EPT;
        float bv[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) bv[e] = bb[e];
#pragma unroll
        for (int r = 0; r < SW_ROWS; ++r) {
          const float kr = kk[r];
#pragma unroll
          for (int e = 0; e < EPT; ++e) acc[r][e] = fmaf(-kr, bv[e], acc[r][e]);
        }
        if (next < a.nTt && k + 1 == a.rT[next]) {
          score<EPT>(acc, a, cells, (next * a.nd + id) * a.nb, lane);
          ++next;
        }
      }
      __syncthreads();
    }
  }

  __syncthreads();
  float* part = (float*)(base + a.o_part) + ((long long)h * a.tiles_t + tt) * (a.ncand + 1);
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

// W[id][h][k][:] = sum_j G16[id][h][k][j] QUd[j][:]  (r_d < D), or
//                = Q G16[id][h][k][:]                  (r_d = D).
template <int EPT>
__global__ void build_w_kernel(char* ws, size_t ub, const int8_t* signs, size_t o_G16,
                               size_t o_QUd, size_t o_W, int H, int RT, int id, int rdv) {
  constexpr int D = 32 * EPT;
  const int u = blockIdx.z, h = blockIdx.y;
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32, nw = blockDim.x / 32;
  char* base = ws + u * ub;
  const __half* G = (const __half*)(base + o_G16) + ((long long)id * H * RT * D) +
                    (long long)h * RT * rdv;
  float* W = (float*)(base + o_W) + ((long long)id * H + h) * RT * D;
  const float rs = rsqrtf((float)D);
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
      const float* QU = (const float*)(base + o_QUd);
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = 0.f;
      for (int j = 0; j < rdv; ++j) {
        const float g = __half2float(G[(long long)k * rdv + j]);
#pragma unroll
        for (int e = 0; e < EPT; ++e) v[e] = fmaf(g, QU[(long long)j * D + lane * EPT + e], v[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) W[(long long)k * D + lane * EPT + e] = v[e];
  }
}

// dist[u][c] = sum_tiles e / sum_tiles ||x||^2 (f64), 0 for an all-zero unit.
__global__ void sweep_reduce_kernel(char* ws, size_t ub, size_t o_part, size_t o_status, int ntiles,
                                    int ncand, double* dist) {
  const int u = blockIdx.x;
  const float* part = (const float*)(ws + u * ub + o_part);
  __shared__ double xn;
  if (threadIdx.x < 32) {
    double s = 0.0;
    for (int i = threadIdx.x; i < ntiles; i += 32) s += (double)part[(long long)i * (ncand + 1) + ncand];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) xn = s;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < ncand; c += blockDim.x) {
    double s = 0.0;
    for (int i = 0; i < ntiles; ++i) s += (double)part[(long long)i * (ncand + 1) + c];
    double d = (xn > 0.0) ? s / xn : 0.0;
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

template <int EPT>
jolt_status launch_sweep_t(const SweepArgs& a, int U, size_t smem, cudaStream_t st) {
  dim3 grid(a.tiles_t, a.H, U);
  if (a.dtype == JOLT_BF16) {
    static bool s1 = false;
    if (!s1) {
      JOLT_CUDA_TRY(cudaFuncSetAttribute(sweep_kernel<__nv_bfloat16, EPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
      s1 = true;
    }
    sweep_kernel<__nv_bfloat16, EPT><<<grid, SW_THREADS, smem, st>>>(a);
  } else {
    static bool s2 = false;
    if (!s2) {
      JOLT_CUDA_TRY(cudaFuncSetAttribute(sweep_kernel<float, EPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
      s2 = true;
    }
    sweep_kernel<float, EPT><<<grid, SW_THREADS, smem, st>>>(a);
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
  if (L.RT > 0) {
    for (int id = 0; id < L.nd; ++id) {
      dim3 g(1, L.H, U);
      if (EPT == 4) build_w_kernel<4><<<g, 256, 0, st>>>(ws, ub, signs, L.o_G16, L.o_QUd, L.o_W, L.H, L.RT, id, L.rd[id]);
      else if (EPT == 2) build_w_kernel<2><<<g, 256, 0, st>>>(ws, ub, signs, L.o_G16, L.o_QUd, L.o_W, L.H, L.RT, id, L.rd[id]);
      else build_w_kernel<1><<<g, 256, 0, st>>>(ws, ub, signs, L.o_G16, L.o_QUd, L.o_W, L.H, L.RT, id, L.rd[id]);
      JOLT_LAUNCH_CHECK();
    }
  }
  return JOLT_OK;
}

jolt_status sweep_run(const Layout& L, int U, const void* X, const int8_t* signs, char* ws,
                      double* dist, int64_t* cost, cudaStream_t st) {
  const size_t ub = L.unit_bytes;
  const int D = L.D, EPT = D / 32;
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
  a.tiles_t = (L.T + SW_TILE - 1) / SW_TILE;
  a.o_UT16 = L.o_UT16; a.o_W = L.o_W; a.o_Y16 = L.o_Y16; a.o_QUd = L.o_QUd; a.o_part = L.o_part;
  const size_t smem = (size_t)(64 * SW_TILE + 64 * D + L.ncand + 1) * sizeof(float);
  jolt_status s;
  if (EPT == 4) s = launch_sweep_t<4>(a, U, smem, st);
  else if (EPT == 2) s = launch_sweep_t<2>(a, U, smem, st);
  else s = launch_sweep_t<1>(a, U, smem, st);
  if (s != JOLT_OK) return s;
  sweep_reduce_kernel<<<U, 128, 0, st>>>(ws, ub, L.o_part, L.o_status, L.H * a.tiles_t, L.ncand,
                                        dist);
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
