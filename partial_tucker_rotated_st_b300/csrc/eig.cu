// Small dense symmetric eigen-solves and Cholesky factors, one CTA per matrix.
//
// Jacobi: the two-sided cyclic Jacobi method (Golub & Van Loan, "Matrix
// Computations", 8.5: symmetric Schur rotation, cyclic sweep), with each
// sweep visited in round-robin order (Brent & Luk 1985) so that the n/2
// rotations of one round act on disjoint index pairs and are applied at once.
// A pair is rotated only while |a_pq| > tol * sqrt(|a_pp a_qq|), the relative
// threshold that keeps small eigenvalues accurate; a sweep without rotations
// ends the solve.  The matrix and the accumulated rotations live in shared
// memory (fp32).
#include "jolt_internal.cuh"

namespace jolt {

namespace {

constexpr int JAC_THREADS = 1024;   // viewed as 32 x 32 (ty, tx)
constexpr int JAC_MAX_SWEEPS = 40;
constexpr float JAC_TOL = 1e-6f;    // relative: |a_pq| vs sqrt(|a_pp a_qq|)
constexpr float JAC_ABS = 1e-10f;   // absolute floor vs ||A||_F: stops rotations on pure noise

__global__ void __launch_bounds__(JAC_THREADS, 1)
jacobi_kernel(const float* __restrict__ Ain, long long a_bs, int lda, int n, int nparts,
              long long part_s, float* __restrict__ evals, long long e_bs,
              float* __restrict__ evecs, long long v_bs, int ldv, int ncols_out, int* status,
              long long s_bs, const int* skip, long long sk_s) {
  const int bidx = blockIdx.x;
  if (skip && skip[bidx * sk_s]) return;
  extern __shared__ float sm[];
  const int ld = n + 1;
  float* A = sm;                 // n x (n+1)
  float* V = A + n * ld;         // n x (n+1)
  const int m = n + (n & 1);     // players incl. a dummy for odd n
  const int half = m / 2;
  float* cs = V + n * ld;        // [half] cosines
  float* sn = cs + half;         // [half] sines
  float* dp = sn + half;         // [half] new a_pp
  float* dq = dp + half;         // [half] new a_qq
  int* pp = (int*)(dq + half);   // [half]
  int* qq = pp + half;           // [half]
  const int t = threadIdx.x, tx = t & 31, ty = t >> 5;

  const float* Ag = Ain + bidx * a_bs;
  __shared__ float fro_part[JAC_THREADS / 32];
  float fro = 0.f;
  for (int i = ty; i < n; i += 32)
    for (int j = tx; j < n; j += 32) {
      float a = 0.f;
      for (int k = 0; k < nparts; ++k)
        a += Ag[k * part_s + (long long)i * lda + j] + Ag[k * part_s + (long long)j * lda + i];
      a *= 0.5f;
      A[i * ld + j] = a;
      V[i * ld + j] = (i == j) ? 1.f : 0.f;
      fro = fmaf(a, a, fro);
    }
  fro = warp_sum(fro);
  if (tx == 0) fro_part[ty] = fro;
  __syncthreads();
  float abs_floor = 0.f;
  for (int i = 0; i < 32; ++i) abs_floor += fro_part[i];
  abs_floor = JAC_ABS * sqrtf(abs_floor);

  bool converged = false;
  int sweep = 0;
  for (; sweep < JAC_MAX_SWEEPS; ++sweep) {
    int rotated = 0;
    for (int r = 0; r < m - 1; ++r) {
      if (t < half) {
        int p, q;
        if (t == 0) { p = m - 1; q = r; }
        else {
          p = r + t; if (p >= m - 1) p -= m - 1;
          q = r - t; if (q < 0) q += m - 1;
        }
        float c = 1.f, s = 0.f, np = 0.f, nq = 0.f;
        if (p < n && q < n) {
          const float apq = A[p * ld + q];
          const float app = A[p * ld + p], aqq = A[q * ld + q];
          np = app; nq = aqq;
          const float thr = JAC_TOL * sqrtf(fabsf(app) * fabsf(aqq));
          if (fabsf(apq) > thr && fabsf(apq) > abs_floor && fabsf(apq) > 1e-30f) {
            const float tau = (aqq - app) / (2.f * apq);
            float tt;
            if (fabsf(tau) > 1e9f) tt = 0.5f / tau;
            else tt = copysignf(1.f, tau) / (fabsf(tau) + sqrtf(1.f + tau * tau));
            c = rsqrtf(1.f + tt * tt);
            s = tt * c;
            np = app - tt * apq;
            nq = aqq + tt * apq;
            rotated = 1;
          }
        }
        pp[t] = p; qq[t] = q; cs[t] = c; sn[t] = s; dp[t] = np; dq[t] = nq;
      }
      __syncthreads();
      // A <- J^T A J on 2x2 blocks (rows of pair i, columns of pair j)
      for (int i = ty; i < half; i += 32) {
        const float ci = cs[i], si = sn[i];
        const int pi = pp[i], qi = qq[i];
        const bool vpi = pi < n, vqi = qi < n;
        for (int j = tx; j < half; j += 32) {
          const float cj = cs[j], sj = sn[j];
          if (si == 0.f && sj == 0.f) continue;
          const int pj = pp[j], qj = qq[j];
          if (i == j) {
            A[pi * ld + pi] = dp[i];
            A[qi * ld + qi] = dq[i];
            A[pi * ld + qi] = 0.f;
            A[qi * ld + pi] = 0.f;
            continue;
          }
          const bool vpj = pj < n, vqj = qj < n;
          const float a = (vpi && vpj) ? A[pi * ld + pj] : 0.f;
          const float b = (vpi && vqj) ? A[pi * ld + qj] : 0.f;
          const float c = (vqi && vpj) ? A[qi * ld + pj] : 0.f;
          const float d = (vqi && vqj) ? A[qi * ld + qj] : 0.f;
          const float a1 = cj * a - sj * b, b1 = sj * a + cj * b;
          const float c1 = cj * c - sj * d, d1 = sj * c + cj * d;
          if (vpi && vpj) A[pi * ld + pj] = ci * a1 - si * c1;
          if (vpi && vqj) A[pi * ld + qj] = ci * b1 - si * d1;
          if (vqi && vpj) A[qi * ld + pj] = si * a1 + ci * c1;
          if (vqi && vqj) A[qi * ld + qj] = si * b1 + ci * d1;
        }
      }
      // V <- V J
      for (int k = tx; k < half; k += 32) {
        const float s = sn[k];
        if (s == 0.f) continue;
        const float c = cs[k];
        const int p = pp[k], q = qq[k];
        for (int row = ty; row < n; row += 32) {
          const float vp = V[row * ld + p], vq = V[row * ld + q];
          V[row * ld + p] = c * vp - s * vq;
          V[row * ld + q] = s * vp + c * vq;
        }
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) { converged = true; break; }
  }
  if (t == 0 && status) {
    if (!converged) atomicOr(status + bidx * s_bs, ST_NOCONVERGE);
    atomicMax(status + bidx * s_bs + 1, sweep);   // diagnostics: most sweeps used
  }

  // descending order, ties to the lower index; each eigenvector's sign is
  // fixed so that its entry of largest magnitude (lowest index on a tie) is
  // positive
  float* ev = evals + bidx * e_bs;
  float* vg = evecs + bidx * v_bs;
  for (int i = t; i < n; i += blockDim.x) {
    const float li = A[i * ld + i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const float lj = A[j * ld + j];
      rank += (lj > li) || (lj == li && j < i);
    }
    ev[rank] = li;
    if (rank < ncols_out) {
      float big = -1.f, sgn = 1.f;
      for (int row = 0; row < n; ++row) {
        const float v = V[row * ld + i];
        if (fabsf(v) > big) { big = fabsf(v); sgn = v < 0.f ? -1.f : 1.f; }
      }
      for (int row = 0; row < n; ++row) vg[(long long)row * ldv + rank] = sgn * V[row * ld + i];
    }
  }
}

// Cholesky G = R^T R of a sum of split-K partials, right-looking: after
// column j is scaled by its pivot, the trailing block takes the rank-1 update
// in parallel.  An exactly zero pivot (a zero column) is kept as a null
// direction; a negative one records ST_NOTPD.  Writes R (upper, f32).
template <typename R>
__global__ void __launch_bounds__(1024, 1)
chol_kernel(const float* __restrict__ G, long long g_bs, int n, int nparts, long long part_s,
            float* __restrict__ Rout, long long r_bs, int* status, long long s_bs,
            const int* skip, long long sk_s, float shift) {
  const int bidx = blockIdx.x;
  if (skip && skip[bidx * sk_s]) return;
  extern __shared__ __align__(16) unsigned char smraw[];
  const int ld = n + 1;
  R* A = (R*)smraw;  // n x (n+1), lower triangle becomes L
  __shared__ int bad;
  const int t = threadIdx.x, tx = t & 31, ty = t >> 5, lane = tx, warp = ty;
  const float* Gg = G + bidx * g_bs;
  if (t == 0) bad = 0;
  R* dsc = A + n * ld;  // [n] column scales sqrt(G_ii)
  for (int i = ty; i < n; i += 32)
    for (int j = tx; j < n; j += 32) {
      float a = 0.f;
      for (int k = 0; k < nparts; ++k) a += Gg[k * part_s + i * n + j] + Gg[k * part_s + j * n + i];
      A[i * ld + j] = (R)(0.5f * a);
    }
  __syncthreads();
  // equilibrate: G' = S^-1 G S^-1 with S = diag(sqrt(G_ii)); R = R' S
  for (int i = t; i < n; i += blockDim.x) {
    const R d = A[i * ld + i];
    dsc[i] = d > (R)0 ? sqrt(d) : (R)0;
  }
  __syncthreads();
  // a shift on the unit diagonal keeps the factorisation definite when the
  // columns are close to dependent (shifted CholeskyQR, Fukaya et al. 2020);
  // the caller then takes an unshifted pass
  for (int i = ty; i < n; i += 32)
    for (int j = tx; j < n; j += 32) {
      const R di = dsc[i], dj = dsc[j];
      R v = (di > (R)0 && dj > (R)0) ? A[i * ld + j] / (di * dj) : (R)0;
      if (i == j && di > (R)0) v += (R)shift;
      A[i * ld + j] = v;
    }
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    if (warp == 0) {
      R d = A[j * ld + j];
      if (d < (R)0 || d != d) { if (lane == 0) bad = 1; d = (R)0; }
      const R piv = sqrt(d);
      for (int i = j + 1 + lane; i < n; i += 32)
        A[i * ld + j] = piv > (R)0 ? A[i * ld + j] / piv : (R)0;
      if (lane == 0) A[j * ld + j] = piv;
    }
    __syncthreads();
    for (int i = j + 1 + ty; i < n; i += 32) {
      const R lij = A[i * ld + j];
      for (int k = j + 1 + tx; k <= i; k += 32) A[i * ld + k] -= lij * A[k * ld + j];
    }
    __syncthreads();
  }
  float* Rg = Rout + bidx * r_bs;
  for (int i = ty; i < n; i += 32)
    for (int j = tx; j < n; j += 32)  // R[i][j] = L'[j][i] * s_j for j >= i
      Rg[i * n + j] = (j >= i) ? (float)(A[j * ld + i] * dsc[j]) : 0.f;
  if (t == 0 && bad && status) atomicOr(status + bidx * s_bs, ST_NOTPD);
}

// Out[row] = In[row] R^{-1} for every row of a T x n block, one row per
// thread (forward substitution x R = z) with the row in registers; R upper
// triangular in shared memory.  A zero diagonal gives a zero column.
template <int N>
__global__ void __launch_bounds__(128)
trsm_rows_kernel(const float* __restrict__ In, float* __restrict__ Out, long long blk_bs,
                 const float* __restrict__ Rg, long long r_bs, int T, const int* skip,
                 long long sk_s) {
  const int u = blockIdx.y;
  if (skip && skip[u * sk_s]) return;
  __shared__ float Rs[N * N];
  __shared__ float rd[N];
  const int t = threadIdx.x;
  for (int e = t; e < N * N; e += blockDim.x) Rs[e] = Rg[u * r_bs + e];
  __syncthreads();
  for (int j = t; j < N; j += blockDim.x) rd[j] = Rs[j * N + j] > 0.f ? 1.f / Rs[j * N + j] : 0.f;
  __syncthreads();
  const int row = blockIdx.x * blockDim.x + t;
  if (row >= T) return;
  const float* z = In + u * blk_bs + (long long)row * N;
  float* x = Out + u * blk_bs + (long long)row * N;
  float v[N];
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = z[j];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    float a = v[j];
#pragma unroll
    for (int i = 0; i < j; ++i) a = fmaf(-v[i], Rs[i * N + j], a);
    v[j] = a * rd[j];
  }
#pragma unroll
  for (int j = 0; j < N; ++j) x[j] = v[j];
}

}  // namespace

jolt_status launch_jacobi(const float* A, long long a_bs, int lda, int n, int nparts,
                          long long part_s, int batch, float* evals, long long e_bs, float* evecs,
                          long long v_bs, int ldv, int ncols_out, int* status, long long s_bs,
                          const int* skip, long long sk_s, cudaStream_t st) {
  if (n <= 0 || n > 128 || batch <= 0) return n <= 0 ? JOLT_OK : JOLT_ERR_INVALID;
  const int half = (n + 1) / 2;
  const size_t smem = (size_t)2 * n * (n + 1) * sizeof(float) + 4 * half * sizeof(float) +
                      (2 * half + 4) * sizeof(int);
  static bool attr_set = false;
  if (!attr_set) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       200 * 1024));
    attr_set = true;
  }
  jacobi_kernel<<<batch, JAC_THREADS, smem, st>>>(A, a_bs, lda, n, nparts < 1 ? 1 : nparts, part_s,
                                                  evals, e_bs, evecs, v_bs, ldv, ncols_out, status,
                                                  s_bs, skip, sk_s);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

template <typename R>
static jolt_status chol_launch(const float* G, long long g_bs, int n, int nparts, long long part_s,
                               int batch, float* Rout, long long r_bs, int* status, long long s_bs,
                               const int* skip, long long sk_s, float shift, cudaStream_t st) {
  const size_t smem = (size_t)(n * (n + 1) + n) * sizeof(R);
  static bool attr_set = false;
  if (!attr_set) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(chol_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       200 * 1024));
    attr_set = true;
  }
  chol_kernel<R><<<batch, 1024, smem, st>>>(G, g_bs, n, nparts < 1 ? 1 : nparts, part_s, Rout, r_bs,
                                           status, s_bs, skip, sk_s, shift);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

jolt_status launch_chol(const float* G, long long g_bs, int n, int nparts, long long part_s,
                        int batch, float* Rout, long long r_bs, int* status, long long s_bs,
                        const int* skip, long long sk_s, bool f64, float shift, cudaStream_t st) {
  if (n <= 0 || batch <= 0) return JOLT_OK;
  if (n > 128 || (f64 && n > 64)) return JOLT_ERR_INVALID;
  if (f64)
    return chol_launch<double>(G, g_bs, n, nparts, part_s, batch, Rout, r_bs, status, s_bs, skip,
                               sk_s, shift, st);
  return chol_launch<float>(G, g_bs, n, nparts, part_s, batch, Rout, r_bs, status, s_bs, skip,
                            sk_s, shift, st);
}

jolt_status launch_trsm_rows(const float* In, float* Out, long long blk_bs, const float* R,
                             long long r_bs, int T, int n, int batch, const int* skip,
                             long long sk_s, cudaStream_t st) {
  if (n <= 0 || batch <= 0 || T <= 0) return JOLT_OK;
  const int nt = 128;
  dim3 grid((T + nt - 1) / nt, batch);
  switch (n) {
    case 64: trsm_rows_kernel<64><<<grid, nt, 0, st>>>(In, Out, blk_bs, R, r_bs, T, skip, sk_s); break;
    case 48: trsm_rows_kernel<48><<<grid, nt, 0, st>>>(In, Out, blk_bs, R, r_bs, T, skip, sk_s); break;
    case 40: trsm_rows_kernel<40><<<grid, nt, 0, st>>>(In, Out, blk_bs, R, r_bs, T, skip, sk_s); break;
    case 32: trsm_rows_kernel<32><<<grid, nt, 0, st>>>(In, Out, blk_bs, R, r_bs, T, skip, sk_s); break;
    default: return JOLT_ERR_INVALID;
  }
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace jolt
