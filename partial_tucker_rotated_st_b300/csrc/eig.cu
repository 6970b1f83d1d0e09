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

constexpr int JAC_THREADS = 512;
constexpr int JAC_MAX_SWEEPS = 40;
constexpr float JAC_TOL = 1e-6f;

__global__ void __launch_bounds__(JAC_THREADS)
jacobi_kernel(const float* __restrict__ Ain, long long a_bs, int lda, int n,
              float* __restrict__ evals, long long e_bs, float* __restrict__ evecs,
              long long v_bs, int ldv, int ncols_out, int* status, long long s_bs,
              const int* skip, long long sk_s) {
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
  int* cnt = qq + half;          // rotation counter
  const int t = threadIdx.x;

  const float* Ag = Ain + bidx * a_bs;
  for (int e = t; e < n * n; e += blockDim.x) {
    const int i = e / n, j = e % n;
    A[i * ld + j] = 0.5f * (Ag[(long long)i * lda + j] + Ag[(long long)j * lda + i]);
    V[i * ld + j] = (i == j) ? 1.f : 0.f;
  }
  __syncthreads();

  bool converged = false;
  for (int sweep = 0; sweep < JAC_MAX_SWEEPS; ++sweep) {
    if (t == 0) *cnt = 0;
    __syncthreads();
    for (int r = 0; r < m - 1; ++r) {
      if (t < half) {
        int p, q;
        if (t == 0) { p = m - 1; q = r; }
        else { p = (r + t) % (m - 1); q = (r - t + (m - 1)) % (m - 1); }
        float c = 1.f, s = 0.f, np = 0.f, nq = 0.f;
        if (p < n && q < n) {
          const float apq = A[p * ld + q];
          const float app = A[p * ld + p], aqq = A[q * ld + q];
          np = app; nq = aqq;
          const float thr = JAC_TOL * sqrtf(fabsf(app) * fabsf(aqq));
          if (fabsf(apq) > thr && fabsf(apq) > 1e-30f) {
            const float tau = (aqq - app) / (2.f * apq);
            float tt;
            if (fabsf(tau) > 1e9f) tt = 0.5f / tau;
            else tt = copysignf(1.f, tau) / (fabsf(tau) + sqrtf(1.f + tau * tau));
            c = 1.f / sqrtf(1.f + tt * tt);
            s = tt * c;
            np = app - tt * apq;
            nq = aqq + tt * apq;
            atomicAdd(cnt, 1);
          }
        }
        pp[t] = p; qq[t] = q; cs[t] = c; sn[t] = s; dp[t] = np; dq[t] = nq;
      }
      __syncthreads();
      // A <- J^T A J on 2x2 blocks (rows of pair i, columns of pair j)
      for (int e = t; e < half * half; e += blockDim.x) {
        const int i = e / half, j = e % half;
        const float ci = cs[i], si = sn[i], cj = cs[j], sj = sn[j];
        if (si == 0.f && sj == 0.f) continue;
        const int pi = pp[i], qi = qq[i], pj = pp[j], qj = qq[j];
        if (i == j) {
          A[pi * ld + pi] = dp[i];
          A[qi * ld + qi] = dq[i];
          A[pi * ld + qi] = 0.f;
          A[qi * ld + pi] = 0.f;
          continue;
        }
        const bool vpi = pi < n, vqi = qi < n, vpj = pj < n, vqj = qj < n;
        const float a = (vpi && vpj) ? A[pi * ld + pj] : 0.f;
        const float b = (vpi && vqj) ? A[pi * ld + qj] : 0.f;
        const float c = (vqi && vpj) ? A[qi * ld + pj] : 0.f;
        const float d = (vqi && vqj) ? A[qi * ld + qj] : 0.f;
        const float a1 = cj * a - sj * b, b1 = sj * a + cj * b;
        const float c1 = cj * c - sj * d, d1 = sj * c + cj * d;
        const float a2 = ci * a1 - si * c1, c2 = si * a1 + ci * c1;
        const float b2 = ci * b1 - si * d1, d2 = si * b1 + ci * d1;
        if (vpi && vpj) A[pi * ld + pj] = a2;
        if (vpi && vqj) A[pi * ld + qj] = b2;
        if (vqi && vpj) A[qi * ld + pj] = c2;
        if (vqi && vqj) A[qi * ld + qj] = d2;
      }
      // V <- V J
      for (int e = t; e < n * half; e += blockDim.x) {
        const int row = e / half, k = e % half;
        const float s = sn[k];
        if (s == 0.f) continue;
        const float c = cs[k];
        const int p = pp[k], q = qq[k];
        const float vp = V[row * ld + p], vq = V[row * ld + q];
        V[row * ld + p] = c * vp - s * vq;
        V[row * ld + q] = s * vp + c * vq;
      }
      __syncthreads();
    }
    if (*cnt == 0) { converged = true; break; }
    __syncthreads();
  }
  if (!converged && t == 0 && status) atomicOr(status + bidx * s_bs, ST_NOCONVERGE);

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

// Cholesky G = L L^T (left-looking, column by column), then R^{-1} = L^{-T}.
template <typename R>
__global__ void chol_inv_kernel(const float* __restrict__ G, long long g_bs, int n,
                                float* __restrict__ Rinv, long long r_bs, int* status,
                                long long s_bs, const int* skip, long long sk_s) {
  const int bidx = blockIdx.x;
  if (skip && skip[bidx * sk_s]) return;
  extern __shared__ __align__(16) unsigned char smraw[];
  R* Lm = (R*)smraw;            // n x n, lower
  R* X = Lm + n * n;            // n x n, L^{-1}
  __shared__ int bad;
  const int t = threadIdx.x;
  const float* Gg = G + bidx * g_bs;
  if (t == 0) bad = 0;
  for (int e = t; e < n * n; e += blockDim.x) {
    const int i = e / n, j = e % n;
    Lm[e] = (R)(0.5f * (Gg[i * n + j] + Gg[j * n + i]));
    X[e] = 0;
  }
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    // pivot
    if (t == 0) {
      R d = Lm[j * n + j];
      for (int k = 0; k < j; ++k) d -= Lm[j * n + k] * Lm[j * n + k];
      // an exactly zero pivot is a zero column (an all-zero block): it is
      // kept as a null direction; a negative one means lost definiteness
      if (d < (R)0 || d != d) { bad = 1; d = (R)0; }
      Lm[j * n + j] = sqrt(d);
    }
    __syncthreads();
    const R piv = Lm[j * n + j];
    for (int i = j + 1 + t; i < n; i += blockDim.x) {
      R v = Lm[i * n + j];
      for (int k = 0; k < j; ++k) v -= Lm[i * n + k] * Lm[j * n + k];
      Lm[i * n + j] = piv > (R)0 ? v / piv : (R)0;
    }
    __syncthreads();
  }
  // columns of L^{-1} by forward substitution, one thread per column
  for (int c = t; c < n; c += blockDim.x) {
    X[c * n + c] = Lm[c * n + c] > (R)0 ? (R)1 / Lm[c * n + c] : (R)0;
    for (int i = c + 1; i < n; ++i) {
      R v = 0;
      for (int k = c; k < i; ++k) v += Lm[i * n + k] * X[k * n + c];
      X[i * n + c] = Lm[i * n + i] > (R)0 ? -v / Lm[i * n + i] : (R)0;
    }
  }
  __syncthreads();
  float* Rg = Rinv + bidx * r_bs;
  // R^{-1} = (L^{-1})^T: Rinv[i][j] = X[j][i]
  for (int e = t; e < n * n; e += blockDim.x) {
    const int i = e / n, j = e % n;
    Rg[e] = (float)X[j * n + i];
  }
  if (t == 0 && bad && status) atomicOr(status + bidx * s_bs, ST_NOTPD);
}

}  // namespace

jolt_status launch_jacobi(const float* A, long long a_bs, int lda, int n, int batch,
                          float* evals, long long e_bs, float* evecs, long long v_bs, int ldv,
                          int ncols_out, int* status, long long s_bs, const int* skip,
                          long long sk_s, cudaStream_t st) {
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
  jacobi_kernel<<<batch, JAC_THREADS, smem, st>>>(A, a_bs, lda, n, evals, e_bs, evecs, v_bs, ldv,
                                                  ncols_out, status, s_bs, skip, sk_s);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

template <typename R>
static jolt_status chol_launch(const float* G, long long g_bs, int n, int batch, float* Rinv,
                               long long r_bs, int* status, long long s_bs, const int* skip,
                               long long sk_s, cudaStream_t st) {
  const size_t smem = (size_t)2 * n * n * sizeof(R);
  static bool attr_set = false;
  if (!attr_set) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(chol_inv_kernel<R>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
    attr_set = true;
  }
  chol_inv_kernel<R><<<batch, 128, smem, st>>>(G, g_bs, n, Rinv, r_bs, status, s_bs, skip, sk_s);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

jolt_status launch_chol_inv(const float* G, long long g_bs, int n, int batch, float* Rinv,
                            long long r_bs, int* status, long long s_bs, const int* skip,
                            long long sk_s, bool f64, cudaStream_t st) {
  if (n <= 0 || batch <= 0) return JOLT_OK;
  if (n > 128 || (f64 && n > 64)) return JOLT_ERR_INVALID;
  if (f64) return chol_launch<double>(G, g_bs, n, batch, Rinv, r_bs, status, s_bs, skip, sk_s, st);
  return chol_launch<float>(G, g_bs, n, batch, Rinv, r_bs, status, s_bs, skip, sk_s, st);
}

}  // namespace jolt
