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
#include "chol_smem.cuh"

namespace jolt {

namespace {

constexpr int JAC_THREADS = 1024;   // viewed as 32 x 32 (ty, tx)
constexpr int JAC_MAX_SWEEPS = 40;
int g_max_sweeps = JAC_MAX_SWEEPS;   // sweep cap of every Jacobi solve (host-settable)
constexpr float JAC_TOL = 1e-6f;    // relative: |a_pq| vs sqrt(|a_pp a_qq|)
constexpr float FEAT_TOL = 4e-6f;   // one-sided: |b_p . b_q| vs |b_p| |b_q| (fp32 dot products)
// absolute floors vs ||A||_F: JAC_ABS_EXACT for solves whose small
// eigenvalues matter; JAC_ABS_RR for Rayleigh-Ritz blocks, whose trailing
// Ritz vectors only seed the next block

__global__ void __launch_bounds__(JAC_THREADS, 1)
jacobi_kernel(const float* __restrict__ Ain, long long a_bs, int lda, int n, int nparts,
              long long part_s, float* __restrict__ evals, long long e_bs,
              float* __restrict__ evecs, long long v_bs, int ldv, int ncols_out, int* status,
              long long s_bs, const int* skip, long long sk_s, float abs_tol, int max_sweeps) {
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
  abs_floor = abs_tol * sqrtf(abs_floor);

  bool converged = false;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
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

// The same cyclic Jacobi method with the matrix and the accumulated
// rotations held in registers, after Brent & Luk (1985): one thread per 2x2
// block.  1024 threads form a 32 x 32 grid; thread (I, J) owns NB x NB blocks
// at block coordinates (I + 32a, J + 32b).  Every round pairs positions
// (2k, 2k+1); after the round the matrix indices move between positions by
// the round-robin (circle) permutation, so that over m - 1 rounds every pair
// of indices meets once and after a whole sweep every index is back in its
// original position.  Per round: the diagonal-block threads compute their
// rotation from their own registers, every thread applies J_i^T B J_j to its
// A blocks and B J_j to its V blocks, then scatters them to the permuted
// positions through shared memory (two barriers per round).
template <int NB>
__global__ void __launch_bounds__(1024, 1)
jacobi_bl_kernel(const float* __restrict__ Ain, long long a_bs, int lda, int n, int nparts,
                 long long part_s, float* __restrict__ evals, long long e_bs,
                 float* __restrict__ evecs, long long v_bs, int ldv, int ncols_out, int* status,
                 long long s_bs, const int* skip, long long sk_s, float abs_tol,
                 int max_sweeps) {
  const int bidx = blockIdx.x;
  if (skip && skip[bidx * sk_s]) return;
  const int m = n + (n & 1);      // even size; a padded index stays zero
  const int nb = m / 2;           // blocks per dimension
  const int pl = nb + 1;          // plane row stride
  extern __shared__ float sm[];
  float* PA = sm;                 // A as 4 planes [x][y][nb][pl]
  float* PV = PA + 4 * nb * pl;   // V as 4 planes
  float4* cs = (float4*)(PV + 4 * nb * pl);   // [nb] (c, s, t, -)
  int* perm = (int*)(cs + nb);                // [m] position -> next position
  const int t = threadIdx.x, J = t & 31, I = t >> 5;

  // circle slots: slot 0 fixed, slots 1..m-1 advance by one per round; the
  // pair (slot k, slot m-1-k) sits at positions (2k, 2k+1)
  for (int sl = t; sl < m; sl += blockDim.x) {
    auto pos = [&](int q) { return q < nb ? 2 * q : 2 * (m - 1 - q) + 1; };
    const int nx = (sl == 0) ? 0 : (sl == m - 1 ? 1 : sl + 1);
    perm[pos(sl)] = pos(nx);
  }
  const float* Ag = Ain + bidx * a_bs;
  float a[NB][NB][4], v[NB][NB][4];
  float fro = 0.f;
#pragma unroll
  for (int x = 0; x < NB; ++x)
#pragma unroll
    for (int y = 0; y < NB; ++y) {
      const int BI = I + 32 * x, BJ = J + 32 * y;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 2 * BI + (e >> 1), c = 2 * BJ + (e & 1);
        float val = 0.f;
        if (BI < nb && BJ < nb && r < n && c < n) {
          for (int k = 0; k < nparts; ++k)
            val += Ag[k * part_s + (long long)r * lda + c] + Ag[k * part_s + (long long)c * lda + r];
          val *= 0.5f;
        }
        a[x][y][e] = val;
        v[x][y][e] = (r == c && r < n) ? 1.f : 0.f;
        fro = fmaf(val, val, fro);
      }
    }
  __shared__ float fro_part[32];
  fro = warp_sum(fro);
  if (J == 0) fro_part[I] = fro;
  __syncthreads();
  float abs_floor = 0.f;
  for (int i = 0; i < 32; ++i) abs_floor += fro_part[i];
  abs_floor = abs_tol * sqrtf(abs_floor);
  // destinations of this thread's elements under the fixed permutation, and
  // its own (gather) offsets, in the 4-plane layout
  int dstA[NB][NB][4], dstV[NB][NB][4], own[NB][NB][4];
#pragma unroll
  for (int x = 0; x < NB; ++x)
#pragma unroll
    for (int y = 0; y < NB; ++y) {
      const int BI = I + 32 * x, BJ = J + 32 * y;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = BI < nb && BJ < nb;
        const int P = in ? perm[2 * BI + (e >> 1)] : 0, Q = in ? perm[2 * BJ + (e & 1)] : 0;
        const int Rw = 2 * BI + (e >> 1);
        dstA[x][y][e] = (((P & 1) * 2 + (Q & 1)) * nb + (P >> 1)) * pl + (Q >> 1);
        dstV[x][y][e] = (((Rw & 1) * 2 + (Q & 1)) * nb + (Rw >> 1)) * pl + (Q >> 1);
        own[x][y][e] = (((e >> 1) * 2 + (e & 1)) * nb + BI) * pl + BJ;
      }
    }

  bool converged = false;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    int rotated = 0;
    for (int r = 0; r < m - 1; ++r) {
      // 1. rotations of the pairs, from the diagonal blocks
#pragma unroll
      for (int x = 0; x < NB; ++x) {
        const int BI = I + 32 * x;
        if (x < NB && J + 32 * x == BI && BI < nb) {
          // this thread owns diagonal block (BI, BI) when y == x
          float* bl = a[x][x];
          const float app = bl[0], aqq = bl[3], apq = bl[1];
          float c = 1.f, sn = 0.f, tt = 0.f;
          const float thr = JAC_TOL * sqrtf(fabsf(app) * fabsf(aqq));
          if (fabsf(apq) > thr && fabsf(apq) > abs_floor && fabsf(apq) > 1e-30f) {
            const float tau = (aqq - app) / (2.f * apq);
            if (fabsf(tau) > 1e9f) tt = 0.5f / tau;
            else tt = copysignf(1.f, tau) / (fabsf(tau) + sqrtf(1.f + tau * tau));
            c = rsqrtf(1.f + tt * tt);
            sn = tt * c;
            rotated = 1;
          }
          cs[BI] = make_float4(c, sn, tt, 0.f);
        }
      }
      __syncthreads();
      // 2. rotate own blocks, 3. scatter to the permuted positions
#pragma unroll
      for (int x = 0; x < NB; ++x)
#pragma unroll
        for (int y = 0; y < NB; ++y) {
          const int BI = I + 32 * x, BJ = J + 32 * y;
          if (BI >= nb || BJ >= nb) continue;
          const float4 ri = cs[BI], rj = cs[BJ];
          float* b = a[x][y];
          if (BI == BJ) {
            const float app = b[0], aqq = b[3], apq = b[1];
            if (ri.y != 0.f) {
              b[0] = app - ri.z * apq;
              b[3] = aqq + ri.z * apq;
              b[1] = 0.f;
              b[2] = 0.f;
            }
          } else {
            const float a1 = rj.x * b[0] - rj.y * b[1], b1 = rj.y * b[0] + rj.x * b[1];
            const float c1 = rj.x * b[2] - rj.y * b[3], d1 = rj.y * b[2] + rj.x * b[3];
            b[0] = ri.x * a1 - ri.y * c1;
            b[2] = ri.y * a1 + ri.x * c1;
            b[1] = ri.x * b1 - ri.y * d1;
            b[3] = ri.y * b1 + ri.x * d1;
          }
          float* w = v[x][y];
          const float w0 = rj.x * w[0] - rj.y * w[1], w1 = rj.y * w[0] + rj.x * w[1];
          const float w2 = rj.x * w[2] - rj.y * w[3], w3 = rj.y * w[2] + rj.x * w[3];
          w[0] = w0; w[1] = w1; w[2] = w2; w[3] = w3;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            PA[dstA[x][y][e]] = b[e];
            PV[dstV[x][y][e]] = w[e];   // V rows do not move
          }
        }
      __syncthreads();
      // 4. gather own positions
#pragma unroll
      for (int x = 0; x < NB; ++x)
#pragma unroll
        for (int y = 0; y < NB; ++y) {
          const int BI = I + 32 * x, BJ = J + 32 * y;
          if (BI >= nb || BJ >= nb) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            a[x][y][e] = PA[own[x][y][e]];
            v[x][y][e] = PV[own[x][y][e]];
          }
        }
    }
    if (!__syncthreads_or(rotated)) { converged = true; break; }
  }
  if (t == 0 && status) {
    if (!converged) atomicOr(status + bidx * s_bs, ST_NOCONVERGE);
    atomicMax(status + bidx * s_bs + 1, sweep);
  }
  // positions are back to the identity: diagonal = eigenvalues, V columns =
  // eigenvectors; write them to plain n x n layouts in shared memory
  float* Dg = PA;                 // [m] eigenvalues
  float* Vf = PA + m;             // [n][n+1]
  __syncthreads();
#pragma unroll
  for (int x = 0; x < NB; ++x)
#pragma unroll
    for (int y = 0; y < NB; ++y) {
      const int BI = I + 32 * x, BJ = J + 32 * y;
      if (BI >= nb || BJ >= nb) continue;
      if (BI == BJ) { Dg[2 * BI] = a[x][y][0]; Dg[2 * BI + 1] = a[x][y][3]; }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 2 * BI + (e >> 1), c = 2 * BJ + (e & 1);
        if (r < n && c < n) Vf[r * (n + 1) + c] = v[x][y][e];
      }
    }
  __syncthreads();
  // descending order, ties to the lower index; sign rule as in jacobi_kernel
  float* ev = evals + bidx * e_bs;
  float* vg = evecs + bidx * v_bs;
  for (int i = t; i < n; i += blockDim.x) {
    const float li = Dg[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const float lj = Dg[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    ev[rank] = li;
    if (rank < ncols_out) {
      float big = -1.f, sgn = 1.f;
      for (int row = 0; row < n; ++row) {
        const float vv = Vf[row * (n + 1) + i];
        if (fabsf(vv) > big) { big = fabsf(vv); sgn = vv < 0.f ? -1.f : 1.f; }
      }
      for (int row = 0; row < n; ++row) vg[(long long)row * ldv + rank] = sgn * Vf[row * (n + 1) + i];
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

// The same factorisation for n = N <= 64 in fp32, returning R^{-1} instead
// of R, blocked by 8 columns so that the serial dependency chain is short:
// per block column, warp 0 factors the 8 x 8 diagonal block in registers
// (pivot and column entries broadcast by shuffle), one thread per row solves
// its panel row against it, and all threads apply the rank-8 update to the
// trailing lower triangle.  X = L'^{-1} follows blockwise: the diagonal
// blocks by substitution (one thread per row), then X_ik = -X_ii sum_{m=k}^{i-1}
// L_im X_mk, one block diagonal at a time.  R^{-1} = S^{-1} X^T with S the
// equilibration scales.
template <int N>
__global__ void __launch_bounds__(256)
chol_inv_kernel(const float* __restrict__ G, long long g_bs, int nparts, long long part_s,
                float* __restrict__ Rinv, long long r_bs, int* status, long long s_bs,
                const int* skip, long long sk_s, float shift) {
  constexpr int NT = 256;
  constexpr int LD = N + 1;
  const int u = blockIdx.x;
  if (skip && skip[u * sk_s]) return;
  __shared__ float S[N * LD];    // the Gram, then L' (lower)
  __shared__ float X[N * LD];    // L'^{-1} (lower); the gathered partial products
  __shared__ float rds[N];
  __shared__ float rpiv[N];      // 1 / L'_jj
  __shared__ int bad;
  const int t = threadIdx.x;
  const float* Gg = G + u * g_bs;
  if (t == 0) bad = 0;
  {
    // every load of the (up to 4) partials in flight at once
    constexpr int PER = (N * N + NT - 1) / NT;
    float g[4][PER];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = t + i * NT;
        g[p][i] = (p < nparts && e < N * N) ? Gg[p * part_s + e] : 0.f;
      }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = t + i * NT;
      if (e < N * N) X[(e / N) * LD + e % N] = (g[0][i] + g[1][i]) + (g[2][i] + g[3][i]);  // raw Gram, staged in X
    }
  }
  chol_inv_smem<N>(S, X, rds, rpiv, &bad, shift);
  // R^{-1}[k][r] = X[r][k] / s_k
  float* Rg = Rinv + u * r_bs;
  for (int e = t; e < N * N; e += NT) {
    const int k = e / N, r = e % N;
    Rg[e] = k <= r ? X[r * LD + k] * rds[k] : 0.f;
  }
  if (t == 0 && bad && status) atomicOr(status + u * s_bs, ST_NOTPD);
}

// The RPT rows of lane l (of 16) in a shared-memory column: rows 4l..4l+3 of
// every 64-row chunk (RPT % 4 == 0), else rows RPT l .. RPT l + RPT - 1; each
// access of the 16 lanes is one contiguous stretch.
template <int RPT>
__device__ __forceinline__ void ld_rows(const float* col, int l, float (&v)[RPT]) {
  if constexpr (RPT % 4 == 0) {
#pragma unroll
    for (int c = 0; c < RPT / 4; ++c) {
      const float4 x = *reinterpret_cast<const float4*>(col + 64 * c + 4 * l);
      v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
    }
  } else if constexpr (RPT == 2) {
    const float2 x = *reinterpret_cast<const float2*>(col + 2 * l);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int i = 0; i < RPT; ++i) v[i] = col[RPT * l + i];
  }
}
template <int RPT>
__device__ __forceinline__ void st_rows(float* col, int l, const float (&v)[RPT]) {
  if constexpr (RPT % 4 == 0) {
#pragma unroll
    for (int c = 0; c < RPT / 4; ++c)
      *reinterpret_cast<float4*>(col + 64 * c + 4 * l) =
          make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  } else if constexpr (RPT == 2) {
    *reinterpret_cast<float2*>(col + 2 * l) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int i = 0; i < RPT; ++i) col[RPT * l + i] = v[i];
  }
}

// Double-float arithmetic (an unevaluated sum hi + lo of two floats, about
// 48 significant bits; Dekker 1971), for the feature Cholesky: the fp64 pipe
// of this part is far slower than fp32, and this factorisation needs more
// than fp32 accuracy.
struct df { float h, l; };
__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ df df_norm(float s, float e) {
  const float h = s + e;
  return df{h, e - (h - s)};
}
__device__ __forceinline__ df df_mul(df a, df b) {
  const float p = a.h * b.h;
  float e = fmaf(a.h, b.h, -p);
  e = fmaf(a.h, b.l, fmaf(a.l, b.h, e));
  return df_norm(p, e);
}
// a - b c
__device__ __forceinline__ df df_fnma(df a, df b, df c) {
  const float p = b.h * c.h;
  float pe = fmaf(b.h, c.h, -p);
  pe = fmaf(b.h, c.l, fmaf(b.l, c.h, pe));
  const float s = a.h - p;
  const float bb = s - a.h;
  float e = (a.h - (s - bb)) + (-p - bb);
  e += a.l - pe;
  return df_norm(s, e);
}
// 1 / sqrt(d) for d > 0: one Newton step y + y (1 - d y^2) / 2 from the fp32
// estimate, the residual taken in double-float.
__device__ __forceinline__ df df_rsqrt(df d) {
  const float y = rsqrtf(d.h);
  const df y2 = df_mul(df{y, 0.f}, df{y, 0.f});
  const df r = df_fnma(df{1.f, 0.f}, d, y2);   // 1 - d y^2
  return df_norm(y, 0.5f * y * r.h);
}

// Eigenpairs of the feature Gram by one-sided Jacobi (Hestenes 1958; its
// relative accuracy: Demmel & Veselic 1992).  S = B B^T with B = diag(s) L',
// L' the Cholesky factor (double-float) of the equilibrated S' = diag(s)^-1
// S diag(s)^-1.  Plane rotations applied to the columns of B (fp32) drive
// them to mutual orthogonality, B J = U Sigma; then S = U Sigma^2 U^T: the
// eigenvectors are the normalised columns and the eigenvalues their squared
// norms, so no rotation product has to be accumulated.  Columns live in
// shared memory; each round of the round-robin (circle) ordering gives the
// N/2 disjoint pairs to N/2 groups of 16 threads, each thread holding N/16
// rows of its two columns in registers (rows 4l..4l+3 of every 64-row chunk
// for lane l, so that the 16-byte loads of a group are contiguous).  A pair
// is rotated while |b_p . b_q| > tol sqrt(|b_p|^2 |b_q|^2) and above an
// absolute floor; a sweep without rotations ends the solve.  A pivot that is
// not positive (rank-deficient S) or a zero column leaves the unit's `done`
// flag clear, and the caller solves that unit with the two-sided Jacobi.
// Input: the sum of nparts partials G + b*g_bs + p*part_s (row stride lda),
// symmetrised; TIn is double or float.
template <int N, typename TIn>
__global__ void __launch_bounds__(8 * N, 1)
sym_eig_kernel(const TIn* __restrict__ G, long long g_bs, int lda, int nparts, long long part_s,
               float* __restrict__ evals, long long e_bs, float* __restrict__ evecs,
               long long v_bs, int ldv, int ncols_out, int* status, long long st_bs, int* done,
               long long d_bs, const int* skip, long long sk_s, float tol, float abs_tol,
               int max_sweeps) {
  constexpr int NT = 8 * N;
  constexpr int TY = NT / 32;   // thread rows of the Cholesky update
  constexpr int RPT = N / 16;   // Jacobi rows per thread
  constexpr int LDA = N + 1;
  constexpr int LDM = N + 4;    // column stride, 16-byte aligned
  extern __shared__ __align__(16) unsigned char fe_sm[];
  df* A = (df*)fe_sm;                    // N x LDA: S', then L' (lower)
  df* dsc = A + N * LDA;                 // [N] sqrt(S_ii)
  float* M = (float*)(dsc + N);          // N columns of LDM floats
  float* lam = M + N * LDM;              // [N] squared column norms
  __shared__ int fail;
  __shared__ float fro_part[NT / 32];
  const int u = blockIdx.x, t = threadIdx.x, tx = t & 31, ty = t >> 5;
  if (skip && skip[u * sk_s]) {
    if (t == 0) done[u * d_bs] = 1;   // nothing to solve
    return;
  }
  if (t == 0) done[u * d_bs] = 0;
  const TIn* Gg = G + u * g_bs;
  if (t == 0) fail = 0;
  // stage sum_p G_p (not yet symmetrised) in A as double-floats; each
  // thread's loads of all partials are in flight together
  constexpr int PER = (N * N + NT - 1) / NT;
  constexpr int CH = PER < 8 ? PER : 8;     // elements per chunk
#pragma unroll 1
  for (int c0 = 0; c0 < PER; c0 += CH) {
    double g[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) g[i] = 0.0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      if (p >= nparts) break;
      TIn v[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int e = t + (c0 + i) * NT;
        v[i] = e < N * N ? Gg[p * part_s + (long long)(e / N) * lda + e % N] : (TIn)0;
      }
#pragma unroll
      for (int i = 0; i < CH; ++i) g[i] += (double)v[i];
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int e = t + (c0 + i) * NT;
      if (e < N * N) {
        const float h = (float)g[i];
        A[(e / N) * LDA + e % N] = df{h, (float)(g[i] - (double)h)};
      }
    }
  }
  __syncthreads();
  // s_i = sqrt(S_ii) and 1 / s_i (f64, N values), Frobenius norm of S
  if (t < N) {
    const df a = A[t * LDA + t];
    const double d = (double)a.h + (double)a.l;
    const double sd = d > 0.0 ? sqrt(d) : 0.0;
    const double r = sd > 0.0 ? 1.0 / sd : 0.0;
    const float sh = (float)sd, rh = (float)r;
    dsc[t] = df{sh, (float)(sd - (double)sh)};
    lam[t] = 0.f;
    M[t] = rh;                                  // scratch: 1 / s_i (hi, lo)
    M[N + t] = (float)(r - (double)rh);
  }
  float fro = 0.f;
  for (int e = t; e < N * N; e += NT) {
    const float v = A[(e / N) * LDA + e % N].h;
    fro = fmaf(v, v, fro);
  }
  fro = warp_sum(fro);
  if (tx == 0) fro_part[ty] = fro;
  __syncthreads();
  float fro_s = 0.f;
  for (int i = 0; i < NT / 32; ++i) fro_s += fro_part[i];
  const float floor_abs = abs_tol * sqrtf(fro_s);
  // S'_ij = (S_ij + S_ji) / (2 s_i s_j), lower triangle, double-float (the
  // upper triangle is only read)
  for (int e = t; e < N * N; e += NT) {
    const int i = e / N, j = e % N;
    if (j <= i) {
      const df x = A[i * LDA + j], y = A[j * LDA + i];
      float sh, se;
      two_sum_f(x.h, y.h, sh, se);
      const df v = df_norm(0.5f * sh, 0.5f * (se + x.l + y.l));
      A[i * LDA + j] = df_mul(df_mul(v, df{M[i], M[N + i]}), df{M[j], M[N + j]});
    }
  }
  __syncthreads();
  // right-looking Cholesky S' = L' L'^T in double-float, lower triangle in
  // place; thread (ty, tx) updates rows ty + TY a and columns tx + 32 b
  for (int j = 0; j < N; ++j) {
    const df d = A[j * LDA + j];
    if (!(d.h > 1e-30f)) {
      if (t == 0) fail = 1;
      break;  // uniform: every thread read the same pivot
    }
    const df rp = df_rsqrt(d);
    for (int i = j + 1 + t; i < N; i += NT) A[i * LDA + j] = df_mul(A[i * LDA + j], rp);
    __syncthreads();
    if (t == 0) A[j * LDA + j] = df_mul(d, rp);
    for (int i = j + 1 + ty; i < N; i += TY) {
      const df li = A[i * LDA + j];
      for (int k = j + 1 + tx; k <= i; k += 32)
        A[i * LDA + k] = df_fnma(A[i * LDA + k], li, A[k * LDA + j]);
    }
    __syncthreads();
  }
  __syncthreads();
  if (fail) return;
  // B = diag(s) L' as fp32 columns: M[c][r] = s_r L'[r][c] (r >= c)
  for (int e = t; e < N * N; e += NT) {
    const int c = e / N, r = e % N;
    M[c * LDM + r] = r >= c ? df_mul(dsc[r], A[r * LDA + c]).h : 0.f;
  }
  __syncthreads();
  const int k = t >> 4, l16 = t & 15;
  bool converged = false;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    // exact squared column norms at the start of every sweep (group k: columns
    // 2k and 2k + 1); each rotation then updates the pair's norms by
    // |b_p'|^2 = |b_p|^2 - t g, |b_q'|^2 = |b_q|^2 + t g (t = tan of the
    // angle), so a round computes only the cross product g
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float v[RPT];
      ld_rows<RPT>(M + (2 * k + cc) * LDM, l16, v);
      float s2 = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) s2 = fmaf(v[i], v[i], s2);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      if (l16 == 0) lam[2 * k + cc] = s2;
    }
    __syncthreads();
    int rot = 0;
    for (int r = 0; r < N - 1; ++r) {
      int p, q;
      if (k == 0) { p = N - 1; q = r; }
      else {
        p = r + k; if (p >= N - 1) p -= N - 1;
        q = r - k; if (q < 0) q += N - 1;
      }
      float cp[RPT], cq[RPT];
      ld_rows<RPT>(M + p * LDM, l16, cp);
      ld_rows<RPT>(M + q * LDM, l16, cq);
      float g0 = 0.f, g1 = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; i += 2) {
        g0 = fmaf(cp[i], cq[i], g0);
        if (i + 1 < RPT) g1 = fmaf(cp[i + 1], cq[i + 1], g1);
      }
      float g = g0 + g1;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
      const float a = lam[p], b = lam[q];
      if (fabsf(g) > tol * sqrtf(a * b) && fabsf(g) > floor_abs) {
        // rotation parameters with the approximate (few-ulp) intrinsics: an
        // angle off by an ulp only leaves a residue for the next sweep, and
        // the column transform stays orthogonal to rounding
        const float zeta = __fdividef(b - a, 2.f * g);
        const float tt = __fdividef(copysignf(1.f, zeta), fabsf(zeta) + __fsqrt_rn(fmaf(zeta, zeta, 1.f)));
        const float c = rsqrtf(fmaf(tt, tt, 1.f)), s = tt * c;
        float np_[RPT], nq_[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          np_[i] = c * cp[i] - s * cq[i];
          nq_[i] = s * cp[i] + c * cq[i];
        }
        st_rows<RPT>(M + p * LDM, l16, np_);
        st_rows<RPT>(M + q * LDM, l16, nq_);
        if (l16 == 0) {
          lam[p] = fmaf(-tt, g, a);
          lam[q] = fmaf(tt, g, b);
        }
        rot = 1;
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rot)) { converged = true; ++sweep; break; }
  }
  // eigenvalues = squared column norms; descending, ties to the lower index
  for (int c = t; c < N; c += NT) {
    float s = 0.f;
    for (int r = 0; r < N; ++r) s = fmaf(M[c * LDM + r], M[c * LDM + r], s);
    lam[c] = s;
    if (!(s > 0.f)) fail = 1;
  }
  __syncthreads();
  if (fail) return;
  float* ev = evals + u * e_bs;
  float* vg = evecs + u * v_bs;
  for (int c = t; c < N; c += NT) {
    const float lc = lam[c];
    int rank = 0;
    for (int j = 0; j < N; ++j) {
      const float lj = lam[j];
      rank += (lj > lc) || (lj == lc && j < c);
    }
    ev[rank] = lc;
    if (rank >= ncols_out) continue;
    // unit column, sign fixed so that its largest-magnitude entry (lowest
    // index on a tie) is positive
    const float inv = rsqrtf(lc);
    float big = -1.f, sgn = 1.f;
    for (int r = 0; r < N; ++r) {
      const float v = M[c * LDM + r];
      if (fabsf(v) > big) { big = fabsf(v); sgn = v < 0.f ? -1.f : 1.f; }
    }
    for (int r = 0; r < N; ++r) vg[(long long)r * ldv + rank] = sgn * inv * M[c * LDM + r];
  }
  if (t == 0) {
    if (status) {
      if (!converged) atomicOr(status + u * st_bs, ST_NOCONVERGE);
      atomicMax(status + u * st_bs + 1, sweep);   // diagnostics: most sweeps used
    }
    done[u * d_bs] = 1;
  }
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
                          const int* skip, long long sk_s, float abs_tol, cudaStream_t st) {
  if (n <= 0 || n > 128 || batch <= 0) return n <= 0 ? JOLT_OK : JOLT_ERR_INVALID;
  const int m = n + (n & 1), nb = m / 2;
  if (nb <= 32) {
    // register-resident Brent-Luk variant
    const size_t pl = (size_t)nb + 1;
    size_t smem = (8 * nb * pl) * sizeof(float) + nb * sizeof(float4) + m * sizeof(int);
    const size_t need_out = ((size_t)m + (size_t)n * (n + 1)) * sizeof(float);
    if (smem < need_out) smem = need_out;
    static bool attr_bl = false;
    if (!attr_bl) {
      JOLT_CUDA_TRY(cudaFuncSetAttribute(jacobi_bl_kernel<1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
      attr_bl = true;
    }
    jacobi_bl_kernel<1><<<batch, 1024, smem, st>>>(A, a_bs, lda, n, nparts < 1 ? 1 : nparts,
                                                   part_s, evals, e_bs, evecs, v_bs, ldv,
                                                   ncols_out, status, s_bs, skip, sk_s, abs_tol,
                                                   g_max_sweeps);
    JOLT_LAUNCH_CHECK();
    return JOLT_OK;
  }
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
                                                  s_bs, skip, sk_s, abs_tol, g_max_sweeps);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

template <typename R>
static jolt_status chol_launch(const float* G, long long g_bs, int n, int nparts, long long part_s,
                               int batch, float* Rout, long long r_bs, int* status, long long s_bs,
                               const int* skip, long long sk_s, float shift, cudaStream_t st) {
  nparts = nparts < 1 ? 1 : nparts;
  const size_t smem = (size_t)(n * (n + 1) + n) * sizeof(R);
  static bool attr_set = false;
  if (!attr_set) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(chol_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       200 * 1024));
    attr_set = true;
  }
  chol_kernel<R><<<batch, 1024, smem, st>>>(G, g_bs, n, nparts, part_s, Rout, r_bs, status, s_bs,
                                           skip, sk_s, shift);
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

jolt_status launch_chol_inv(const float* G, long long g_bs, int n, int nparts, long long part_s,
                            int batch, float* Rinv, long long r_bs, int* status, long long s_bs,
                            const int* skip, long long sk_s, float shift, cudaStream_t st) {
  if (n <= 0 || batch <= 0) return JOLT_OK;
  nparts = nparts < 1 ? 1 : nparts;
  if (nparts > 4) return JOLT_ERR_INVALID;
  switch (n) {
    case 64: chol_inv_kernel<64><<<batch, 256, 0, st>>>(G, g_bs, nparts, part_s, Rinv, r_bs, status, s_bs, skip, sk_s, shift); break;
    case 48: chol_inv_kernel<48><<<batch, 256, 0, st>>>(G, g_bs, nparts, part_s, Rinv, r_bs, status, s_bs, skip, sk_s, shift); break;
    case 40: chol_inv_kernel<40><<<batch, 256, 0, st>>>(G, g_bs, nparts, part_s, Rinv, r_bs, status, s_bs, skip, sk_s, shift); break;
    case 32: chol_inv_kernel<32><<<batch, 256, 0, st>>>(G, g_bs, nparts, part_s, Rinv, r_bs, status, s_bs, skip, sk_s, shift); break;
    default: return JOLT_ERR_INVALID;
  }
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

jolt_status launch_sym_eig(const void* G, bool f64_in, long long g_bs, int lda, int n, int nparts,
                           long long part_s, int batch, float* evals, long long e_bs,
                           float* evecs, long long v_bs, int ldv, int ncols_out, int* status,
                           long long st_bs, int* done, long long d_bs, const int* skip,
                           long long sk_s, float abs_tol, cudaStream_t st) {
  if (batch <= 0) return JOLT_OK;
  if (!done) return JOLT_ERR_INVALID;
  nparts = nparts < 1 ? 1 : nparts;
  auto go = [&](auto kern, int N, auto* gp) -> jolt_status {
    const size_t smem = (size_t)N * (N + 1) * 8 + (size_t)N * 8 + (size_t)N * (N + 4) * 4 + N * 4;
    JOLT_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<batch, 8 * N, smem, st>>>(gp, g_bs, lda, nparts, part_s, evals, e_bs, evecs, v_bs, ldv,
                                     ncols_out, status, st_bs, done, d_bs, skip, sk_s, FEAT_TOL,
                                     abs_tol, g_max_sweeps);
    JOLT_LAUNCH_CHECK();
    return JOLT_OK;
  };
  const double* gd = (const double*)G;
  const float* gf = (const float*)G;
  switch (n) {
    case 128: return f64_in ? go(sym_eig_kernel<128, double>, 128, gd) : go(sym_eig_kernel<128, float>, 128, gf);
    case 64: return f64_in ? go(sym_eig_kernel<64, double>, 64, gd) : go(sym_eig_kernel<64, float>, 64, gf);
    case 32: return f64_in ? go(sym_eig_kernel<32, double>, 32, gd) : go(sym_eig_kernel<32, float>, 32, gf);
    default: return JOLT_ERR_INVALID;
  }
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

void set_max_sweeps(int n) { g_max_sweeps = n > 0 ? n : JAC_MAX_SWEEPS; }

}  // namespace jolt
