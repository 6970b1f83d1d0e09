// Cholesky factorisation and inverse of a small equilibrated Gram in shared
// memory, shared by the CholeskyQR kernels (csrc/eig.cu, csrc/cholqr.cu).
//
// On entry X (N x (N + 1), row stride N + 1) holds the raw Gram G (not yet
// symmetrised).  The block of 256 threads forms S' = D^-1 sym(G) D^-1 + shift I
// (D = diag(sqrt(G_ii))), factors S' = L' L'^T blocked by 8 columns (per
// block column, warp 0 factors the 8 x 8 diagonal block in registers with the
// pivot and column entries broadcast by shuffle, one thread per row solves its
// panel row against it, and all threads apply the rank-8 update to the
// trailing lower triangle), and inverts it blockwise: the diagonal blocks by
// substitution (one thread per row), then X_ik = -X_ii sum_{m=k}^{i-1} L_im
// X_mk, one block diagonal at a time.  On exit X's lower triangle holds
// L'^{-1} and rds[k] = 1 / sqrt(G_kk), so that R^{-1}[k][r] = X[r][k] rds[k]
// (k <= r) with R = L'^T D.  A pivot that is not positive sets *bad and is
// taken as zero.  Ends with the block synchronised.
#pragma once

namespace jolt {

template <int N>
__device__ __forceinline__ void chol_inv_smem(float* S, float* X, float* rds, float* rpiv,
                                              int* bad, float shift) {
  constexpr int NB = 8, NBLK = N / NB, NT = 256;
  constexpr int LD = N + 1;
  static_assert(N % NB == 0 && N <= 64, "block size");
  const int t = threadIdx.x, lane = t & 31, tx = t & 31, ty = t >> 5;
  __syncthreads();
  if (t < N) {
    const float d = X[t * LD + t];
    rds[t] = d > 0.f ? rsqrtf(d) : 0.f;
  }
  __syncthreads();
  // S' = D^-1 sym(G) D^-1 (+ shift on the diagonal), lower triangle
  for (int e = t; e < N * N; e += NT) {
    const int i = e / N, k = e % N;
    if (k <= i) {
      float v = 0.5f * (X[i * LD + k] + X[k * LD + i]) * rds[i] * rds[k];
      if (k == i && rds[i] > 0.f) v += shift;
      S[i * LD + k] = v;
    }
  }
  __syncthreads();
  for (int kb = 0; kb < NBLK; ++kb) {
    const int c0 = kb * NB, c1 = c0 + NB;
    // (a) diagonal block, warp 0: lane r < 8 holds row c0 + r
    if (t < 32) {
      float a[NB];
#pragma unroll
      for (int m = 0; m < NB; ++m) a[m] = (lane < NB && m <= lane) ? S[(c0 + lane) * LD + c0 + m] : 0.f;
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        float d = __shfl_sync(0xffffffffu, a[j], j);
        if (!(d >= 0.f)) { if (lane == 0) *bad = 1; d = 0.f; }
        const float rp = d > 0.f ? rsqrtf(d) : 0.f;
        if (lane == j) { a[j] = d * rp; rpiv[c0 + j] = rp; }
        else if (lane > j) a[j] *= rp;
#pragma unroll
        for (int m = j + 1; m < NB; ++m) {
          const float lm = __shfl_sync(0xffffffffu, a[j], m);
          if (lane >= m && lane < NB) a[m] = fmaf(-a[j], lm, a[m]);
        }
      }
      if (lane < NB)
#pragma unroll
        for (int m = 0; m < NB; ++m)
          if (m <= lane) S[(c0 + lane) * LD + c0 + m] = a[m];
    }
    __syncthreads();
    if (c1 >= N) break;
    // (b) panel: row i solves x L11^T = a, x_m = (a_m - sum_{q<m} x_q L11[m][q]) / L11[m][m]
    for (int i = c1 + t; i < N; i += NT) {
      float x[NB];
#pragma unroll
      for (int m = 0; m < NB; ++m) {
        float v = S[i * LD + c0 + m];
#pragma unroll
        for (int q = 0; q < m; ++q) v = fmaf(-x[q], S[(c0 + m) * LD + c0 + q], v);
        x[m] = v * rpiv[c0 + m];
      }
#pragma unroll
      for (int m = 0; m < NB; ++m) S[i * LD + c0 + m] = x[m];
    }
    __syncthreads();
    // (c) trailing update of the lower triangle: a_ik -= sum_m L[i][c0+m] L[k][c0+m]
    for (int i = c1 + ty; i < N; i += NT / 32) {
      float li[NB];
#pragma unroll
      for (int m = 0; m < NB; ++m) li[m] = S[i * LD + c0 + m];
      for (int k = c1 + tx; k <= i; k += 32) {
        float v = S[i * LD + k];
#pragma unroll
        for (int m = 0; m < NB; ++m) v = fmaf(-li[m], S[k * LD + c0 + m], v);
        S[i * LD + k] = v;
      }
    }
    __syncthreads();
  }
  // X = L'^{-1}: diagonal blocks first, row r of block kb by substitution
  // (x L_kk = e_r: x_r = 1 / L_rr, x_j = -(sum_{m=j+1}^{r} x_m L_mj) / L_jj)
  if (t < N) {
    const int kb = t / NB, r = t % NB, c0 = kb * NB;
    float x[NB];
#pragma unroll
    for (int j = NB - 1; j >= 0; --j) {
      float v = 0.f;
      if (j == r) v = rpiv[c0 + r];
      else if (j < r) {
        float acc = 0.f;
#pragma unroll
        for (int m = j + 1; m < NB; ++m)
          if (m <= r) acc = fmaf(x[m], S[(c0 + m) * LD + c0 + j], acc);
        v = -acc * rpiv[c0 + j];
      }
      x[j] = v;
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) X[(c0 + r) * LD + c0 + j] = x[j];
  }
  __syncthreads();
  // off-diagonal blocks, one block diagonal d = i - k at a time:
  // P_ik = sum_{m=k}^{i-1} L_im X_mk (into the upper triangle of X as scratch),
  // then X_ik = -X_ii P_ik
  for (int d = 1; d < NBLK; ++d) {
    const int nblk = NBLK - d;
    for (int e = t; e < nblk * NB * NB; e += NT) {
      const int k = e / (NB * NB), rc = e % (NB * NB), r = rc / NB, c = rc % NB;
      const int i = k + d;
      const int row = i * NB + r, col = k * NB + c;
      float acc = 0.f;
      for (int m = k * NB + c; m < i * NB; ++m)   // X_mk is zero above its diagonal
        acc = fmaf(S[row * LD + m], X[m * LD + col], acc);
      X[col * LD + row] = acc;                     // P^T, upper triangle
    }
    __syncthreads();
    for (int e = t; e < nblk * NB * NB; e += NT) {
      const int k = e / (NB * NB), rc = e % (NB * NB), r = rc / NB, c = rc % NB;
      const int i = k + d;
      const int row = i * NB + r, col = k * NB + c;
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < NB; ++q)
        if (q <= r) acc = fmaf(X[row * LD + i * NB + q], X[col * LD + i * NB + q], acc);
      X[row * LD + col] = -acc;
    }
    __syncthreads();
  }
  __syncthreads();
}

}  // namespace jolt
