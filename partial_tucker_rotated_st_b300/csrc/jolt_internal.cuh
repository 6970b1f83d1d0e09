// Internal declarations of libjolt: workspace layout, launch helpers and the
// kernel launchers each .cu file provides.  Host + device.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>
#include <climits>

#include "../../include/jolt.h"

namespace jolt {

// ------------------------------------------------------------------ status
// Device status word bits, OR-ed into the unit's status slot.
enum : int {
  ST_NOCONVERGE = 1,
  ST_NONFINITE = 2,
  ST_NOTPD = 4,     // Cholesky met a non-positive pivot (reported as NOCONVERGE)
  ST_TIMEOUT = 8,   // a bounded device wait gave up (reported as JOLT_ERR_CUDA)
};

extern unsigned long long g_launches;
extern void* g_sweep_ev[2];   // cudaEvent_t pair recorded around the fused sweep kernel, or null
extern void* g_factor_ev[5];  // cudaEvent_t recorded at the factor's stage boundaries, or null
inline void count_launch(int n = 1) { g_launches += (unsigned long long)n; }

#define JOLT_CUDA_TRY(expr)                                   \
  do {                                                        \
    cudaError_t e_ = (expr);                                  \
    if (e_ != cudaSuccess) return JOLT_ERR_CUDA;              \
  } while (0)

#define JOLT_LAUNCH_CHECK()                                   \
  do {                                                        \
    ::jolt::count_launch();                                   \
    cudaError_t e_ = cudaGetLastError();                      \
    if (e_ != cudaSuccess) return JOLT_ERR_CUDA;              \
  } while (0)

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ layout
// Resolved grid + byte offsets of every per-unit workspace section.
struct Layout {
  int H, T, D, dtype;
  int nT, nd, nb;
  int rT[JOLT_MAX_GRID];   // resolved (FULL -> T)
  int rd[JOLT_MAX_GRID];   // resolved (FULL -> D)
  int b[4];
  int nTt;        // truncated token ranks (all but a trailing FULL)
  int RT;         // largest truncated token rank (0 if none)
  int hasFullT;
  int ndt;        // truncated feature ranks
  int RD;         // largest truncated feature rank (0 if none)
  int hasFullD;
  int token_mode;
  int L;          // subspace-iteration block width (exact mode)
  int ell;        // sketch width RT + oversample (randomized mode)
  int power_iters;
  int nsplit, chunk;     // feature-Gram split over rows
  int ks;                // row chunks of the small Grams (divides T)
  int hs;                // head groups of the randomized Rayleigh-Ritz Gram (divides H)
  int tile_rows;         // sweep rows per CTA
  int ntiles;            // sweep CTAs per unit
  int ncand;
  int cost_model, align, block;
  // section offsets, bytes from the unit's base (unit u at ws + u * unit_bytes)
  size_t o_status, o_Sd, o_Sd64, o_Sdp, o_evd, o_Vd, o_Ud16, o_QUd, o_Y, o_Y16;
  size_t o_UT32, o_UT16, o_tokev, o_G32, o_G16, o_W, o_part, o_P;
  size_t o_Yt;           // Y relaid [T][RD*H] and its tf32 low part (token Gram)
  size_t o_Hs;           // diag(sigma) H_D as bf16 [D][D] (tensor-core sweep), or 0
  size_t o_Vs3;          // U_d in three bf16 parts [3 * 32][D] (tensor-core projection), or 0
  size_t o_Ub3;          // every rank's U_T in three bf16 parts [T][512] (tensor-core cores), or 0
  size_t o_cap;          // f64 [nd][RT]: sum over h, i < r_d of G(r_d)[h][j][i]^2, unrounded cores
  size_t o_Bx, o_Qs, o_C; // randomized token mode on the tensor cores: per-head B blocks
                          // [H][512][D] bf16, Q parts [T][512] bf16, C = X_h^T Q [H][D][160]
                          // fp32 (0 when that path is not taken)
  size_t unit_bytes;
  // Token-mode problems, one per (unit, feature rank), in a region after the
  // n unit regions of a call: truncated rank id of unit u is problem
  // u * ndt + id, the whole-feature rank of unit u is problem n * ndt + u;
  // problem p at ws + n * unit_bytes + p * prob_bytes.  Offsets from the
  // problem's base:
  int nprob;             // problems per unit (nd, or 0 without a token rank)
  size_t prob_bytes;
  size_t p_status, p_flag, p_ST, p_STs, p_Vs, p_V, p_Z, p_V2, p_Z2, p_Hm, p_Wm, p_Gram,
      p_Rinv, p_theta, p_UT, p_ev;
  size_t unit_total;     // workspace bytes per unit: unit_bytes + nprob * prob_bytes
};

jolt_status make_layout(const jolt_config* cfg, Layout* L);

// CholeskyQR (passes 1 or 2) of np T x 64 blocks (problem i at base + i *
// stride, offsets src / dst / o_status), one cluster launch; supported when
// every problem's cluster fits on the device at once
bool cholqr_fused_supported(int T, int Lw, int np);
jolt_status cholqr_fused(char* base, size_t stride, int np, size_t src, size_t dst,
                         size_t o_status, const int* skip, long long sk_s, int T, int passes,
                         float shift, cudaStream_t st, size_t vt = 0);

// FlashJoLT's range finder with its products over X on the tensor cores: the
// ranks rid[0..nr) of every unit in lockstep, problem (u, r) at pbase +
// (u * pmul + pidx0[r]) * prob_bytes; leaves Q in p_V and the Rayleigh-Ritz
// matrix, as L.hs partials of ell x ell, in p_Hm of every problem.
bool flash_tc_supported(const Layout& L);
jolt_status flash_tc_solve(const Layout& L, int U, const void* X, const float* sketch, char* ws,
                           char* pbase, int pmul, const int* pidx0, const int* rid, int nr,
                           cudaStream_t st);
// CholeskyQR2 (f64 Cholesky) of the T x ell blocks p_Z -> p_V of np problems
jolt_status cholqr2_set(const Layout& L, char* base, size_t stride, int np, cudaStream_t st);

// iteration caps of the eigensolvers (0 -> default)
void set_max_sweeps(int n);
void set_subspace_blocks(int n);

// ------------------------------------------------------------------ GEMM
// C[b1,b2] = alpha * sum_s A[b1,b2,s] (M x K) * B[b1,b2,s] (K x N) + beta * C
// with arbitrary element strides.  dtype codes: JOLT_F32, JOLT_BF16, JOLT_F16.
struct Opnd {
  const void* p;
  int dtype;
  long long s0, s1;        // strides of the two matrix indices (A: m,k; B: k,n)
  long long sseg, sb1, sb2;
};
struct GemmDesc {
  int M, N, K, nseg, nb1, nb2;
  Opnd A, B;
  float* C;
  long long cm, cn, cb1, cb2;
  float alpha, beta;
  const int* skip;         // optional per-b1 flag skip[b1 * skip_stride]; nonzero -> skipped
  long long skip_stride;
};
jolt_status launch_gemm(const GemmDesc& g, cudaStream_t st);

// ------------------------------------------------------------------ eigen
// Batched cyclic Jacobi (one CTA per symmetric n x n matrix, n <= 128).
// in: A[b] = sum over nparts partials at A + b*a_bstride + k*part_s, row
// stride lda.  out: evals[b][n] descending, evecs[b] with column i the i-th
// eigenvector (row stride ldv, first ncols_out columns written).
// abs_tol: rotations with |a_pq| below abs_tol * ||A||_F are not taken.
constexpr float JAC_ABS_EXACT = 1e-10f;
constexpr float JAC_ABS_RR = 1e-7f;
jolt_status launch_jacobi(const float* A, long long a_bstride, int lda, int n, int nparts,
                          long long part_s, int batch, float* evals, long long e_bstride,
                          float* evecs, long long v_bstride, int ldv, int ncols_out, int* status,
                          long long status_bstride, const int* skip, long long skip_stride,
                          float abs_tol, cudaStream_t st);
// Batched Cholesky G = R^T R of a sum of nparts partials (n x n, n <= 128;
// n <= 64 in f64), writes the upper factor R in f32.  The Gram is
// equilibrated to a unit diagonal first; `shift` is added to that diagonal.
jolt_status launch_chol(const float* G, long long g_bstride, int n, int nparts, long long part_s,
                        int batch, float* R, long long r_bstride, int* status,
                        long long status_bstride, const int* skip, long long skip_stride,
                        bool f64, float shift, cudaStream_t st);
// Eigenpairs of a batch of symmetric positive-definite n x n matrices (n in
// {32, 64, 128}) by Cholesky + one-sided Jacobi, same input (sum of nparts
// partials, f64 or fp32) and outputs as launch_jacobi.  done[b] is set to 1
// on success or when skip[b] is set, and left 0 where the matrix is not
// definite: launch_jacobi with skip = done then solves exactly those.
// Returns JOLT_ERR_INVALID for another n (nothing launched).
jolt_status launch_sym_eig(const void* G, bool f64_in, long long g_bstride, int lda, int n,
                           int nparts, long long part_s, int batch, float* evals,
                           long long e_bstride, float* evecs, long long v_bstride, int ldv,
                           int ncols_out, int* status, long long status_bstride, int* done,
                           long long done_bstride, const int* skip, long long skip_stride,
                           float abs_tol, cudaStream_t st);
// The same Cholesky (fp32, n in {32, 40, 48, 64}) writing R^{-1} instead of R.
jolt_status launch_chol_inv(const float* G, long long g_bstride, int n, int nparts,
                            long long part_s, int batch, float* Rinv, long long r_bstride,
                            int* status, long long status_bstride, const int* skip,
                            long long skip_stride, float shift, cudaStream_t st);
// Out[b] = In[b] R[b]^{-1} for a T x n block per batch entry, row-parallel.
jolt_status launch_trsm_rows(const float* In, float* Out, long long blk_bstride, const float* R,
                             long long r_bstride, int T, int n, int batch, const int* skip,
                             long long skip_stride, cudaStream_t st);

// ------------------------------------------------------------------ tensor cores
bool gram_tc_supported(const Layout& L);
// S_T of problem p = sum_h X_h X_h^T of unit p (T x T fp32 at pbase + p * pstride + p_ST).
jolt_status gram_tok_tc(const Layout& L, int n_units, const void* X, char* pbase, size_t pstride,
                        cudaStream_t st);
jolt_status gram_feat_tc(const Layout& L, int n_units, const void* X, char* ws, cudaStream_t st);
bool sv_tc_supported(const Layout& L);
// p_STs = tf32 low part of p_ST for np problems.
jolt_status split_tok_gram(const Layout& L, int np, char* pbase, size_t pstride, cudaStream_t st);
// (o_Z) = p_ST p_V for every problem whose p_flag is zero; vs_ready: p_Vs
// already holds p_V^T and its low part.
jolt_status sv_tc(const Layout& L, int np, char* pbase, size_t pstride, size_t o_Z,
                  cudaStream_t st, bool vs_ready = false);
bool ygram_tc_supported(const Layout& L);
// Y = X U_d[:, :RD] (bf16 X, D = 128, RD <= 32) on the tensor cores: U_d16,
// Y16, Yt and its tf32 low part (when the layout has Yt), and Y in fp32 when
// write_y.
bool proj_tc_supported(const Layout& L);
jolt_status proj_tc(const Layout& L, int n_units, const void* X, char* ws, bool write_y,
                    cudaStream_t st);
// The cores of every feature rank from X and U_T (bf16 X, D = 128, r_T <= 32):
// G16 of every rank and U_T16.
bool cores_tc_supported(const Layout& L);
jolt_status cores_tc(const Layout& L, int n_units, const void* X, char* ws, cudaStream_t st);
// Yt (unit region) = Y relaid [T][RD * H] and its tf32 low part.
jolt_status ytrans(const Layout& L, int n_units, char* ws, cudaStream_t st);
// p_ST of truncated problem p = u * ndt + id: the Gram of feature ranks
// [0, rd[id]) of unit u's Y.
jolt_status ygram_tc(const Layout& L, int n_units, const char* ws, char* pbase, size_t pstride,
                     cudaStream_t st);

// ------------------------------------------------------------------ steps
jolt_status factor_run(const Layout& L, int n_units, const void* X, const float* sketch,
                       char* ws, cudaStream_t st);
// Rotated factor rows for the sweep and the encoder: Q U_d and W = G (Q U_d)^T.
bool sweep_tc_supported(const Layout& L);
// The tensor-core sweep over all units: per-tile partial sums at part (unit
// stride part_us floats); *tiles_t_out = row tiles per head.
jolt_status sweep_tc_run(const Layout& L, int n_units, const void* X, char* ws, float* part,
                         long long part_us, int* tiles_t_out, cudaStream_t st);
jolt_status sweep_prep(const Layout& L, int n_units, const int8_t* signs, char* ws,
                       cudaStream_t st);
// part_override: where the per-tile partial sums go (n_units * ntiles *
// (ncand + 1) floats); nullptr = the workspace section.
jolt_status sweep_run(const Layout& L, int n_units, const void* X, const int8_t* signs,
                      char* ws, double* dist, int64_t* cost, cudaStream_t st,
                      float* part_override = nullptr);
jolt_status model_table_run(const Layout& L, int n_units, const char* ws, const double* eps2_host,
                            double* dist, cudaStream_t st);
jolt_status eps2_run(const float* rows, int n, int D, const int* bits_host, int nb, double* scratch,
                     double* eps2, cudaStream_t st);
jolt_status refine_run(int n_units, int n_cand, const double* dist, const int64_t* cost,
                       int64_t budget, int32_t* choice, int32_t* n_swaps, cudaStream_t st);
jolt_status uniform_run(int n_units, int n_cand, const double* dist, const int64_t* cost,
                        int64_t budget, const int32_t* cand_host, int n_list, int32_t* choice,
                        int32_t* status, cudaStream_t st);
jolt_status alloc_run(int n_units, int n_cand, const double* dist, const int64_t* cost,
                      int64_t budget, int align, int32_t* choice, double* lambda,
                      int32_t* status, cudaStream_t st);
jolt_status encode_run(const Layout& L, int n_units, const void* X, const int8_t* signs,
                       const char* ws, const int32_t* choice_host, char* blob,
                       size_t blob_stride, jolt_blob_desc* desc, cudaStream_t st);
jolt_status decode_run(int n_units, const jolt_blob_desc* desc, const char* blob,
                       size_t blob_stride, void* xhat, int out_dtype, cudaStream_t st);
bool decode_tc_supported(int D);
jolt_status decode_tc_status(int* out, cudaStream_t st);
jolt_status decode_tc_run(int n_units, const jolt_blob_desc* desc, const char* blob,
                          size_t blob_stride, void* xhat, int out_dtype, cudaStream_t st);
size_t admit_ws_unit_bytes(int H, int tau, int D);
jolt_status admit_run(int n_units, const jolt_blob_desc* desc_in, const char* blob_in,
                      size_t stride_in, const void* X_new, int x_dtype, int tau, int align,
                      char* ws, char* blob_out, size_t stride_out, jolt_blob_desc* desc_out,
                      cudaStream_t st);
size_t attend_ws_bytes(int n_groups, int H, int T, int D, int nq);
jolt_status attend_run(int n_groups, const jolt_blob_desc* desc, const char* blob,
                       size_t stride, const float* q, int nq, float scale, float* ws,
                       float* out, cudaStream_t st);

// ------------------------------------------------------------------ cost/blob
// Candidate (iT, id, ib) <-> flat index, iT-major.
static inline void cand_split(const Layout& L, int c, int* iT, int* id, int* ib) {
  *ib = c % L.nb;
  *id = (c / L.nb) % L.nd;
  *iT = c / (L.nb * L.nd);
}
int64_t cost_formula(int H, int T, int D, int rT, int rd, int b, int block, int align);
void blob_layout(int H, int T, int D, int rT, int rd, int b, int block, int align,
                 jolt_blob_desc* d);

// ------------------------------------------------------------------ device helpers
#ifdef __CUDACC__
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// fp32 -> nearest fp16 value (round to nearest even), returned as fp32.
__device__ __forceinline__ float round_f16(float x) { return __half2float(__float2half_rn(x)); }

// Round to nearest integer, ties to even, for |z| < 2^22, in two adds.
__device__ __forceinline__ float rint_magic(float z) {
  const float M = 12582912.0f;  // 1.5 * 2^23
  return __fsub_rn(__fadd_rn(z, M), M);
}

// Fast Walsh-Hadamard transform (Sylvester order) of a row spread over a warp:
// element i = lane * EPT + e.
template <int EPT>
__device__ __forceinline__ void fwht_row(float (&v)[EPT], int lane) {
#pragma unroll
  for (int h = 1; h < EPT; h <<= 1)
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if (!(e & h)) {
        const float a = v[e], b = v[e + h];
        v[e] = a + b;
        v[e + h] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = (lane & m) ? (o - v[e]) : (v[e] + o);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
#endif

}  // namespace jolt
