/*
 * libjolt -- KV-cache encode and decode by partial Tucker + rotated residual
 * + Lagrangian allocation (JoLT), for NVIDIA B300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [P1] "Joint Tucker-rank and residual-bit KV allocator": Formulas,
 *        Mathematical statement, Implementation notes.
 *   [P4] "Rotated Tucker residual for outlier-resistant KV quantization":
 *        Mathematical statement, Key formulas, Implementation notes.
 *   [P5] "Technical Summary: A JOLT for the KV Cache": Methodology 1-4.
 *
 * Vocabulary.  A *unit* is one group tensor X[H][T][D] of one cache type
 * (K or V) of one layer group: H = layers-in-group x KV heads (kept whole),
 * T tokens, D features (a power of two, 32..128).  A *candidate* is
 * z = (r_T, r_d, b): token rank, feature rank, residual bits.  Candidates are
 * numbered flat, iT-major, then id, then ib, over the grid of the config.
 *
 * Conventions shared by every call.
 *   - All tensor arguments are DEVICE pointers unless the name ends in
 *     `_host`.  The caller owns every buffer; the library never allocates
 *     device memory.  Batches of units are contiguous: X is
 *     [n_units][H][T][D], signs is [n_units][D], and so on.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and returns after its launches are queued.  Argument
 *     errors are detected on the host before anything is launched and are
 *     returned as JOLT_ERR_INVALID / JOLT_ERR_WORKSPACE.  Errors found on the
 *     device (no convergence, non-finite input) are recorded in a status word
 *     inside the workspace; jolt_read_status() synchronises and reports them.
 *     No kernel traps or asserts.
 *   - Random draws of the method (the rotation's sign vector and the
 *     FlashJoLT Gaussian sketch) are inputs, never generated inside.
 *   - One GPU per process: kernels that need more than 48 KB of dynamic
 *     shared memory have their limit raised (cudaFuncSetAttribute) once per
 *     process, on the device current at the first call, and the attribute
 *     holds for that device only.  Drive the library from one device per
 *     process (the usual one-rank-per-GPU launch); a call on a second device
 *     of the same process may fail with JOLT_ERR_CUDA.
 */
#ifndef JOLT_H
#define JOLT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JOLT_OK = 0,
  JOLT_ERR_INVALID = 1,     /* bad argument (shape, grid, pointer, dtype) */
  JOLT_ERR_INFEASIBLE = 2,  /* budget below the cheapest allocation */
  JOLT_ERR_NONFINITE = 3,   /* NaN/Inf met in X or in a scale */
  JOLT_ERR_NOCONVERGE = 4,  /* an eigensolver hit its iteration cap */
  JOLT_ERR_WORKSPACE = 5,   /* workspace missing or too small */
  JOLT_ERR_CUDA = 6,        /* a CUDA runtime call failed */
  JOLT_ERR_TOO_LARGE = 7    /* batch beyond the no-allocation entry point's static scratch */
} jolt_status;

typedef enum { JOLT_F32 = 0, JOLT_BF16 = 1, JOLT_F16 = 2 } jolt_dtype;

typedef enum {
  JOLT_TOKEN_EXACT = 0,      /* token-mode eigenvectors solved to convergence */
  JOLT_TOKEN_RANDOMIZED = 1  /* FlashJoLT randomized range finder [P5 Methodology 4] */
} jolt_token_mode;

typedef enum {
  JOLT_COST_FORMULA = 0,     /* the printed cost expression [P1 Formulas] */
  JOLT_COST_SERIALIZED = 1   /* bytes of the serialized blob [P1 Implementation notes] */
} jolt_cost_model;

/* Grid sentinel: keep a mode untruncated (r_T = T or r_d = D). */
#define JOLT_FULL (-1)
#define JOLT_MAX_GRID 8
#define JOLT_MAX_CAND (JOLT_MAX_GRID * JOLT_MAX_GRID * 4)   /* largest candidate grid */
#define JOLT_HEADER_BYTES 256
#define JOLT_ATTN_MAX_Q 8          /* queries per head of one jolt_attend call */
#define JOLT_ATTN_MAX_RANK 128     /* longest low-rank token row jolt_attend accepts */

/*
 * Shape, candidate grid and options of one batch of units.
 *   rT[], rd[]   ascending; truncated ranks first, JOLT_FULL (at most once,
 *                last) for the untruncated mode; truncated r_T <= 64,
 *                truncated r_d <= 64 and < D, r_T < T.
 *   b[]          ascending subset of {0, 2, 4, 8} [P1 Implementation notes].
 *   quant_block  values per quantization block; must equal D (one block is
 *                one (h, t) row of the rotated residual).
 *   oversample, power_iters   FlashJoLT sketch width p and power steps q.
 *   align        section alignment of the blob and of the cost model.
 */
typedef struct {
  int H, T, D;
  jolt_dtype dtype;                 /* X element type: JOLT_F32 or JOLT_BF16 */
  int n_rT, rT[JOLT_MAX_GRID];
  int n_rd, rd[JOLT_MAX_GRID];
  int n_b, b[4];
  int quant_block;
  jolt_token_mode token_mode;
  int oversample;
  int power_iters;
  jolt_cost_model cost_model;
  int align;
} jolt_config;

/* Host-side description of one serialized unit (the blob's header fields). */
typedef struct {
  int H, T, D, rT, rd, b, block;
  int flags;                        /* bit 0: U_T omitted (r_T = T); bit 1: U_d omitted (r_d = D) */
  uint64_t off_UT, off_Ud, off_G, off_scale, off_codes, bytes;
} jolt_blob_desc;

/* Number of candidates n_rT * n_rd * n_b of a config (0 if invalid). */
int jolt_num_candidates(const jolt_config* cfg);

/* Bytes of workspace one unit needs; a batch of n units needs n times this,
 * contiguous, 256-byte aligned.  0 if the config is invalid. */
size_t jolt_workspace_size(const jolt_config* cfg);

/*
 * Partial Tucker factors of every unit, by ST-HOSVD over the feature mode and
 * then the token mode, head axis kept [P1 Mathematical statement,
 * Implementation notes; P5 Methodology 1]:
 *   S_d = sum_{h,t} x_{h,t} x_{h,t}^T, U_d = its leading eigenvectors;
 *   for every r_d of the grid: Y = X x_3 U_d(r_d)^T, S_T = Y_(T) Y_(T)^T,
 *   U_T(r_d) = its leading eigenvectors (exact mode) or the FlashJoLT
 *   randomized range finder's (randomized mode, [P5 Methodology 4]);
 *   cores G = Y x_2 U_T^T.  Factors and cores are rounded to fp16, the
 *   storage type, and kept in the workspace for the calls below.
 *   X       [n_units][H][T][D], cfg->dtype
 *   sketch  [n_units][H][D][max truncated r_T + oversample] fp32 Gaussian
 *           test matrix (randomized mode only, else may be NULL); the sketch
 *           for feature rank r_d is the leading r_d rows of each head's slab.
 *   ws      n_units * jolt_workspace_size(cfg) bytes.
 * Device errors: JOLT_ERR_NOCONVERGE (eigensolver cap) in the status word.
 */
jolt_status jolt_factor_group(const jolt_config* cfg, int n_units, const void* X,
                              const float* sketch, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * Distortion and byte cost of every candidate of every unit [P1 Formulas]:
 *   dist[u][iT][id][ib] = ||X - X^||_F^2 / ||X||_F^2 (0 for an all-zero X),
 *   X^ = X~ + Q^T Q_b(Q R), R = X - X~, Q = H_D diag(sigma) / sqrt(D)
 *   [P4 Key formulas, Implementation notes], Q_b the symmetric per-block
 *   absmax quantizer with fp16 block scale, b = 0 meaning X^ = X~.
 *   cost[u][iT][id][ib] in bytes, per cfg->cost_model.
 *   signs  [n_units][D] int8, each +1 or -1 (diag(sigma) of the rotation).
 *   dist   [n_units][n_cand] float64; cost [n_units][n_cand] int64.
 * Requires jolt_factor_group on the same ws first.
 * Device errors: JOLT_ERR_NONFINITE in the status word.
 */
jolt_status jolt_sweep_candidates(const jolt_config* cfg, int n_units, const void* X,
                                  const int8_t* signs, void* ws, size_t ws_bytes,
                                  double* dist, int64_t* cost, void* stream);

/*
 * One candidate per unit under a global byte budget by bisection on the
 * Lagrange multiplier lambda [P1 Formulas, Mathematical statement,
 * Implementation notes; P5 Methodology 3]: z(lambda) = argmin_z
 * dist + lambda * cost per unit (product rounded before the sum; ties to the
 * smaller cost, then the lower index).  If z(0) fits, it is returned with
 * lambda = 0.  If the cheapest allocation does not fit, it is returned with
 * status JOLT_ERR_INFEASIBLE.  Otherwise hi = 1 is doubled until z(hi) fits,
 * then (lo, hi) is bisected (at most 200 steps) until the total cost lies
 * within one `align` block below the budget or the interval is at the
 * resolution of a double; z(hi) is returned.
 *   dist [n_units][n_cand] f64, cost [n_units][n_cand] int64 (device).
 *   choice [n_units] int32, lambda [1] f64, status [1] int32 (device,
 *   JOLT_OK or JOLT_ERR_INFEASIBLE).
 * Runs in one thread block.
 */
jolt_status jolt_allocate(int n_units, int n_cand, const double* dist, const int64_t* cost,
                          int64_t budget, int align, int32_t* choice, double* lambda,
                          int32_t* status, void* stream);

/*
 * Greedy improvement of a feasible allocation, run after jolt_allocate
 * [P1 Implementation notes: after the bisection, optionally improve the
 * result by swapping candidates with the best distortion reduction per added
 * byte].  A swap replaces unit u's candidate z by c when it adds
 * dc = cost[u][c] - cost[u][z] bytes with 0 < dc <= the slack
 * (budget - total cost) and lowers the unit's distortion by
 * dd = dist[u][z] - dist[u][c] > 0; its rate is dd / dc (f64, correctly
 * rounded).  Each round applies the swap of highest rate (ties: smaller dc,
 * then lower unit, then lower candidate index) until none fits.
 *   dist, cost as for jolt_allocate; choice [n_units] int32 (device), read
 *   and rewritten in place (it must fit the budget); n_swaps [1] int32
 *   (device, may be NULL) receives the number of swaps applied.
 * Runs in one thread block.
 */
jolt_status jolt_refine(int n_units, int n_cand, const double* dist, const int64_t* cost,
                        int64_t budget, int32_t* choice, int32_t* n_swaps, void* stream);

/*
 * Uniform baseline allocation [P1 Verification, Stage 1: the comparison
 * against every group on the same candidate, fixed at 4 bits]: every unit
 * takes the same candidate, chosen among `cand_host` (n_list flat indices,
 * host memory, 1 <= n_list <= JOLT_MAX_CAND) as the one of least total
 * distortion (the units' dists summed in unit order, f64) whose total cost
 * fits the budget, ties to the lower index.  If none fits, every unit takes
 * the list's candidate of least total cost (ties: lower index) and *status
 * is JOLT_ERR_INFEASIBLE.  Fixed-bit: the list of every rank pair at one bit
 * width; fixed-rank: every bit width at one rank pair.
 *   choice [n_units] int32, status [1] int32 (device).
 */
jolt_status jolt_allocate_uniform(int n_units, int n_cand, const double* dist,
                                  const int64_t* cost, int64_t budget, const int32_t* cand_host,
                                  int n_list, int32_t* choice, int32_t* status, void* stream);

/*
 * Measurement hook: when both are non-NULL, the two CUDA events (cudaEvent_t
 * created with timing enabled, owned by the caller) are recorded on the call's
 * stream immediately before and after the fused sweep kernel of every later
 * jolt_sweep_candidates / jolt_sweep_candidates_noalloc call, so that the
 * kernel's own duration can be read with cudaEventElapsedTime.  NULL, NULL
 * turns it off.  Process-wide setting, not thread-safe; JOLT_ERR_INVALID if
 * only one is NULL.
 */
jolt_status jolt_set_sweep_events(void* start, void* stop);

/*
 * Measurement hook for the factor step: when `events` is non-NULL it points
 * to five CUDA events (cudaEvent_t created with timing enabled, owned by the
 * caller) that every later jolt_factor_group call records at its stage
 * boundaries:
 *   [0] the start of the call (caller's stream);
 *   [1] the feature stage done: feature Gram, eigen-solve, projection Y and
 *       the truncated ranks' token Grams (the library's side stream);
 *   [2] the whole-feature token-mode solve done (caller's stream; recorded
 *       as [0] when there is no such solve);
 *   [3] every token-mode solve done, after the two streams joined;
 *   [4] the cores and fp16 factors done (the end of the call's work).
 * The critical path is max([1], [2]) - [0], then [3], then [4].  NULL turns it
 * off.  Process-wide setting, not thread-safe.
 */
jolt_status jolt_set_factor_events(void* const* events);

/*
 * Iteration caps of the factor step's eigensolvers, for exercising the
 * non-convergence path: `max_sweeps` bounds the sweeps of every Jacobi solve
 * (feature Gram, token Gram, Rayleigh-Ritz blocks; default 40) and
 * `max_subspace_blocks` the blocks of the exact token mode's subspace
 * iteration (default 25).  0 restores a default; negative values return
 * JOLT_ERR_INVALID and change nothing.  A solve that reaches its cap sets the
 * unit's status, and jolt_read_status then returns JOLT_ERR_NOCONVERGE.
 * Process-wide setting read at launch time, not thread-safe.
 */
jolt_status jolt_set_solver_limits(int max_sweeps, int max_subspace_blocks);

/*
 * Modeled-error distortion table, an alternative to jolt_sweep_candidates
 * that needs no pass over X ["A JoLT for the KV cache" verdict page, referee
 * report on Section 4, Eq. (2): e ~ eps^2(b) tau; P5 Methodology 4: tail-mass
 * accounting].  From the spectra of jolt_factor_group on the same ws:
 *   tau(r_T, r_d) = sum_{i >= r_d} lambda_i              (r_T = T)
 *                 = ||X||^2 - sum_{j < r_T} mu_j(r_d)    (r_T < T),
 * lambda the feature eigenvalues (||X||^2 = their sum), mu the token
 * eigenvalues of feature rank r_d; dist[u][cand] = eps2[ib] tau / ||X||^2
 * (eps2 of b = 0 taken as 1; 0 for an all-zero unit).
 *   eps2_host [cfg->n_b] f64 (host), e.g. from jolt_calibrate_eps2;
 *   dist [n_units][n_cand] f64 (device).
 */
jolt_status jolt_model_candidates(const jolt_config* cfg, int n_units, const void* ws,
                                  size_t ws_bytes, const double* eps2_host, double* dist,
                                  void* stream);

/*
 * Calibration of eps^2(b) on a Gaussian round trip [same passage]: rows
 * (device, n_rows x D fp32, D in {32, 64, 128}) are the caller's standard
 * normal draws; each row goes through the per-row absmax quantizer with fp16
 * scale of the codec, and eps2[ib] = sum ||y - Q_b(y)||^2 / sum ||y||^2
 * (1 for b = 0).  bits_host [n_b] (host, each 0, 2, 4 or 8); scratch [8] f64
 * and eps2 [n_b] f64 (device).
 */
jolt_status jolt_calibrate_eps2(const float* rows, int n_rows, int D, const int32_t* bits_host,
                                int n_b, double* scratch, double* eps2, void* stream);

/* Size in bytes of the serialized blob of candidate `cand` (flat index). */
size_t jolt_blob_bytes(const jolt_config* cfg, int cand);

/*
 * Serialize each unit's chosen candidate [P4 Implementation notes: store the
 * block scale and the integer codes]: a 256-byte header, then U_T (fp16
 * T x r_T, omitted when r_T = T), U_d (fp16 D x r_d, omitted when r_d = D),
 * G (fp16 H x r_T x r_d), scales (fp16, one per row) and codes (b-bit
 * offset-binary q + 2^(b-1), packed LSB-first), sections aligned to
 * cfg->align.
 *   choice_host [n_units] flat candidate indices (host memory).
 *   blob        [n_units] slots of blob_stride bytes each (device).
 *   desc_out    [n_units] filled on the host.
 */
jolt_status jolt_encode(const jolt_config* cfg, int n_units, const void* X,
                        const int8_t* signs, const void* ws, size_t ws_bytes,
                        const int32_t* choice_host, void* blob, size_t blob_stride,
                        jolt_blob_desc* desc_out, void* stream);

/*
 * Rebuild X^ = G x_2 U_T x_3 U_d + Q^T (s * codes) of each unit from its blob
 * [P1 Formulas; P4 Implementation notes: multiply codes by s, apply the
 * inverse transform, add X~].  The kernel reads each blob's header on the
 * device; desc gives the host the shapes for validation.
 *   xhat  [n_units][H][T][D] in out_dtype (JOLT_F32 or JOLT_BF16, RNE).
 * D = 128 with 16-byte aligned xhat, blob, stride and code / core sections
 * (as jolt_encode lays them out) runs on the tensor cores; other shapes run
 * the same arithmetic on the SIMT decoder.  A tensor-core tile whose
 * bounded wait gave up is written as NaN (no kernel traps) and is reported
 * by jolt_decode_status.
 */
jolt_status jolt_decode(int n_units, const jolt_blob_desc* desc, const void* blob,
                        size_t blob_stride, void* xhat, jolt_dtype out_dtype, void* stream);

/*
 * The decoder's device-side status since the last call: synchronises `stream`,
 * then returns JOLT_ERR_CUDA when a bounded wait of a tensor-core decode gave
 * up (those tiles were written as NaN), else JOLT_OK, and clears it.  The
 * status is one word per device, shared by every decode on that device.
 */
jolt_status jolt_decode_status(void* stream);

/*
 * Attention of each group's queries over its compressed K and V, with the
 * rebuild fused in [P1 Implementation notes: rebuild the low-rank part and
 * the residual right before attention, preferably in a fused kernel; P5
 * Results (deployment cost): a fused reconstruction-and-attention kernel]:
 *   O[g][h][i] = sum_t p_t V^[g][h][t],
 *   p = softmax_t(scale * q[g][h][i] . K^[g][h][t]),
 * with K^, V^ the decodes of blobs 2g and 2g+1 (jolt_decode's X^).  Neither
 * is written to memory: the rotation moves onto the queries and the
 * output, the low-rank part is scored through U_T / G rows, and the codes
 * are read once per call.
 *   n_groups     groups; blob slot 2g holds K, slot 2g+1 holds V of group g
 *                (the unit order jolt_encode writes for K/V pairs)
 *   desc         [2 * n_groups] blob descriptions (host); all with the same
 *                H, T, D (D in {32, 64, 128}), block = D, truncated ranks
 *                <= 64, sections aligned as jolt_encode lays them out
 *   blob         [2 * n_groups] slots of blob_stride bytes (device)
 *   q            [n_groups][H][nq][D] fp32 queries (device), 1 <= nq <=
 *                JOLT_ATTN_MAX_Q (e.g. the query heads that share one KV head)
 *   scale        softmax scale (1/sqrt(D) for standard attention)
 *   ws, ws_bytes scratch of at least jolt_attend_workspace_size() bytes
 *                (device; per-chunk partial results, no clearing needed)
 *   out          [n_groups][H][nq][D] fp32 (device)
 * Returns JOLT_ERR_INVALID for a bad shape, rank, alignment or pointer and
 * JOLT_ERR_WORKSPACE for a short ws, before any launch.
 */
size_t jolt_attend_workspace_size(int n_groups, int H, int T, int D, int nq);
jolt_status jolt_attend(int n_groups, const jolt_blob_desc* desc, const void* blob,
                        size_t blob_stride, const float* q, int nq, float scale, void* ws,
                        size_t ws_bytes, float* out, void* stream);

/*
 * Admission of a block of tau new tokens into encoded units [P4
 * Implementation notes: the Tucker factors are kept, X~ is rebuilt for each
 * incoming token block and only R = X - X~ is coded; P1 Implementation
 * notes: at KV-cache admission time].  Each unit keeps its candidate
 * (r_T, r_d, b), factors and signs:
 *   Y = X_new U_d (X_new itself when r_d = D);
 *   r_T < T: U_T gains the fp16 rows u_t solving (sum_h G_h G_h^T) u_t =
 *            sum_h G_h Y[h][t]^T (the fold-in of the token under the fixed
 *            core; Cholesky pivots at most 2^-40 max diag dropped, that
 *            coordinate 0);
 *   r_T = T: G gains the rows fp16(Y), and r_T becomes T + tau;
 *   the residual of the new tokens is rotated and quantized as in
 *   jolt_encode.  Every section of the old tokens is copied bit for bit.
 *   desc_in, blob_in, stride_in   the units' blobs (as jolt_decode takes them)
 *   X_new       [n_units][H][tau][D] in x_dtype (JOLT_F32 or JOLT_BF16), device
 *   align       section alignment of the new blobs (cfg->align; power of two
 *               >= 16)
 *   ws          jolt_admit_workspace_size(n_units, H, tau, D) bytes, device
 *   blob_out    [n_units] slots of stride_out bytes (device, not overlapping
 *               blob_in); desc_out [n_units] filled on the host
 * Returns JOLT_ERR_INVALID / JOLT_ERR_WORKSPACE before any launch.
 */
size_t jolt_admit_workspace_size(int n_units, int H, int tau, int D);
jolt_status jolt_admit(int n_units, const jolt_blob_desc* desc_in, const void* blob_in,
                       size_t stride_in, const void* X_new, jolt_dtype x_dtype, int tau,
                       int align, void* ws, size_t ws_bytes, void* blob_out, size_t stride_out,
                       jolt_blob_desc* desc_out, void* stream);

/*
 * The same sweep as jolt_sweep_candidates, for callers that cannot allocate
 * device memory (code that runs where cudaMalloc is not allowed, or whose
 * memory belongs to an allocator it may not call at this point).  The pages
 * have no counterpart: this is a deployment variant of the call above, with
 * the same arguments and the same results.
 *   - Scratch: the per-tile partial sums go to one static device array of
 *     jolt_noalloc_scratch_bytes() bytes (16 MiB) that the library holds on
 *     every GPU it is loaded on until the process exits; nothing is
 *     allocated.  A batch needs n_units * ceil(T / (8192 / D)) * H *
 *     (n_cand + 1) * 4 bytes of it; a larger batch returns
 *     JOLT_ERR_TOO_LARGE before any launch (split it into smaller batches).
 *     The bound counts the SIMT kernel's 8192 / D-row tiles for every path;
 *     the tensor-core sweep (bf16, D = 128) writes 128-row tiles at the same
 *     stride, so there the bound is conservative by a factor of two.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - One device per process: the kernels' shared-memory limits are raised
 *     once per process (see the note at the top of this file), so although
 *     the array address is kept per device, use this call from one GPU per
 *     process.
 *   - Sharing: every call on a device uses the same array.  Calls that
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it; order them on one stream or with events.  Every entry a call
 *     reads is written by that call first, so nothing needs clearing.
 *   - ws must hold the factors of jolt_factor_group as for the call above.
 */
jolt_status jolt_sweep_candidates_noalloc(const jolt_config* cfg, int n_units, const void* X,
                                          const int8_t* signs, void* ws, size_t ws_bytes,
                                          double* dist, int64_t* cost, void* stream);

/* Size of the static scratch array of jolt_sweep_candidates_noalloc. */
size_t jolt_noalloc_scratch_bytes(void);

/* Synchronise `stream` and return the worst device status recorded in the
 * workspace of the n_units units (then clear it). */
jolt_status jolt_read_status(const jolt_config* cfg, int n_units, void* ws, void* stream);

/* Human-readable name of a status code. */
const char* jolt_status_string(jolt_status s);

/* Number of kernel launches the library has queued since load (counter for
 * benchmarks). */
uint64_t jolt_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* JOLT_H */
