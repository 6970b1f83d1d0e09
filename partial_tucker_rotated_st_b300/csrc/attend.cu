// Attention of queries over the compressed K and V of each group, without
// rebuilding K^ or V^ in memory.
//
// [Joint Tucker-rank and residual-bit KV allocator, Implementation notes: the
//  low-rank part and the residual are rebuilt right before attention, ideally
//  in one fused kernel.  Technical Summary: A JOLT for the KV Cache, Results
//  (deployment cost): the fused reconstruction-and-attention kernel.]
//
// The rebuild is fused into the attention algebraically.  For head h, query
// v and token t of a blob (r_T, r_d, b, signs sigma, scale s_t, codes u_t):
//   v . X^[t] = c . R[t] + s_t * (v~ . (u_t - 2^(b-1)))
// with
//   v~  = H_D diag(sigma) v / sqrt(D)            (the rotation moved onto v)
//   R[t] = U_T[t]            (r_T < T),   c = G[h] (U_d^T v)   (or G[h] v)
//   R[t] = G[h][t]           (r_T = T),   c = U_d^T v          (or v)
// so a score costs one r_T- (or r_d-) long dot and one D-long dot with the
// integer codes.  The value side accumulates, per query,
//   cv = sum_t p_t R_V[t],     z = sum_t p_t s_t (u_t - 2^(b-1))
// and maps back once at the end:
//   O = (back-projection of cv + sigma_V o H_D z / sqrt(D)) / sum_t p_t,
// the back-projection being U_d G[h]^T cv (r_T < T) or U_d cv (r_T = T), with
// an identity U_d when r_d = D.
//
// Three kernels.  attend_prep computes c and v~ once per (head, group).
// attend_chunk takes ATT_CHUNK tokens per CTA: it first copies the chunk's
// codes and low-rank rows of both blobs and the query coefficients into
// shared memory with cp.async, so that the whole working set of the CTA is
// in flight at once; then phase 1 scores the chunk's tokens (one thread per
// token), phase 2 turns them into probabilities against the chunk's max,
// phase 3 accumulates cv and z (a warp per 32 tokens, lanes over the feature
// / rank index), and the CTA writes its max, sum, cv and z.  attend_merge
// combines the chunks of each (head, group, query) (flash-decoding) and
// applies the back-projection and the inverse rotation.
#include <algorithm>

#include "jolt_internal.cuh"

namespace jolt {

namespace {

constexpr int ATT_CHUNK = 128;     // tokens per CTA = threads per CTA
constexpr int ATT_WARPS = ATT_CHUNK / 32;
constexpr int ATT_MAX_G = 16;      // groups per launch
constexpr int KM = JOLT_ATTN_MAX_RANK;
constexpr int ATT_STAGE_RANK = 64; // low-rank rows up to this length go through shared memory

struct AttUnit {
  int rT, rd, b, pad;
  unsigned long long off_UT, off_Ud, off_G, off_scale, off_codes;
};

struct AttArgs {
  int H, T, nq, nch;
  float scale;
  const char* blob;
  unsigned long long stride;
  const float* q;       // [groups][H][nq][D]
  float* qc;            // [groups][H][KM + D][NQ]: c, then v~
  float* part;          // [groups][H][nch][rec]
  float* out;           // [groups][H][nq][D]
  int g0;               // first group of this launch
  // attend_chunk's data region (bytes, 16-aligned offsets): K codes, K rows,
  // V codes, V rows; `data` >= their end and >= the phase-3 partial sums
  int o_kr, o_vc, o_vr, data;
  AttUnit k[ATT_MAX_G], v[ATT_MAX_G];
};

__host__ __device__ constexpr int nq_pad(int nq) { return nq <= 1 ? 1 : nq <= 2 ? 2 : nq <= 4 ? 4 : 8; }

// b-bit code u as the float u - 2^(b-1), exactly: 2^23 + u has u in its low
// mantissa bits.
__device__ __forceinline__ float code_f(unsigned u, float bias) {
  return __uint_as_float(0x4B000000u | u) - bias;
}

__host__ __device__ __forceinline__ size_t rec_floats(int nq, int D) {
  return (size_t)nq * (2 + D + KM);
}

// Asynchronous copy of nbytes (even) from global to shared memory by nthr
// threads, in 16-, 8- or 4-byte pieces as the source alignment allows (the
// last piece reads only the bytes that remain); 2-byte aligned sources are
// copied with plain loads.
__device__ __forceinline__ void copy_async(void* dst, const void* src, int nbytes, int tid,
                                           int nthr) {
  char* d = (char*)dst;
  const char* s = (const char*)src;
  const uintptr_t al = (uintptr_t)src;
  if ((al & 15) == 0) {
    for (int p = tid; p * 16 < nbytes; p += nthr) {
      const int rem = nbytes - p * 16;
      const uint32_t sd = (uint32_t)__cvta_generic_to_shared(d + p * 16);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sd), "l"(s + p * 16),
                   "r"(rem < 16 ? rem : 16) : "memory");
    }
  } else if ((al & 7) == 0) {
    for (int p = tid; p * 8 < nbytes; p += nthr) {
      const int rem = nbytes - p * 8;
      const uint32_t sd = (uint32_t)__cvta_generic_to_shared(d + p * 8);
      asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(sd), "l"(s + p * 8),
                   "r"(rem < 8 ? rem : 8) : "memory");
    }
  } else if ((al & 3) == 0) {
    for (int p = tid; p * 4 < nbytes; p += nthr) {
      const int rem = nbytes - p * 4;
      const uint32_t sd = (uint32_t)__cvta_generic_to_shared(d + p * 4);
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(sd), "l"(s + p * 4),
                   "r"(rem < 4 ? rem : 4) : "memory");
    }
  } else {
    for (int p = tid; p * 2 < nbytes; p += nthr)
      reinterpret_cast<__half*>(d)[p] = reinterpret_cast<const __half*>(s)[p];
  }
}

// NQ consecutive floats of shared memory (16-byte aligned for NQ >= 4) into
// registers with vector loads.
template <int NQ>
__device__ __forceinline__ void load_q(const float* p, float (&o)[NQ]) {
  if constexpr (NQ >= 4) {
#pragma unroll
    for (int c = 0; c < NQ / 4; ++c) {
      const float4 v = reinterpret_cast<const float4*>(p)[c];
      o[4 * c] = v.x; o[4 * c + 1] = v.y; o[4 * c + 2] = v.z; o[4 * c + 3] = v.w;
    }
  } else if constexpr (NQ == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    o[0] = v.x; o[1] = v.y;
  } else {
    o[0] = p[0];
  }
}

// One token's residual dot products sum_d v~_i[d] (u_d - 2^(b-1)) for every
// query, the codes row read as 32-bit words (B bits per code), all loads
// issued before the arithmetic.
template <int D, int NQ, int B>
__device__ __forceinline__ void res_dots(const uint32_t* __restrict__ row,
                                         const float* __restrict__ vt, float (&r)[NQ]) {
  constexpr int PER = 32 / B;              // codes per word
  constexpr int NW = D * B / 32;           // words per row
  constexpr unsigned MASK = (1u << B) - 1u;
  const float bias = 8388608.0f + (float)(1 << (B - 1));
  uint32_t wd[NW];
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int w4 = 0; w4 < NW / 4; ++w4) {
      const uint4 v = reinterpret_cast<const uint4*>(row)[w4];
      wd[4 * w4] = v.x; wd[4 * w4 + 1] = v.y; wd[4 * w4 + 2] = v.z; wd[4 * w4 + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) wd[w] = row[w];
  }
#pragma unroll
  for (int i = 0; i < NQ; ++i) r[i] = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w)
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int d = w * PER + j;
      const float f = code_f((wd[w] >> (j * B)) & MASK, bias);
      float v[NQ];
      load_q<NQ>(vt + d * NQ, v);
#pragma unroll
      for (int i = 0; i < NQ; ++i) r[i] = fmaf(v[i], f, r[i]);
    }
}

// z[i][e] += ps[i] * (u - 2^(b-1)) for this lane's EPT codes of one row.
template <int EPT, int NQ, int B>
__device__ __forceinline__ void res_accum(const uint32_t* __restrict__ row, int lane,
                                          const float (&ps)[NQ], float (&z)[NQ][EPT]) {
  constexpr unsigned MASK = (1u << B) - 1u;
  const float bias = 8388608.0f + (float)(1 << (B - 1));
  // EPT * B divides 32, so a lane's bits never straddle a word
  const int bit = lane * EPT * B;
  const uint32_t wd = row[bit >> 5] >> (bit & 31);
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const float f = code_f((wd >> (e * B)) & MASK, bias);
#pragma unroll
    for (int i = 0; i < NQ; ++i) z[i][e] = fmaf(ps[i], f, z[i][e]);
  }
}

// n halves from global to shared memory, every load independent.
__device__ __forceinline__ void stage_halves(__half* dst, const __half* __restrict__ src, int n,
                                             int tid, int nthr) {
#pragma unroll 8
  for (int i = tid; i < n; i += nthr) dst[i] = src[i];
}

__device__ __forceinline__ float sign_of(const unsigned char* sb, int d) {
  return ((sb[d >> 3] >> (d & 7)) & 1) ? -1.f : 1.f;
}

// Query coefficients of the K blob for one (head, group): c (score weights
// of the low-rank row R[t]) and v~ (the rotated query).
template <int EPT, int NQ>
__global__ void __launch_bounds__(128) attend_prep_kernel(AttArgs a) {
  constexpr int D = 32 * EPT;
  __shared__ float vq[NQ][D], wq[NQ][KM];
  __shared__ __half st_Ud[D * 64], st_G[64 * (KM > D ? KM : D)];
  // attend_chunk may start now: it stages its own data first and waits for
  // this grid before it reads c and v~
  asm volatile("griddepcontrol.launch_dependents;");
  const int h = blockIdx.x, gl = blockIdx.y, g = a.g0 + gl;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int T = a.T, H = a.H, nq = a.nq;
  const AttUnit ku = a.k[gl];
  const char* kb = a.blob + (unsigned long long)(2 * g) * a.stride;
  const bool kfT = (ku.rT == T), kfD = (ku.rd == D);
  const int Kk = kfT ? ku.rd : ku.rT;
  float* qc = a.qc + ((size_t)g * H + h) * (KM + D) * NQ;
  const float* qg = a.q + ((size_t)g * H + h) * nq * D;
  for (int x = tid; x < NQ * D; x += 128) vq[x / D][x % D] = (x / D) < nq ? qg[x] : 0.f;
  if (!kfD) stage_halves(st_Ud, (const __half*)(kb + ku.off_Ud), D * ku.rd, tid, 128);
  if (!kfT)
    stage_halves(st_G, (const __half*)(kb + ku.off_G) + (size_t)h * ku.rT * ku.rd,
                 ku.rT * ku.rd, tid, 128);
  __syncthreads();
  // w = U_d^T v (or v)
  for (int x = tid; x < NQ * ku.rd; x += 128) {
    const int i = x / ku.rd, j = x % ku.rd;
    float s = 0.f;
    if (kfD) {
      s = vq[i][j];
    } else {
#pragma unroll 8
      for (int d = 0; d < D; ++d) s = fmaf(__half2float(st_Ud[d * ku.rd + j]), vq[i][d], s);
    }
    wq[i][j] = s;
  }
  __syncthreads();
  // c = G[h] w (r_T < T) or w (r_T = T)
  for (int x = tid; x < NQ * Kk; x += 128) {
    const int i = x / Kk, k = x % Kk;
    float s;
    if (kfT) {
      s = wq[i][k];
    } else {
      s = 0.f;
#pragma unroll 8
      for (int j = 0; j < ku.rd; ++j) s = fmaf(__half2float(st_G[k * ku.rd + j]), wq[i][j], s);
    }
    qc[k * NQ + i] = s;
  }
  // v~ = H_D diag(sigma) v / sqrt(D), a warp per query
  if (ku.b > 0) {
    const unsigned char* sb = (const unsigned char*)kb + 88;
    const float rs = rsqrtf((float)D);
    for (int i = w; i < NQ; i += 4) {
      float v[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = sign_of(sb, lane * EPT + e) * vq[i][lane * EPT + e];
      fwht_row<EPT>(v, lane);
#pragma unroll
      for (int e = 0; e < EPT; ++e) qc[(KM + lane * EPT + e) * NQ + i] = v[e] * rs;
    }
  }
}

// One chunk CTA's view of its (chunk, head, group): the two blobs, the
// low-rank row length of each (U_T rows, or G rows when r_T = T), whether
// the rows are short enough to stage, and the chunk's first rows.
struct ChunkView {
  int chunk, h, g, t0, n, Kk, Kv, kcb, vcb;   // kcb, vcb: code bytes per row
  bool kst, vst;
  AttUnit ku, vu;
  const char* kb;
  const char* vb;
  const __half* kR;
  const __half* vR;
};

template <int D>
__device__ __forceinline__ ChunkView chunk_view(const AttArgs& a) {
  ChunkView c;
  c.chunk = blockIdx.x;
  c.h = blockIdx.y;
  const int gl = blockIdx.z, T = a.T;
  c.g = a.g0 + gl;
  c.t0 = c.chunk * ATT_CHUNK;
  c.n = min(ATT_CHUNK, T - c.t0);
  c.ku = a.k[gl];
  c.vu = a.v[gl];
  c.kb = a.blob + (unsigned long long)(2 * c.g) * a.stride;
  c.vb = a.blob + (unsigned long long)(2 * c.g + 1) * a.stride;
  const bool kfT = (c.ku.rT == T), vfT = (c.vu.rT == T);
  c.Kk = kfT ? c.ku.rd : c.ku.rT;
  c.Kv = vfT ? c.vu.rd : c.vu.rT;
  c.kst = c.Kk <= ATT_STAGE_RANK;
  c.vst = c.Kv <= ATT_STAGE_RANK;
  c.kR = kfT ? (const __half*)(c.kb + c.ku.off_G) + ((size_t)c.h * T + c.t0) * c.ku.rd
             : (const __half*)(c.kb + c.ku.off_UT) + (size_t)c.t0 * c.ku.rT;
  c.vR = vfT ? (const __half*)(c.vb + c.vu.off_G) + ((size_t)c.h * T + c.t0) * c.vu.rd
             : (const __half*)(c.vb + c.vu.off_UT) + (size_t)c.t0 * c.vu.rT;
  c.kcb = D * c.ku.b / 8;
  c.vcb = D * c.vu.b / 8;
  return c;
}

// n rows of row_bytes (a multiple of 16; 16-byte aligned source) from
// global to shared memory at a pitch of row_bytes + 16, 16 bytes per copy.
__device__ __forceinline__ void copy_rows_async(char* dst, const char* src, int n, int row_bytes,
                                                int tid, int nthr) {
  const int per = row_bytes >> 4;
  for (int p = tid; p < n * per; p += nthr) {
    const int r = p / per, q = p - r * per;
    const uint32_t sd = (uint32_t)__cvta_generic_to_shared(dst + r * (row_bytes + 16) + 16 * q);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sd), "l"(src + 16 * p)
                 : "memory");
  }
}

// Everything the CTA reads, in flight at once: the chunk's codes and short
// low-rank rows of both blobs and the V scales (into sv), then, once the
// prep grid has finished, c and v~ (into qcs).  PADV: the V code rows land
// at a pitch of 16 bytes more than their length.  Returns this thread's
// token's K scale.
template <int D, int NQ, bool PADV = false>
__device__ __forceinline__ float chunk_stage(const AttArgs& a, const ChunkView& c, float* qcs,
                                             float* sv, char* data, int tid) {
  const int T = a.T, t = c.t0 + tid;
  // the merge grid may start staging its factors
  asm volatile("griddepcontrol.launch_dependents;");
  if (c.ku.b > 0)
    copy_async(data, c.kb + c.ku.off_codes + ((size_t)c.h * T + c.t0) * c.kcb, c.n * c.kcb, tid,
               ATT_CHUNK);
  if (c.kst) copy_async(data + a.o_kr, c.kR, c.n * c.Kk * 2, tid, ATT_CHUNK);
  if (c.vu.b > 0) {
    const char* src = c.vb + c.vu.off_codes + ((size_t)c.h * T + c.t0) * c.vcb;
    if (PADV) copy_rows_async(data + a.o_vc, src, c.n, c.vcb, tid, ATT_CHUNK);
    else copy_async(data + a.o_vc, src, c.n * c.vcb, tid, ATT_CHUNK);
  }
  if (c.vst) copy_async(data + a.o_vr, c.vR, c.n * c.Kv * 2, tid, ATT_CHUNK);
  asm volatile("cp.async.commit_group;" ::: "memory");
  const float ks =
      (c.ku.b > 0 && t < T)
          ? __half2float(((const __half*)(c.kb + c.ku.off_scale))[(size_t)c.h * T + t]) : 0.f;
  sv[tid] = (c.vu.b > 0 && t < T)
                ? __half2float(((const __half*)(c.vb + c.vu.off_scale))[(size_t)c.h * T + t]) : 0.f;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  copy_async(qcs, a.qc + ((size_t)c.g * a.H + c.h) * (KM + D) * NQ, (KM + D) * NQ * 4, tid,
             ATT_CHUNK);
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  return ks;
}

// Phase 2: the chunk's scores sc[x][i] become probabilities against the
// chunk's max (a warp per query); stat gets the max and the sum.
template <int NQ>
__device__ __forceinline__ void chunk_softmax(float* sc, float* stat, int w, int lane) {
  for (int i = w; i < NQ; i += ATT_WARPS) {
    float m = -INFINITY;
    for (int x = lane; x < ATT_CHUNK; x += 32) m = fmaxf(m, sc[x * NQ + i]);
    m = warp_max(m);
    float l = 0.f;
    for (int x = lane; x < ATT_CHUNK; x += 32) {
      const float p = expf(sc[x * NQ + i] - m);
      sc[x * NQ + i] = p;
      l += p;
    }
    l = warp_sum(l);
    if (lane == 0) { stat[i] = m; stat[8 + i] = l; }
  }
}

// The chunk's record: max, sum, then z and cv of each query, summed over
// the warps' partials red[warp][query][D + KM].
template <int D, int NQ>
__device__ __forceinline__ void chunk_record(const AttArgs& a, const ChunkView& c,
                                             const float* stat, const float* red, int tid) {
  const int nq = a.nq;
  float* rec = a.part + (((size_t)c.g * a.H + c.h) * a.nch + c.chunk) * rec_floats(nq, D);
  if (tid < nq) {
    rec[tid] = stat[tid];
    rec[nq + tid] = stat[8 + tid];
  }
  for (int x = tid; x < nq * (D + KM); x += ATT_CHUNK) {
    const int i = x / (D + KM), col = x % (D + KM);
    if (col >= D + c.Kv) continue;
    float s = 0.f;
#pragma unroll
    for (int ww = 0; ww < ATT_WARPS; ++ww) s += red[(size_t)ww * NQ * (D + KM) + i * (D + KM) + col];
    rec[2 * nq + (size_t)i * (D + KM) + col] = s;
  }
}

template <int EPT, int NQ>
__global__ void __launch_bounds__(ATT_CHUNK) attend_chunk_kernel(AttArgs a) {
  constexpr int D = 32 * EPT;
  extern __shared__ __align__(16) float asm_[];
  float* qcs = asm_;                      // [KM + D][NQ]  c, then v~
  float* sc = qcs + (KM + D) * NQ;        // [CHUNK][NQ]   scores, then p
  float* stat = sc + ATT_CHUNK * NQ;      // [2][8]        max, sum
  float* sv = stat + 16;                  // [CHUNK]       V scales
  char* data = reinterpret_cast<char*>(sv + ATT_CHUNK);   // codes and rows; later the partials
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const ChunkView c = chunk_view<D>(a);
  const AttUnit ku = c.ku, vu = c.vu;
  const int T = a.T, t = c.t0 + tid, n = c.n, Kk = c.Kk, Kv = c.Kv;
  const float ks = chunk_stage<D, NQ>(a, c, qcs, sv, data, tid);

  // ---- phase 1: one thread per token, the scores of every query
  {
    float acc[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) acc[i] = 0.f;
    if (t < T) {
      const __half* R = c.kst ? reinterpret_cast<const __half*>(data + a.o_kr) + (size_t)tid * Kk
                              : c.kR + (size_t)tid * Kk;
      if ((Kk & 1) == 0) {
        const __half2* R2 = reinterpret_cast<const __half2*>(R);
#pragma unroll 8
        for (int k2 = 0; k2 < Kk / 2; ++k2) {
          const float2 r = __half22float2(R2[k2]);
          float c0[NQ], c1[NQ];
          load_q<NQ>(qcs + 2 * k2 * NQ, c0);
          load_q<NQ>(qcs + (2 * k2 + 1) * NQ, c1);
#pragma unroll
          for (int i = 0; i < NQ; ++i) acc[i] = fmaf(r.y, c1[i], fmaf(r.x, c0[i], acc[i]));
        }
      } else {
#pragma unroll 8
        for (int k = 0; k < Kk; ++k) {
          const float r = __half2float(R[k]);
          float c0[NQ];
          load_q<NQ>(qcs + k * NQ, c0);
#pragma unroll
          for (int i = 0; i < NQ; ++i) acc[i] = fmaf(r, c0[i], acc[i]);
        }
      }
      if (ku.b > 0) {
        float r[NQ];
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(data + tid * c.kcb);
        const float* vt = qcs + KM * NQ;
        if (ku.b == 2) res_dots<D, NQ, 2>(cw, vt, r);
        else if (ku.b == 4) res_dots<D, NQ, 4>(cw, vt, r);
        else res_dots<D, NQ, 8>(cw, vt, r);
#pragma unroll
        for (int i = 0; i < NQ; ++i) acc[i] = fmaf(ks, r[i], acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < NQ; ++i) sc[tid * NQ + i] = (t < T) ? a.scale * acc[i] : -INFINITY;
  }
  __syncthreads();
  chunk_softmax<NQ>(sc, stat, w, lane);
  __syncthreads();

  // ---- phase 3: cv and z over this warp's 32 tokens
  constexpr int KPL = KM / 32;
  float z[NQ][EPT], cv[NQ][KPL];
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) z[i][e] = 0.f;
#pragma unroll
    for (int j = 0; j < KPL; ++j) cv[i][j] = 0.f;
  }
  {
    const uint32_t* cvw = reinterpret_cast<const uint32_t*>(data + a.o_vc);
    const int rw = D * vu.b / 32;
    const __half* Rb = c.vst ? reinterpret_cast<const __half*>(data + a.o_vr) : c.vR;
    const int ntok = min(32, n - w * 32);
#pragma unroll 4
    for (int j = 0; j < ntok; ++j) {
      const int x = w * 32 + j;
      float p[NQ];
      load_q<NQ>(sc + x * NQ, p);
      const __half* R = Rb + (size_t)x * Kv;
#pragma unroll
      for (int jj = 0; jj < KPL; ++jj) {
        const int k = lane + 32 * jj;
        if (k < Kv) {
          const float r = __half2float(R[k]);
#pragma unroll
          for (int i = 0; i < NQ; ++i) cv[i][jj] = fmaf(p[i], r, cv[i][jj]);
        }
      }
      if (vu.b > 0) {
        const float s = sv[x];
        float ps[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) ps[i] = p[i] * s;
        if (vu.b == 2) res_accum<EPT, NQ, 2>(cvw + x * rw, lane, ps, z);
        else if (vu.b == 4) res_accum<EPT, NQ, 4>(cvw + x * rw, lane, ps, z);
        else res_accum<EPT, NQ, 8>(cvw + x * rw, lane, ps, z);
      }
    }
  }
  __syncthreads();   // the data region becomes the per-warp partial sums
  float* red = reinterpret_cast<float*>(data);
  float* rw_ = red + (size_t)w * NQ * (D + KM);
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) rw_[i * (D + KM) + lane * EPT + e] = z[i][e];
#pragma unroll
    for (int jj = 0; jj < KPL; ++jj) rw_[i * (D + KM) + D + lane + 32 * jj] = cv[i][jj];
  }
  __syncthreads();
  chunk_record<D, NQ>(a, c, stat, red, tid);
}

// ------------------------------------------------ tensor-core chunk, D = 128
// The same three phases for D = 128 with the per-token contractions on
// mma.sync m16n8k16 (fp16 operands, fp32 accumulators; a warp's 32 tokens
// are two 16-row tiles, the queries the 8 columns):
//   phase 1   scores = R_K[t] . c  +  s_t (u_t - 2^(b-1)) . v~   (K = k, d)
//   phase 3   cv^T = R_V^T p,  z^T = (u - 2^(b-1))^T (p s)       (K = tokens)
// The integer codes and the fp16 rows are exact fp16 operands.  The fp32
// side of each product (c, v~, p, p s) is scaled by a power of two that
// brings its largest magnitude just below 2^14, then split into fp16 hi +
// lo (hi = fp16(x), lo = fp16(x - hi)): two MMAs carry 22 bits of each
// value, against the 24 of the fp32 FMAs, and the scale comes off exactly.
// The codes are unpacked as in the decoder (0x6400 | u = 1024 + u, less
// 1024 + 2^(b-1) in half2), sixteen codes of one row at a time, in the
// order unpack16 gives; the K (or M) index of each product follows that
// order, and the other operand is built in the same order.

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// The power of two that brings a largest magnitude m just below 2^14 (1
// for m = 0), built from m's exponent field and clamped to the normal range.
__device__ __forceinline__ float fp16_scale(float m) {
  if (!(m > 0.f)) return 1.f;
  const int e = ((__float_as_int(m) >> 23) & 0xFF) - 126;   // m < 2^e
  const int k = max(-126, min(127, 14 - e));
  return __int_as_float((127 + k) << 23);
}

// hi and lo fp16 parts of two values, packed as half2 (first value low).
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  hi = h2u(__halves2half2(h0, h1));
  lo = h2u(__floats2half2_rn(x0 - __half2float(h0), x1 - __half2float(h1)));
}

// Position, within a group of sixteen codes, of the p-th value unpack16
// gives (value pair m holds positions (lpos(2m), lpos(2m + 1))).
template <int B>
__device__ __forceinline__ int lpos(int p) {
  const int m = p >> 1, e = p & 1;
  if constexpr (B == 2) return 8 * (m & 1) + 4 * e + (m >> 1);
  else if constexpr (B == 4) return 8 * (m >> 2) + 4 * (m & 1) + ((m & 3) >> 1) + 2 * e;
  else return p;
}

// Sixteen b-bit codes (b / 2 words, code i at bits b i) as eight half2 of
// u - 2^(b-1), in lpos order.
template <int B>
__device__ __forceinline__ void unpack16(const uint32_t* w, uint32_t (&hv)[8]) {
  if constexpr (B == 2) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t x = (w[0] >> (2 * s)) & 0x03030303u;
      hv[2 * s] = __byte_perm(x, 0x64646464u, 0x5140);
      hv[2 * s + 1] = __byte_perm(x, 0x64646464u, 0x7362);
    }
  } else if constexpr (B == 4) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t ev = w[j] & 0x0F0F0F0Fu, od = (w[j] >> 4) & 0x0F0F0F0Fu;
      hv[4 * j] = __byte_perm(ev, 0x64646464u, 0x5140);
      hv[4 * j + 1] = __byte_perm(ev, 0x64646464u, 0x7362);
      hv[4 * j + 2] = __byte_perm(od, 0x64646464u, 0x5140);
      hv[4 * j + 3] = __byte_perm(od, 0x64646464u, 0x7362);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hv[2 * j] = __byte_perm(w[j], 0x64646464u, 0x5140);
      hv[2 * j + 1] = __byte_perm(w[j], 0x64646464u, 0x7362);
    }
  }
  const __half2 off = u2h(0x64006400u | (1u << (B - 1)) | (1u << (B + 15)));
#pragma unroll
  for (int m = 0; m < 8; ++m) hv[m] = h2u(__hsub2(u2h(hv[m]), off));
}

// n consecutive 32-bit words of shared memory (n = 1, 2, 4 or 8, 16-byte
// aligned for n >= 4).
template <int N>
__device__ __forceinline__ void lds_words(const uint32_t* p, uint32_t (&o)[N]) {
  if constexpr (N == 1) {
    o[0] = p[0];
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    o[0] = v.x; o[1] = v.y;
  } else {
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[q];
      o[4 * q] = v.x; o[4 * q + 1] = v.y; o[4 * q + 2] = v.z; o[4 * q + 3] = v.w;
    }
  }
}

// Phase 1, residual: acc[mt] += (scaled) v~ . (u - 2^(b-1)) for the warp's
// two 16-token tiles.  Thread (g, q) of the MMA layout takes the 32 codes
// d in [32 q, 32 q + 32) of its rows, sixteen per k-block group: k-block kb
// (0..7) uses group kb / 4, value pairs 2 (kb % 4) and 2 (kb % 4) + 1.
template <int B, int NQ>
__device__ __forceinline__ float res_scores_tc(const char* codes, int kcb, const float* vt,
                                               int w, int lane, float (&acc)[2][4]) {
  const int mg = lane >> 2, mq = lane & 3;
  uint32_t bh[8][2], bl[8][2];
  float vmax = 0.f;
  {
    float vv[8][4];
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 32 * mq + 16 * (kb >> 2) + lpos<B>(4 * (kb & 3) + e);
        vv[kb][e] = mg < NQ ? vt[d * NQ + mg] : 0.f;
        vmax = fmaxf(vmax, fabsf(vv[kb][e]));
      }
    const float sig = fp16_scale(warp_max(vmax));
    vmax = sig;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      split_h2(vv[kb][0] * sig, vv[kb][1] * sig, bh[kb][0], bl[kb][0]);
      split_h2(vv[kb][2] * sig, vv[kb][3] * sig, bh[kb][1], bl[kb][1]);
    }
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int x0 = 32 * w + 16 * mt + mg;
    uint32_t w0[B], w1[B];
    lds_words<B>(reinterpret_cast<const uint32_t*>(codes + x0 * kcb) + mq * B, w0);
    lds_words<B>(reinterpret_cast<const uint32_t*>(codes + (x0 + 8) * kcb) + mq * B, w1);
    uint32_t h0[2][8], h1[2][8];
    unpack16<B>(w0, h0[0]);
    unpack16<B>(w0 + B / 2, h0[1]);
    unpack16<B>(w1, h1[0]);
    unpack16<B>(w1 + B / 2, h1[1]);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const int gq = kb >> 2, m2 = 2 * (kb & 3);
      mma16816(acc[mt], h0[gq][m2], h1[gq][m2], h0[gq][m2 + 1], h1[gq][m2 + 1], bh[kb][0], bh[kb][1]);
      mma16816(acc[mt], h0[gq][m2], h1[gq][m2], h0[gq][m2 + 1], h1[gq][m2 + 1], bl[kb][0], bl[kb][1]);
    }
  }
  return 1.f / vmax;   // the inverse scale (a power of two)
}

// Two fp16 values of low-rank rows as one half2: row x0 at k and row x1 at
// k (pair = false), or row x0 at k and k + 1 (pair = true); zero past the
// row length K or the chunk's n rows.
__device__ __forceinline__ uint32_t row_pair(const __half* R, int K, int n, int x0, int x1, int k,
                                             bool pair) {
  const unsigned short z = 0;
  unsigned short v0, v1;
  if (pair) {
    v0 = (x0 < n && k < K) ? __half_as_ushort(R[(size_t)x0 * K + k]) : z;
    v1 = (x0 < n && k + 1 < K) ? __half_as_ushort(R[(size_t)x0 * K + k + 1]) : z;
  } else {
    v0 = (x0 < n && k < K) ? __half_as_ushort(R[(size_t)x0 * K + k]) : z;
    v1 = (x1 < n && k < K) ? __half_as_ushort(R[(size_t)x1 * K + k]) : z;
  }
  return (uint32_t)v0 | ((uint32_t)v1 << 16);
}

// Per-warp partial sums of the tensor-core chunk: a row of NQ floats per
// entry (z at d, then cv at D + k), each 16 entries followed by one unused
// row, so that the 8-byte stores of a fragment (8 row groups x 4 query
// pairs) fall in different banks.
constexpr int TC_RED_ROWS = (128 + KM) + (128 + KM) / 16;
__device__ __forceinline__ int tc_red_row(int e) { return e + (e >> 4); }

template <int NQ>
__global__ void __launch_bounds__(ATT_CHUNK) attend_chunk_tc_kernel(AttArgs a) {
  constexpr int D = 128;
  extern __shared__ __align__(16) float asm_[];
  float* qcs = asm_;                      // [KM + D][NQ]  c, then v~
  float* sc = qcs + (KM + D) * NQ;        // [CHUNK][NQ]   scores, then p
  float* stat = sc + ATT_CHUNK * NQ;      // [2][8]        max, sum
  float* sv = stat + 16;                  // [CHUNK]       V scales
  char* data = reinterpret_cast<char*>(sv + ATT_CHUNK);   // codes and rows; later the partials
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int mg = lane >> 2, mq = lane & 3;   // MMA fragment row group, column pair
  const ChunkView c = chunk_view<D>(a);
  const int n = c.n, Kk = c.Kk, Kv = c.Kv;
  const float ks = chunk_stage<D, NQ, true>(a, c, qcs, sv, data, tid);

  // ---- phase 1: scores of the warp's 32 tokens (rows 16 mt + mg, + 8)
  {
    float accr[2][4] = {}, accl[2][4] = {};
    float ir = 0.f;
    if (c.ku.b == 2) ir = res_scores_tc<2, NQ>(data, c.kcb, qcs + KM * NQ, w, lane, accr);
    else if (c.ku.b == 4) ir = res_scores_tc<4, NQ>(data, c.kcb, qcs + KM * NQ, w, lane, accr);
    else if (c.ku.b == 8) ir = res_scores_tc<8, NQ>(data, c.kcb, qcs + KM * NQ, w, lane, accr);
    // low rank: R_K[t] . c, k-blocks of 16 (thread pairs 2 mq, 2 mq + 8)
    const int nkb = (Kk + 15) >> 4;
    float cmax = 0.f;
    for (int kb = 0; kb < nkb; ++kb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 16 * kb + 2 * mq + (e & 1) + 8 * (e >> 1);
        if (k < Kk && mg < NQ) cmax = fmaxf(cmax, fabsf(qcs[k * NQ + mg]));
      }
    const float sl = fp16_scale(warp_max(cmax));
    const __half* R = c.kst ? reinterpret_cast<const __half*>(data + a.o_kr) : c.kR;
    // staged rows of even length: one 32-bit load per pair (rows past the
    // chunk's n only feed their own scores, which are dropped)
    const bool fastk = c.kst && (Kk & 1) == 0;
    const uint32_t* R32 = reinterpret_cast<const uint32_t*>(data + a.o_kr);
    for (int kb = 0; kb < nkb; ++kb) {
      float cv4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 16 * kb + 2 * mq + (e & 1) + 8 * (e >> 1);
        cv4[e] = (k < Kk && mg < NQ) ? qcs[k * NQ + mg] * sl : 0.f;
      }
      uint32_t bh0, bl0, bh1, bl1;
      split_h2(cv4[0], cv4[1], bh0, bl0);
      split_h2(cv4[2], cv4[3], bh1, bl1);
      const int k0 = 16 * kb + 2 * mq;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int x0 = 32 * w + 16 * mt + mg, x1 = x0 + 8;
        uint32_t a0, a1, a2, a3;
        if (fastk) {
          a0 = k0 < Kk ? R32[(x0 * Kk + k0) >> 1] : 0u;
          a1 = k0 < Kk ? R32[(x1 * Kk + k0) >> 1] : 0u;
          a2 = k0 + 8 < Kk ? R32[(x0 * Kk + k0 + 8) >> 1] : 0u;
          a3 = k0 + 8 < Kk ? R32[(x1 * Kk + k0 + 8) >> 1] : 0u;
        } else {
          a0 = row_pair(R, Kk, n, x0, x0, k0, true);
          a1 = row_pair(R, Kk, n, x1, x1, k0, true);
          a2 = row_pair(R, Kk, n, x0, x0, k0 + 8, true);
          a3 = row_pair(R, Kk, n, x1, x1, k0 + 8, true);
        }
        mma16816(accl[mt], a0, a1, a2, a3, bh0, bh1);
        mma16816(accl[mt], a0, a1, a2, a3, bl0, bl1);
      }
    }
    const float il = 1.f / sl;
    // score = scale (lr + s_t res); c0, c1: row mg, queries 2 mq, 2 mq + 1;
    // c2, c3: row mg + 8; the K scale of token x sits in lane x % 32
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int xr = 16 * mt + mg + 8 * hr, x = 32 * w + xr;
        const float kx = __shfl_sync(0xffffffffu, ks, xr);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = 2 * mq + j;
          const float s = a.scale * fmaf(kx, accr[mt][2 * hr + j] * ir, accl[mt][2 * hr + j] * il);
          if (i < NQ) sc[x * NQ + i] = x < n ? s : -INFINITY;
        }
      }
  }
  __syncthreads();
  chunk_softmax<NQ>(sc, stat, w, lane);
  __syncthreads();

  // ---- phase 3: z^T (d x queries) and cv^T (k x queries) over the warp's
  // 32 tokens, two k-blocks of 16 (thread tokens 2 mq, 2 mq + 1, + 8, + 9)
  float zacc[8][4] = {}, cacc[8][4] = {};
  const int vb = c.vu.b;
  float pmax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 8) pmax = fmaxf(pmax, sv[32 * w + j + (lane & 7)]);
  const float sz = fp16_scale(warp_max(pmax));   // p s <= max s: p <= 1
  const float sp = 16384.f;                       // p <= 1
  const int nmk = (Kv + 15) >> 4;
  const __half* RV = c.vst ? reinterpret_cast<const __half*>(data + a.o_vr) : c.vR;
  const unsigned short* RV16 = reinterpret_cast<const unsigned short*>(data + a.o_vr);
  const char* vcodes = data + a.o_vc;
  const int vpitch = c.vcb + 16;   // padded rows: lanes 2 mq apart hit different banks
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    const int xb = 32 * w + 16 * kb + 2 * mq;
    const int xs[4] = {xb, xb + 1, xb + 8, xb + 9};
    float p[4], ps[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = mg < NQ ? sc[xs[e] * NQ + mg] : 0.f;
      ps[e] = p[e] * sv[xs[e]] * sz;
      p[e] *= sp;
    }
    uint32_t bzh0, bzl0, bzh1, bzl1, bch0, bcl0, bch1, bcl1;
    split_h2(ps[0], ps[1], bzh0, bzl0);
    split_h2(ps[2], ps[3], bzh1, bzl1);
    split_h2(p[0], p[1], bch0, bcl0);
    split_h2(p[2], p[3], bch1, bcl1);
    if (vb > 0) {
      uint32_t hv[4][8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t* row = reinterpret_cast<const uint32_t*>(vcodes + xs[e] * vpitch);
        if (vb == 2) {
          uint32_t wd[1];
          lds_words<1>(row + mg, wd);
          unpack16<2>(wd, hv[e]);
        } else if (vb == 4) {
          uint32_t wd[2];
          lds_words<2>(row + 2 * mg, wd);
          unpack16<4>(wd, hv[e]);
        } else {
          uint32_t wd[4];
          lds_words<4>(row + 4 * mg, wd);
          unpack16<8>(wd, hv[e]);
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t a0 = __byte_perm(hv[0][m], hv[1][m], 0x5410);
        const uint32_t a1 = __byte_perm(hv[0][m], hv[1][m], 0x7632);
        const uint32_t a2 = __byte_perm(hv[2][m], hv[3][m], 0x5410);
        const uint32_t a3 = __byte_perm(hv[2][m], hv[3][m], 0x7632);
        mma16816(zacc[m], a0, a1, a2, a3, bzh0, bzh1);
        mma16816(zacc[m], a0, a1, a2, a3, bzl0, bzl1);
      }
    }
    // the rows of tokens past the chunk's n are zero here: they multiply
    // every query's weights
    bool xv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) xv[e] = xs[e] < n;
#pragma unroll
    for (int mk = 0; mk < 8; ++mk) {
      if (mk < nmk) {
        const int k0 = 16 * mk + mg;
        uint32_t a0, a1, a2, a3;
        if (c.vst) {
          uint32_t v[4][2];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[e][0] = (xv[e] && k0 < Kv) ? RV16[xs[e] * Kv + k0] : 0u;
            v[e][1] = (xv[e] && k0 + 8 < Kv) ? RV16[xs[e] * Kv + k0 + 8] : 0u;
          }
          a0 = v[0][0] | (v[1][0] << 16);
          a1 = v[0][1] | (v[1][1] << 16);
          a2 = v[2][0] | (v[3][0] << 16);
          a3 = v[2][1] | (v[3][1] << 16);
        } else {
          a0 = row_pair(RV, Kv, n, xs[0], xs[1], k0, false);
          a1 = row_pair(RV, Kv, n, xs[0], xs[1], k0 + 8, false);
          a2 = row_pair(RV, Kv, n, xs[2], xs[3], k0, false);
          a3 = row_pair(RV, Kv, n, xs[2], xs[3], k0 + 8, false);
        }
        mma16816(cacc[mk], a0, a1, a2, a3, bch0, bch1);
        mma16816(cacc[mk], a0, a1, a2, a3, bcl0, bcl1);
      }
    }
  }
  __syncthreads();   // the data region becomes the per-warp partial sums
  float* red = reinterpret_cast<float*>(data);
  float* rw_ = red + (size_t)w * TC_RED_ROWS * NQ;
  const float iz = 1.f / sz, ip = 1.f / sp;
  // a query pair (2 mq, 2 mq + 1) of one row, as one 8-byte store
  auto put = [&](int row, float v0, float v1) {
    if constexpr (NQ == 1) {
      if (mq == 0) rw_[row] = v0;
    } else {
      if (2 * mq < NQ) *reinterpret_cast<float2*>(rw_ + row * NQ + 2 * mq) = make_float2(v0, v1);
    }
  };
  // z^T rows of tile m: mg <-> d = 16 mg + lpos(2 m), mg + 8 <-> lpos(2 m + 1)
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    int d0, d1;
    if (vb == 2) { d0 = lpos<2>(2 * m); d1 = lpos<2>(2 * m + 1); }
    else if (vb == 4) { d0 = lpos<4>(2 * m); d1 = lpos<4>(2 * m + 1); }
    else { d0 = 2 * m; d1 = 2 * m + 1; }
    d0 += 16 * mg;
    d1 += 16 * mg;
    put(tc_red_row(d0), zacc[m][0] * iz, zacc[m][1] * iz);
    put(tc_red_row(d1), zacc[m][2] * iz, zacc[m][3] * iz);
  }
#pragma unroll
  for (int mk = 0; mk < 8; ++mk) {
    if (mk < nmk) {
      const int k0 = 16 * mk + mg;
      put(tc_red_row(D + k0), cacc[mk][0] * ip, cacc[mk][1] * ip);
      put(tc_red_row(D + k0 + 8), cacc[mk][2] * ip, cacc[mk][3] * ip);
    }
  }
  __syncthreads();
  // the chunk's record: max, sum, z, cv, each entry summed over the warps
  const int nq = a.nq;
  float* rec = a.part + (((size_t)c.g * a.H + c.h) * a.nch + c.chunk) * rec_floats(nq, D);
  if (tid < nq) {
    rec[tid] = stat[tid];
    rec[nq + tid] = stat[8 + tid];
  }
  for (int x = tid; x < (D + Kv) * NQ; x += ATT_CHUNK) {
    const int col = x / NQ, i = x % NQ;
    if (i >= nq) continue;
    const int row = tc_red_row(col);
    float s = 0.f;
#pragma unroll
    for (int ww = 0; ww < ATT_WARPS; ++ww) s += red[(ww * TC_RED_ROWS + row) * NQ + i];
    rec[2 * nq + (size_t)i * (D + KM) + col] = s;
  }
}

// Merge the chunks of one (head, group) for each of its queries and map
// back to feature space: U_d and G[h] are staged once for all the queries.
template <int EPT>
__global__ void __launch_bounds__(128) attend_merge_kernel(AttArgs a) {
  constexpr int D = 32 * EPT, QM = JOLT_ATTN_MAX_Q;
  __shared__ float zf[QM][D], cf[QM][KM], ef[QM][KM > D ? KM : D], sM[QM], sL[QM];
  __shared__ __half st_Ud[D * 64], st_G[64 * (KM > D ? KM : D)];
  const int h = blockIdx.x, gl = blockIdx.y, g = a.g0 + gl;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int T = a.T, H = a.H, nq = a.nq, nch = a.nch;
  const AttUnit vu = a.v[gl];
  const char* vb = a.blob + (unsigned long long)(2 * g + 1) * a.stride;
  const bool vfT = (vu.rT == T), vfD = (vu.rd == D);
  const int Kv = vfT ? vu.rd : vu.rT;
  const size_t rf = rec_floats(nq, D);
  const float* base = a.part + ((size_t)g * H + h) * nch * rf;
  if (!vfD) stage_halves(st_Ud, (const __half*)(vb + vu.off_Ud), D * vu.rd, tid, 128);
  if (!vfT)
    stage_halves(st_G, (const __half*)(vb + vu.off_G) + (size_t)h * vu.rT * vu.rd,
                 vu.rT * vu.rd, tid, 128);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the global max M and sum L of each query (a warp per query)
  for (int i = w; i < nq; i += 4) {
    float m = -INFINITY;
    for (int c = lane; c < nch; c += 32) m = fmaxf(m, base[c * rf + i]);
    m = warp_max(m);
    float l = 0.f;
    for (int c = lane; c < nch; c += 32) l += expf(base[c * rf + i] - m) * base[c * rf + nq + i];
    l = warp_sum(l);
    if (lane == 0) { sM[i] = m; sL[i] = l; }
  }
  __syncthreads();
  // z and cv of every query: the chunk records weighted by exp(m_c - M)
  const int ne = D + Kv;
  for (int x = tid; x < nq * ne; x += 128) {
    const int i = x / ne, col = x - i * ne;
    const float M = sM[i];
    const size_t at = 2 * nq + (size_t)i * (D + KM) + col;
    float s = 0.f;
#pragma unroll 4
    for (int c = 0; c < nch; ++c) {
      const float* r = base + c * rf;
      s = fmaf(expf(r[i] - M), r[at], s);
    }
    if (col < D) zf[i][col] = s; else cf[i][col - D] = s;
  }
  __syncthreads();
  // back-projection, stage 1: e = G[h]^T cv (r_T < T) or cv itself (r_T = T)
  for (int x = tid; x < nq * vu.rd; x += 128) {
    const int i = x / vu.rd, j = x - i * vu.rd;
    float s;
    if (vfT) {
      s = cf[i][j];
    } else {
      s = 0.f;
#pragma unroll 8
      for (int k = 0; k < vu.rT; ++k) s = fmaf(__half2float(st_G[k * vu.rd + j]), cf[i][k], s);
    }
    ef[i][j] = s;
  }
  __syncthreads();
  // stage 2 (U_d e) plus the inverse rotation of z: a warp per query
  const unsigned char* sb = (const unsigned char*)vb + 88;
  const float rs = rsqrtf((float)D);
  for (int i = w; i < nq; i += 4) {
    float v[EPT];
    if (vu.b > 0) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = zf[i][lane * EPT + e];
      fwht_row<EPT>(v, lane);
    }
    const float inv = 1.f / sL[i];
    float* o = a.out + (((size_t)g * H + h) * nq + i) * D;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int d = lane * EPT + e;
      float lo;
      if (vfD) {
        lo = ef[i][d];
      } else {
        lo = 0.f;
#pragma unroll 8
        for (int j = 0; j < vu.rd; ++j) lo = fmaf(__half2float(st_Ud[d * vu.rd + j]), ef[i][j], lo);
      }
      const float res = (vu.b > 0) ? sign_of(sb, d) * v[e] * rs : 0.f;
      o[d] = (lo + res) * inv;
    }
  }
}

template <int EPT, int NQ>
jolt_status launch_attend(const AttArgs& a, int ng, cudaStream_t st) {
  constexpr int D = 32 * EPT;
  const size_t smem = sizeof(float) * ((KM + D) * NQ + ATT_CHUNK * NQ + 16 + ATT_CHUNK) + a.data;
  if (smem > 227 * 1024) return JOLT_ERR_INVALID;
  // D = 128 takes the tensor-core chunk kernel
  auto chunk = EPT == 4 ? attend_chunk_tc_kernel<NQ> : attend_chunk_kernel<EPT, NQ>;
  static int attr = 0;
  if ((int)smem > attr) {
    JOLT_CUDA_TRY(
        cudaFuncSetAttribute(chunk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = (int)smem;
  }
  attend_prep_kernel<EPT, NQ><<<dim3(a.H, ng), 128, 0, st>>>(a);
  JOLT_LAUNCH_CHECK();
  // the chunk and merge grids are programmatic dependents of the grid
  // before them: their CTAs start staging data while it still runs and wait
  // for it (griddepcontrol.wait) before reading its results
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.stream = st;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(a.nch, a.H, ng);
  cfg.blockDim = dim3(ATT_CHUNK);
  cfg.dynamicSmemBytes = smem;
  JOLT_CUDA_TRY(cudaLaunchKernelEx(&cfg, chunk, a));
  JOLT_LAUNCH_CHECK();
  cfg.gridDim = dim3(a.H, ng);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  JOLT_CUDA_TRY(cudaLaunchKernelEx(&cfg, attend_merge_kernel<EPT>, a));
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

template <int EPT>
jolt_status launch_attend_nq(const AttArgs& a, int ng, cudaStream_t st) {
  switch (nq_pad(a.nq)) {
    case 1: return launch_attend<EPT, 1>(a, ng, st);
    case 2: return launch_attend<EPT, 2>(a, ng, st);
    case 4: return launch_attend<EPT, 4>(a, ng, st);
    default: return launch_attend<EPT, 8>(a, ng, st);
  }
}

AttUnit att_unit(const jolt_blob_desc& d) {
  AttUnit u;
  u.rT = d.rT; u.rd = d.rd; u.b = d.b; u.pad = 0;
  u.off_UT = d.off_UT; u.off_Ud = d.off_Ud; u.off_G = d.off_G;
  u.off_scale = d.off_scale; u.off_codes = d.off_codes;
  return u;
}

// Low-rank row length of a blob (r_T < T: U_T rows; r_T = T: G rows).
int row_len(const jolt_blob_desc& d) { return d.rT == d.T ? d.rd : d.rT; }

size_t part_bytes(int n_groups, int H, int T, int D, int nq) {
  return align_up((size_t)n_groups * H * ((T + ATT_CHUNK - 1) / ATT_CHUNK) * rec_floats(nq, D) *
                      sizeof(float), 256);
}

}  // namespace

size_t attend_ws_bytes(int n_groups, int H, int T, int D, int nq) {
  return part_bytes(n_groups, H, T, D, nq) +
         (size_t)n_groups * H * (KM + D) * nq_pad(nq) * sizeof(float);
}

jolt_status attend_run(int n_groups, const jolt_blob_desc* desc, const char* blob,
                       size_t stride, const float* q, int nq, float scale, float* ws,
                       float* out, cudaStream_t st) {
  const int H = desc[0].H, T = desc[0].T, D = desc[0].D;
  float* part = ws;
  float* qc = (float*)((char*)ws + part_bytes(n_groups, H, T, D, nq));
  for (int g0 = 0; g0 < n_groups; g0 += ATT_MAX_G) {
    const int ng = (n_groups - g0) < ATT_MAX_G ? (n_groups - g0) : ATT_MAX_G;
    AttArgs a;
    memset(&a, 0, sizeof(a));
    a.H = H; a.T = T; a.nq = nq; a.nch = (T + ATT_CHUNK - 1) / ATT_CHUNK;
    a.scale = scale; a.blob = blob; a.stride = stride; a.q = q; a.qc = qc; a.part = part;
    a.out = out; a.g0 = g0;
    // the data region holds the largest K codes, K rows, V codes, V rows of
    // this launch's groups (rows only when short enough to stage)
    size_t kc = 0, kr = 0, vc = 0, vr = 0;
    for (int i = 0; i < ng; ++i) {
      const jolt_blob_desc& kd = desc[2 * (g0 + i)];
      const jolt_blob_desc& vd = desc[2 * (g0 + i) + 1];
      a.k[i] = att_unit(kd);
      a.v[i] = att_unit(vd);
      kc = std::max(kc, (size_t)ATT_CHUNK * D * kd.b / 8);
      // D = 128: V code rows at a pitch of 16 bytes more than their length
      vc = std::max(vc, (size_t)ATT_CHUNK * (D * vd.b / 8 + (D == 128 && vd.b > 0 ? 16 : 0)));
      if (row_len(kd) <= ATT_STAGE_RANK) kr = std::max(kr, (size_t)ATT_CHUNK * row_len(kd) * 2);
      if (row_len(vd) <= ATT_STAGE_RANK) vr = std::max(vr, (size_t)ATT_CHUNK * row_len(vd) * 2);
    }
    a.o_kr = (int)align_up(kc, 16);
    a.o_vc = (int)align_up(a.o_kr + kr, 16);
    a.o_vr = (int)align_up(a.o_vc + vc, 16);
    const size_t red = sizeof(float) * ATT_WARPS * nq_pad(nq) *
                       (D == 128 ? (size_t)TC_RED_ROWS : (size_t)(D + KM));
    a.data = (int)align_up(std::max((size_t)a.o_vr + vr, red), 16);
    jolt_status s;
    switch (D) {
      case 128: s = launch_attend_nq<4>(a, ng, st); break;
      case 64: s = launch_attend_nq<2>(a, ng, st); break;
      default: s = launch_attend_nq<1>(a, ng, st);
    }
    if (s != JOLT_OK) return s;
  }
  return JOLT_OK;
}

}  // namespace jolt
