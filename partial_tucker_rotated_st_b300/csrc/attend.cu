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
// Tokens are split into chunks of ATT_CHUNK, one CTA per (chunk, head, group):
// phase 1 scores the chunk's tokens (one thread per token), phase 2 turns them
// into probabilities against the chunk's max, phase 3 accumulates cv and z
// (a warp per 32 tokens, lanes over the feature / rank index), and the CTA
// writes its max, sum, cv and z.  A second kernel merges the chunks
// (flash-decoding) and applies the back-projection and the inverse rotation.
#include "jolt_internal.cuh"

namespace jolt {

namespace {

constexpr int ATT_CHUNK = 128;     // tokens per CTA = threads per CTA
constexpr int ATT_WARPS = ATT_CHUNK / 32;
constexpr int ATT_MAX_G = 16;      // groups per launch

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
  float* part;          // [groups][H][nch][rec]
  float* out;           // [groups][H][nq][D]
  int g0;               // first group of this launch
  AttUnit k[ATT_MAX_G], v[ATT_MAX_G];
};

// b-bit code u as the float u - 2^(b-1), exactly: 2^23 + u has u in its low
// mantissa bits.
__device__ __forceinline__ float code_f(unsigned u, float bias) {
  return __uint_as_float(0x4B000000u | u) - bias;
}

__device__ __forceinline__ size_t rec_floats(int nq, int D) {
  return (size_t)nq * (2 + D + JOLT_ATTN_MAX_RANK);
}

// One token's residual dot products sum_d v~_i[d] (u_d - 2^(b-1)) for every
// query, the codes row read as 32-bit words (B bits per code).
template <int D, int NQ, int B>
__device__ __forceinline__ void res_dots(const uint32_t* __restrict__ row,
                                         const float* __restrict__ vt, float (&r)[NQ]) {
  constexpr int PER = 32 / B;              // codes per word
  constexpr int NW = D * B / 32;           // words per row
  constexpr unsigned MASK = (1u << B) - 1u;
  const float bias = 8388608.0f + (float)(1 << (B - 1));
#pragma unroll
  for (int i = 0; i < NQ; ++i) r[i] = 0.f;
  if constexpr (NW % 4 == 0) {
#pragma unroll 2
    for (int w4 = 0; w4 < NW / 4; ++w4) {
      const uint4 wv = reinterpret_cast<const uint4*>(row)[w4];
      const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int d = (w4 * 4 + c) * PER + j;
          const float f = code_f((ws[c] >> (j * B)) & MASK, bias);
#pragma unroll
          for (int i = 0; i < NQ; ++i) r[i] = fmaf(vt[d * NQ + i], f, r[i]);
        }
    }
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t wd = row[w];
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int d = w * PER + j;
        const float f = code_f((wd >> (j * B)) & MASK, bias);
#pragma unroll
        for (int i = 0; i < NQ; ++i) r[i] = fmaf(vt[d * NQ + i], f, r[i]);
      }
    }
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

template <int EPT, int NQ>
__global__ void __launch_bounds__(ATT_CHUNK) attend_chunk_kernel(AttArgs a) {
  constexpr int D = 32 * EPT;
  constexpr int KM = JOLT_ATTN_MAX_RANK;
  extern __shared__ __align__(16) float asm_[];
  float* vq = asm_;                       // [NQ][D]   queries
  float* wq = vq + NQ * D;                // [NQ][KM]  U_d^T v
  float* cq = wq + NQ * KM;               // [KM][NQ]  score coefficients of R[t]
  float* vt = cq + KM * NQ;               // [D][NQ]   rotated queries v~
  float* sc = vt + D * NQ;                // [CHUNK][NQ] scores, then p
  float* red = sc + ATT_CHUNK * NQ;       // [WARPS][NQ][D + KM]
  float* stat = red + ATT_WARPS * NQ * (D + KM);   // [2][NQ] max, sum
  const int chunk = blockIdx.x, h = blockIdx.y, gl = blockIdx.z;
  const int g = a.g0 + gl;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int T = a.T, H = a.H, nq = a.nq;
  const int t0 = chunk * ATT_CHUNK;
  const AttUnit ku = a.k[gl], vu = a.v[gl];
  const char* kb = a.blob + (unsigned long long)(2 * g) * a.stride;
  const char* vb = a.blob + (unsigned long long)(2 * g + 1) * a.stride;

  // ---- queries and their coefficients for the K blob
  const float* qg = a.q + ((size_t)g * H + h) * nq * D;
  for (int x = tid; x < NQ * D; x += ATT_CHUNK) {
    const int i = x / D;
    vq[x] = i < nq ? qg[x] : 0.f;
  }
  __syncthreads();
  const bool kfT = (ku.rT == T), kfD = (ku.rd == D);
  const int Kk = kfT ? ku.rd : ku.rT;
  {
    const __half* Ud = (const __half*)(kb + ku.off_Ud);
    for (int x = tid; x < NQ * ku.rd; x += ATT_CHUNK) {
      const int i = x / ku.rd, j = x % ku.rd;
      float s = 0.f;
      if (kfD) {
        s = vq[i * D + j];
      } else {
        for (int d = 0; d < D; ++d) s = fmaf(__half2float(Ud[d * ku.rd + j]), vq[i * D + d], s);
      }
      wq[i * KM + j] = s;
    }
  }
  __syncthreads();
  if (kfT) {
    for (int x = tid; x < NQ * Kk; x += ATT_CHUNK) {
      const int i = x / Kk, k = x % Kk;
      cq[k * NQ + i] = wq[i * KM + k];
    }
  } else {
    const __half* Gh = (const __half*)(kb + ku.off_G) + (size_t)h * ku.rT * ku.rd;
    for (int x = tid; x < NQ * Kk; x += ATT_CHUNK) {
      const int i = x / Kk, k = x % Kk;
      float s = 0.f;
      for (int j = 0; j < ku.rd; ++j) s = fmaf(__half2float(Gh[k * ku.rd + j]), wq[i * KM + j], s);
      cq[k * NQ + i] = s;
    }
  }
  if (ku.b > 0) {
    const unsigned char* sb = (const unsigned char*)kb + 88;
    const float rs = rsqrtf((float)D);
    for (int i = w; i < NQ; i += ATT_WARPS) {
      float v[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const int d = lane * EPT + e;
        v[e] = (((sb[d >> 3] >> (d & 7)) & 1) ? -1.f : 1.f) * vq[i * D + d];
      }
      fwht_row<EPT>(v, lane);
#pragma unroll
      for (int e = 0; e < EPT; ++e) vt[(lane * EPT + e) * NQ + i] = v[e] * rs;
    }
  }
  __syncthreads();

  // ---- phase 1: one thread per token, the scores of every query
  {
    const int t = t0 + tid;
    float acc[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) acc[i] = 0.f;
    if (t < T) {
      const __half* R = kfT ? (const __half*)(kb + ku.off_G) + ((size_t)h * T + t) * ku.rd
                            : (const __half*)(kb + ku.off_UT) + (size_t)t * ku.rT;
      if ((Kk & 1) == 0) {
        const __half2* R2 = reinterpret_cast<const __half2*>(R);
        for (int k2 = 0; k2 < Kk / 2; ++k2) {
          const float2 r = __half22float2(R2[k2]);
#pragma unroll
          for (int i = 0; i < NQ; ++i)
            acc[i] = fmaf(r.y, cq[(2 * k2 + 1) * NQ + i], fmaf(r.x, cq[2 * k2 * NQ + i], acc[i]));
        }
      } else {
        for (int k = 0; k < Kk; ++k) {
          const float r = __half2float(R[k]);
#pragma unroll
          for (int i = 0; i < NQ; ++i) acc[i] = fmaf(r, cq[k * NQ + i], acc[i]);
        }
      }
      if (ku.b > 0) {
        const size_t row = (size_t)h * T + t;
        const float s = __half2float(((const __half*)(kb + ku.off_scale))[row]);
        float r[NQ];
        const uint32_t* cw = (const uint32_t*)(kb + ku.off_codes) + row * (size_t)(D * ku.b / 32);
        if (ku.b == 2) res_dots<D, NQ, 2>(cw, vt, r);
        else if (ku.b == 4) res_dots<D, NQ, 4>(cw, vt, r);
        else res_dots<D, NQ, 8>(cw, vt, r);
#pragma unroll
        for (int i = 0; i < NQ; ++i) acc[i] = fmaf(s, r[i], acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < NQ; ++i) sc[tid * NQ + i] = (t < T) ? a.scale * acc[i] : -INFINITY;
  }
  __syncthreads();

  // ---- phase 2: probabilities against the chunk's max (a warp per query)
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
    if (lane == 0) { stat[i] = m; stat[NQ + i] = l; }
  }
  __syncthreads();

  // ---- phase 3: cv and z over this warp's 32 tokens
  const bool vfT = (vu.rT == T);
  const int Kv = vfT ? vu.rd : vu.rT;
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
    const __half* sv = (const __half*)(vb + vu.off_scale);
    const uint32_t* cvw = (const uint32_t*)(vb + vu.off_codes);
    const size_t rw = (size_t)D * vu.b / 32;
    for (int j = 0; j < 32; ++j) {
      const int x = w * 32 + j, t = t0 + x;
      if (t >= T) break;
      float p[NQ];
#pragma unroll
      for (int i = 0; i < NQ; ++i) p[i] = sc[x * NQ + i];
      const __half* R = vfT ? (const __half*)(vb + vu.off_G) + ((size_t)h * T + t) * vu.rd
                            : (const __half*)(vb + vu.off_UT) + (size_t)t * vu.rT;
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
        const size_t row = (size_t)h * T + t;
        const float s = __half2float(sv[row]);
        float ps[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) ps[i] = p[i] * s;
        if (vu.b == 2) res_accum<EPT, NQ, 2>(cvw + row * rw, lane, ps, z);
        else if (vu.b == 4) res_accum<EPT, NQ, 4>(cvw + row * rw, lane, ps, z);
        else res_accum<EPT, NQ, 8>(cvw + row * rw, lane, ps, z);
      }
    }
  }
  float* rw_ = red + (size_t)w * NQ * (D + KM);
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) rw_[i * (D + KM) + lane * EPT + e] = z[i][e];
#pragma unroll
    for (int jj = 0; jj < KPL; ++jj) rw_[i * (D + KM) + D + lane + 32 * jj] = cv[i][jj];
  }
  __syncthreads();

  // ---- the chunk's record: max, sum, z, cv (summed over the warps)
  float* rec = a.part + (((size_t)g * H + h) * a.nch + chunk) * rec_floats(nq, D);
  for (int i = tid; i < nq; i += ATT_CHUNK) {
    rec[i] = stat[i];
    rec[nq + i] = stat[NQ + i];
  }
  for (int x = tid; x < nq * (D + KM); x += ATT_CHUNK) {
    const int i = x / (D + KM), c = x % (D + KM);
    if (c >= D + Kv) continue;
    float s = 0.f;
#pragma unroll
    for (int ww = 0; ww < ATT_WARPS; ++ww) s += red[(size_t)ww * NQ * (D + KM) + i * (D + KM) + c];
    rec[2 * nq + (size_t)i * (D + KM) + c] = s;
  }
}

// Merge the chunks of one (head, group) and map back to feature space.
template <int EPT, int NQ>
__global__ void __launch_bounds__(128) attend_merge_kernel(AttArgs a) {
  constexpr int D = 32 * EPT;
  constexpr int KM = JOLT_ATTN_MAX_RANK;
  __shared__ float zf[NQ][D], cf[NQ][KM], ef[NQ][KM > D ? KM : D];
  __shared__ float Mx[NQ], Lx[NQ];
  const int h = blockIdx.x, gl = blockIdx.y, g = a.g0 + gl;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int T = a.T, H = a.H, nq = a.nq, nch = a.nch;
  const AttUnit vu = a.v[gl];
  const char* vb = a.blob + (unsigned long long)(2 * g + 1) * a.stride;
  const bool vfT = (vu.rT == T), vfD = (vu.rd == D);
  const int Kv = vfT ? vu.rd : vu.rT;
  const size_t rf = rec_floats(nq, D);
  const float* base = a.part + ((size_t)g * H + h) * nch * rf;

  // global max and sum of every query
  for (int i = w; i < nq; i += 4) {
    float m = -INFINITY;
    for (int c = lane; c < nch; c += 32) m = fmaxf(m, base[c * rf + i]);
    m = warp_max(m);
    float l = 0.f;
    for (int c = lane; c < nch; c += 32) l += expf(base[c * rf + i] - m) * base[c * rf + nq + i];
    l = warp_sum(l);
    if (lane == 0) { Mx[i] = m; Lx[i] = l; }
  }
  __syncthreads();
  // z and cv: chunk records weighted by exp(m_c - M)
  for (int x = tid; x < nq * (D + KM); x += 128) {
    const int i = x / (D + KM), c = x % (D + KM);
    if (c >= D + Kv) continue;
    float s = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
      const float* r = base + ch * rf;
      s = fmaf(expf(r[i] - Mx[i]), r[2 * nq + (size_t)i * (D + KM) + c], s);
    }
    if (c < D) zf[i][c] = s;
    else cf[i][c - D] = s;
  }
  __syncthreads();
  // back-projection, stage 1: e = G[h]^T cv (r_T < T) or cv itself (r_T = T)
  if (vfT) {
    for (int x = tid; x < nq * vu.rd; x += 128) ef[x / vu.rd][x % vu.rd] = cf[x / vu.rd][x % vu.rd];
  } else {
    const __half* Gh = (const __half*)(vb + vu.off_G) + (size_t)h * vu.rT * vu.rd;
    for (int x = tid; x < nq * vu.rd; x += 128) {
      const int i = x / vu.rd, j = x % vu.rd;
      float s = 0.f;
      for (int k = 0; k < vu.rT; ++k) s = fmaf(__half2float(Gh[k * vu.rd + j]), cf[i][k], s);
      ef[i][j] = s;
    }
  }
  __syncthreads();
  // stage 2 (U_d e) plus the inverse rotation of z, a warp per query
  const __half* Ud = (const __half*)(vb + vu.off_Ud);
  const unsigned char* sb = (const unsigned char*)vb + 88;
  const float rs = rsqrtf((float)D);
  for (int i = w; i < nq; i += 4) {
    float v[EPT];
    if (vu.b > 0) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = zf[i][lane * EPT + e];
      fwht_row<EPT>(v, lane);
    }
    const float inv = 1.f / Lx[i];
    float* o = a.out + (((size_t)g * H + h) * nq + i) * D;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int d = lane * EPT + e;
      float lo;
      if (vfD) {
        lo = ef[i][d];
      } else {
        lo = 0.f;
        for (int j = 0; j < vu.rd; ++j) lo = fmaf(__half2float(Ud[d * vu.rd + j]), ef[i][j], lo);
      }
      float res = 0.f;
      if (vu.b > 0) res = (((sb[d >> 3] >> (d & 7)) & 1) ? -1.f : 1.f) * v[e] * rs;
      o[d] = (lo + res) * inv;
    }
  }
}

template <int EPT, int NQ>
jolt_status launch_attend(const AttArgs& a, int ng, cudaStream_t st) {
  constexpr int D = 32 * EPT;
  constexpr int KM = JOLT_ATTN_MAX_RANK;
  const size_t smem = sizeof(float) * (NQ * D + NQ * KM + KM * NQ + D * NQ + ATT_CHUNK * NQ +
                                       ATT_WARPS * NQ * (D + KM) + 2 * NQ);
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(attend_chunk_kernel<EPT, NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  attend_chunk_kernel<EPT, NQ><<<dim3(a.nch, a.H, ng), ATT_CHUNK, smem, st>>>(a);
  JOLT_LAUNCH_CHECK();
  attend_merge_kernel<EPT, NQ><<<dim3(a.H, ng), 128, 0, st>>>(a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

template <int EPT>
jolt_status launch_attend_nq(const AttArgs& a, int ng, cudaStream_t st) {
  if (a.nq <= 1) return launch_attend<EPT, 1>(a, ng, st);
  if (a.nq <= 2) return launch_attend<EPT, 2>(a, ng, st);
  if (a.nq <= 4) return launch_attend<EPT, 4>(a, ng, st);
  return launch_attend<EPT, 8>(a, ng, st);
}

AttUnit att_unit(const jolt_blob_desc& d) {
  AttUnit u;
  u.rT = d.rT; u.rd = d.rd; u.b = d.b; u.pad = 0;
  u.off_UT = d.off_UT; u.off_Ud = d.off_Ud; u.off_G = d.off_G;
  u.off_scale = d.off_scale; u.off_codes = d.off_codes;
  return u;
}

}  // namespace

size_t attend_chunks(int T) { return (size_t)((T + ATT_CHUNK - 1) / ATT_CHUNK); }

size_t attend_ws_bytes(int n_groups, int H, int T, int D, int nq) {
  return (size_t)n_groups * H * attend_chunks(T) * nq * (2 + D + JOLT_ATTN_MAX_RANK) *
         sizeof(float);
}

jolt_status attend_run(int n_groups, const jolt_blob_desc* desc, const char* blob,
                       size_t stride, const float* q, int nq, float scale, float* part,
                       float* out, cudaStream_t st) {
  const int H = desc[0].H, T = desc[0].T, D = desc[0].D;
  for (int g0 = 0; g0 < n_groups; g0 += ATT_MAX_G) {
    const int ng = (n_groups - g0) < ATT_MAX_G ? (n_groups - g0) : ATT_MAX_G;
    AttArgs a;
    memset(&a, 0, sizeof(a));
    a.H = H; a.T = T; a.nq = nq; a.nch = (int)attend_chunks(T);
    a.scale = scale; a.blob = blob; a.stride = stride; a.q = q; a.part = part; a.out = out;
    a.g0 = g0;
    for (int i = 0; i < ng; ++i) {
      a.k[i] = att_unit(desc[2 * (g0 + i)]);
      a.v[i] = att_unit(desc[2 * (g0 + i) + 1]);
    }
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
