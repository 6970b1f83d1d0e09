// Serialization of the chosen candidate and the decoder.
//
// ["Rotated Tucker residual for outlier-resistant KV quantization",
//  Implementation notes: store the block scale s and the integer codes
//  clip(round(Y/s), ...); decode by multiplying codes by s, applying the
//  inverse orthogonal transform and adding X~; for b = 0 return X~ only.
//  "Joint Tucker-rank and residual-bit KV allocator", Implementation notes:
//  actual storage includes factors, core, codes, scales, transform metadata
//  and alignment padding.]
//
// Blob (little-endian): 256-byte header
//   0: u32 magic "JOLT", u32 version, i32 H, T, D, r_T, r_d, b, block, u32 flags
//  40: u64 offsets of U_T, U_d, G, scales, codes, and the total size
//  88: sign bits of diag(sigma), bit i set when sigma_i = -1, LSB first
// then the sections, each starting on an `align` boundary:
//   U_T fp16 [T][r_T] (absent when r_T = T), U_d fp16 [D][r_d] (absent when
//   r_d = D), G fp16 [H][r_T][r_d] (fp16(X) when both modes are whole),
//   scales fp16 [H*T] (one per row block), codes b-bit offset-binary
//   u = q + 2^(b-1), element k in bits [k b, (k+1) b) of the byte stream.
#include "jolt_internal.cuh"

#include <string.h>

namespace jolt {

namespace {

constexpr uint32_t MAGIC = 0x544C4F4Au;  // "JOLT"
constexpr uint32_t VERSION = 1;
constexpr int CD_WARPS = 8, CD_ROWS = 8, CD_TILE = 64, CD_THREADS = 256;

struct HeaderArgs {
  unsigned char fixed[88];
  int D;
};

struct EncArgs {
  const void* X;
  const int8_t* signs;
  int H, T, D, dtype;
  int b, mode, K;     // mode 0/1: X~ = K B chain; 2: whole modes, X~ = fp16(X)
  const __half* Kg;   // chain coefficients K[t][k] at Kg + h*k_hs + t*k_ld + k
  long long k_hs, k_ld;
  const __half* B16;  // fp16 chain rows B[k][d] at B16 + h*b_hs + k*b_ks + d*b_ds, or
  long long b_hs, b_ks, b_ds;
  const float* Bhi;   // double-float rows (Bhi + Blo)[h][k][d], row stride D
  const float* Blo;
  float rs_hi, rs_lo;  // 1/sqrt(D) as a double-float
  char* blob;
  unsigned long long off_scale, off_codes;
  long long row_ld, row_off;   // token t of head h is row h * row_ld + row_off + t of the blob
};

// Error-free transformations (Knuth TwoSum; TwoProduct through the fused
// multiply-add).  Double-float values are unevaluated sums hi + lo.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Walsh-Hadamard transform of a warp row of double-floats (element
// lane * EPT + e), each butterfly a TwoSum with the low parts carried along.
template <int EPT>
__device__ __forceinline__ void fwht_row_df(float (&hi)[EPT], float (&lo)[EPT], int lane) {
#pragma unroll
  for (int h = 1; h < EPT; h <<= 1)
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if (!(e & h)) {
        float s, es, d, ed;
        two_sum(hi[e], hi[e + h], s, es);
        two_sum(hi[e], -hi[e + h], d, ed);
        const float l0 = lo[e], l1 = lo[e + h];
        hi[e] = s; lo[e] = (l0 + l1) + es;
        hi[e + h] = d; lo[e + h] = (l0 - l1) + ed;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const float oh = __shfl_xor_sync(0xffffffffu, hi[e], m);
      const float ol = __shfl_xor_sync(0xffffffffu, lo[e], m);
      float s, es;
      if (lane & m) {
        two_sum(oh, -hi[e], s, es);
        lo[e] = (ol - lo[e]) + es;
      } else {
        two_sum(hi[e], oh, s, es);
        lo[e] = (lo[e] + ol) + es;
      }
      hi[e] = s;
    }
}

// fp16 rounding (to nearest, ties to even) of the value zh + zl >= 0, where
// zh is fp32-rounded: only when zh sits exactly on the midpoint of two fp16
// neighbours does the low part decide.
__device__ __forceinline__ float round_f16_df(float zh, float zl) {
  const __half h = __float2half_rn(zh);
  const float hf = __half2float(h);
  const float d = zh - hf;
  if (d == 0.f || zl == 0.f) return hf;
  const unsigned short hb = __half_as_ushort(h);
  const __half nb = __ushort_as_half((unsigned short)(d > 0.f ? hb + 1 : hb - 1));
  const float nf = __half2float(nb);
  if (zh == 0.5f * (hf + nf) && (d > 0.f) == (zl > 0.f)) return nf;
  return hf;
}

// Codes of one residual row: R = X - K B in double-float (the chain
// products are exact or TwoProduct-split), y = Q R by a double-float
// Walsh-Hadamard transform, then the block scale and the codes decided on
// the double-float y so that they agree with a correctly rounded evaluation
// except where y sits within ~2^-44 |y| of a rounding boundary.
// ["Rotated Tucker residual for outlier-resistant KV quantization",
//  Formulas: Y = Q R, s = max|y| / (2^(b-1) - 1) in fp16, codes = round(y / s)
//  clipped to the b-bit range.]
constexpr int ENC_MAX_UNITS = 16;
struct EncBatch {
  EncArgs u[ENC_MAX_UNITS];
};

// The block scale and codes of one rotated residual row from its exact
// value: the residual of the row in double-float (the chain products are
// exact or TwoProduct-split), rotated by a double-float Walsh-Hadamard
// transform, and every decision taken on the double-float y, so that it
// agrees with a correctly rounded evaluation except within ~2^-44 |y| of a
// boundary.  x: this lane's EPT inputs of the row (x - fp16(x) for the
// whole modes); the chain coefficients of the row are Ks[k * CD_TILE + rr].
template <int EPT>
__device__ __forceinline__ void exact_row(const EncArgs& a, const float (&x)[EPT], const float* Ks,
                                          int rr, const float* Bsh, const float* Bsl,
                                          const float (&sg)[EPT], float qmax, int lane,
                                          float (&q)[EPT], float& s_out) {
  constexpr int D = 32 * EPT;
  float yh[EPT], yl[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    yh[e] = x[e];
    yl[e] = 0.f;
  }
  if (a.mode != 2) {
    for (int k = 0; k < a.K; ++k) {
      const float c = Ks[k * CD_TILE + rr];
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const float bh = Bsh[k * D + lane * EPT + e], bl = Bsl[k * D + lane * EPT + e];
        const float p = c * bh;
        const float pe = fmaf(c, bh, -p);  // c bh = p + pe exactly
        float sm, es;
        two_sum(yh[e], -p, sm, es);
        yh[e] = sm;
        yl[e] = fmaf(-c, bl, yl[e] + (es - pe));
      }
    }
  }
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    yh[e] *= sg[e];
    yl[e] *= sg[e];
  }
  fwht_row_df<EPT>(yh, yl, lane);
  // times 1/sqrt(D), renormalised so that yh is the fp32 rounding of y
  float mh = 0.f, ml = 0.f;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const float p = yh[e] * a.rs_hi;
    const float l = fmaf(yh[e], a.rs_hi, -p) + fmaf(yh[e], a.rs_lo, yl[e] * a.rs_hi);
    yh[e] = p + l;
    yl[e] = l - (yh[e] - p);
    const float ay = fabsf(yh[e]), aly = yh[e] < 0.f ? -yl[e] : yl[e];
    if (ay > mh || (ay == mh && aly > ml)) { mh = ay; ml = aly; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, mh, o);
    const float ol = __shfl_xor_sync(0xffffffffu, ml, o);
    if (oh > mh || (oh == mh && ol > ml)) { mh = oh; ml = ol; }
  }
  // s = fp16(max|y| / qmax) from the double-float max
  const float z0 = __fdiv_rn(mh, qmax);
  const float z1 = __fdiv_rn(fmaf(-z0, qmax, mh) + ml, qmax);
  const float zh = z0 + z1;  // renormalised: zh is the fp32 rounding of the quotient
  const float s = round_f16_df(zh, z1 - (zh - z0));
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    float qq = 0.f;
    if (s > 0.f) {
      qq = rintf(__fdiv_rn(yh[e], s));
      // the boundaries (q +- 1/2) s are exact in fp32; their side is the
      // sign of y - (q +- 1/2) s, taken on the double-float y
      const float up = fmaf(-(qq + 0.5f), s, yh[e]) + yl[e];
      const float dn = fmaf(-(qq - 0.5f), s, yh[e]) + yl[e];
      if (up > 0.f || (up == 0.f && fmodf(qq, 2.f) != 0.f)) qq += 1.f;
      else if (dn < 0.f || (dn == 0.f && fmodf(qq, 2.f) != 0.f)) qq -= 1.f;
    }
    q[e] = qq;
  }
  s_out = s;
}

// Codes of one tile of rows (64 tokens of one head; a warp holds 8 rows, a
// lane EPT elements of each).
// ["Rotated Tucker residual for outlier-resistant KV quantization",
//  Formulas: Y = Q R, s = max|y| / (2^(b-1) - 1) in fp16, codes = round(y / s)
//  clipped to the b-bit range.]
// Each row is first formed in fp32 with an a-posteriori bound on its
// rounding error: the chain R = X - K B by fused multiply-adds (each rounding
// at most u |partial residual|, u = 2^-24, the partials' magnitudes summed
// per element), the Walsh-Hadamard transform (at most 8 u ||v||_1 / sqrt(D)
// for its seven levels and the scaling).  Where the bound proves that the
// fp32 row decides the fp16 scale and every code the same way as the exact
// value, those decisions are taken; any other row (a value within the bound
// of a rounding boundary) is recomputed by exact_row.  The codes are
// therefore those of the exact evaluation.
template <typename TX, int EPT>
__global__ void __launch_bounds__(CD_THREADS, 2) encode_codes_kernel(const __grid_constant__ EncBatch eb) {
  const EncArgs& a = eb.u[blockIdx.z];
  constexpr int D = 32 * EPT;
  constexpr float U = 5.9604645e-08f;          // 2^-24
  extern __shared__ __align__(16) float dsm[];
  float* Ks = dsm;                       // [64][CD_TILE]
  float* Bsh = Ks + 64 * CD_TILE;        // [64][D]
  float* Bsl = Bsh + 64 * D;             // [64][D]
  unsigned char (*codes)[D] = reinterpret_cast<unsigned char (*)[D]>(Bsl + 64 * D);  // [warps][D]
  const int h = blockIdx.y, t0 = blockIdx.x * CD_TILE;
  const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
  const TX* Xh = (const TX*)a.X + (long long)h * a.T * D;
  float rv[CD_ROWS][EPT], sv[CD_ROWS][EPT];   // fp32 residuals, sums of |partial residuals|
#pragma unroll
  for (int r = 0; r < CD_ROWS; ++r) {
    const int t = t0 + w * CD_ROWS + r;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const float x = (t < a.T) ? to_f32(Xh[(long long)t * D + lane * EPT + e]) : 0.f;
      rv[r][e] = a.mode == 2 ? x - round_f16(x) : x;  // exact
      sv[r][e] = 0.f;
    }
  }
  // double-float chain rows (B = hi + lo): the fp32 chain takes hi only, its
  // error |c lo| <= 2^-24 |c hi| per term added to the bound with |c hi|
  const bool lo_part = (a.mode != 2 && a.K > 0 && a.B16 == nullptr);
  if (a.mode != 2 && a.K > 0) {
    for (int i = threadIdx.x; i < CD_TILE * a.K; i += CD_THREADS) {
      const int row = i / a.K, k = i % a.K;
      const int t = t0 + row;
      Ks[k * CD_TILE + row] = (t < a.T) ? __half2float(a.Kg[h * a.k_hs + (long long)t * a.k_ld + k]) : 0.f;
    }
    if (a.B16) {
      const __half* Bh = a.B16 + h * a.b_hs;
      for (int i = threadIdx.x; i < a.K * D; i += CD_THREADS) {
        const int k = i / D, d = i % D;
        Bsh[i] = __half2float(Bh[k * a.b_ks + d * a.b_ds]);
        Bsl[i] = 0.f;
      }
    } else {
      const float* Bh = a.Bhi + (long long)h * a.b_hs;
      const float* Bl = a.Blo + (long long)h * a.b_hs;
      for (int i = threadIdx.x; i < a.K * D; i += CD_THREADS) {
        Bsh[i] = Bh[i];
        Bsl[i] = Bl[i];
      }
    }
    __syncthreads();
    for (int k = 0; k < a.K; ++k) {
      const float* kk = Ks + k * CD_TILE + w * CD_ROWS;
      float bh[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) bh[e] = Bsh[k * D + lane * EPT + e];
#pragma unroll
      for (int r = 0; r < CD_ROWS; ++r) {
        const float c = kk[r];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          const float v = fmaf(-c, bh[e], rv[r][e]);
          rv[r][e] = v;
          sv[r][e] += fabsf(v);
          if (lo_part) sv[r][e] = fmaf(fabsf(c), fabsf(bh[e]), sv[r][e]);
        }
      }
    }
  }
  float sg[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) sg[e] = (float)a.signs[lane * EPT + e];
  const int b = a.b;
  const float qmax = (float)((1 << (b - 1)) - 1);
  const int qoff = 1 << (b - 1);
  const int nbytes = D * b / 8;
  const float rs = a.rs_hi;
  // one row at a time, not unrolled (the row's values are picked out of the
  // register arrays by static selects, which keeps the code small)
#pragma unroll 1
  for (int r = 0; r < CD_ROWS; ++r) {
    const int t = t0 + w * CD_ROWS + r;
    float y[EPT], l1s = 0.f, l1v = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      float vh = rv[0][e], vs = sv[0][e];
#pragma unroll
      for (int rr = 1; rr < CD_ROWS; ++rr)
        if (rr == r) { vh = rv[rr][e]; vs = sv[rr][e]; }
      y[e] = vh * sg[e];
      l1v += fabsf(vh);
      l1s += vs;
    }
    fwht_row<EPT>(y, lane);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      y[e] *= rs;
      m = fmaxf(m, fabsf(y[e]));
    }
    m = warp_max(m);
    l1s = warp_sum(l1s);
    l1v = warp_sum(l1v);
    // bound on |y - exact y| for every element of the row: the chain's
    // roundings and dropped low parts (l1s u), the transform's seven levels and the scaling
    // (8 u l1v), over sqrt(D); each element adds 2 u |y| (the product by the
    // fp32 1/sqrt(D) and its rounding).  The sums themselves are rounded:
    // 1% of slack covers them.
    const float E = 1.01f * U * (l1s + 8.f * l1v) * rs;
    const float Em = E + 2.f * U * m;
    // the scale: certain when no fp16 rounding boundary lies within the
    // bound of max|y| / qmax
    bool sure = true;
    float s = 0.f;
    {
      const float z = __fdiv_rn(m, qmax);
      const float dz = 1.01f * (Em / qmax + U * z);
      const __half hz = __float2half_rn(z);
      const float hf = __half2float(hz);
      const unsigned short hb = __half_as_ushort(hz);
      // neighbours of hz among the fp16 values (z >= 0)
      const float up = __half2float(__ushort_as_half((unsigned short)(hb + 1)));
      const float dn = hb > 0 ? __half2float(__ushort_as_half((unsigned short)(hb - 1))) : -hf;
      const float mid_hi = 0.5f * (hf + up), mid_lo = 0.5f * (hf + dn);
      if (!(z - dz > mid_lo && z + dz < mid_hi)) sure = false;
      if (m == 0.f && E > 0.f) sure = false;
      s = hf;
    }
    float q[EPT];
    // the quotient by the reciprocal: a code it rounds the wrong way lies
    // within a few ulps of a tie, where the check below fails anyway
    const float inv_s = s > 0.f ? __fdiv_rn(1.f, s) : 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      float qq = 0.f;
      if (s > 0.f) {
        qq = rintf(y[e] * inv_s);
        // the exact y must lie strictly between (q - 1/2) s and (q + 1/2) s
        const float Ee = 1.01f * (E + 2.f * U * fabsf(y[e]));
        const float up = fmaf(-(qq + 0.5f), s, y[e]);
        const float dn = fmaf(-(qq - 0.5f), s, y[e]);
        if (!(up + Ee + U * fabsf(up) < 0.f && dn - Ee - U * fabsf(dn) > 0.f)) sure = false;
      }
      q[e] = qq;
    }
    if (__any_sync(0xffffffffu, !sure)) {
      // recompute the row from its exact value
      float xr[EPT];
      const bool okr = t < a.T;
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const float x = okr ? to_f32(Xh[(long long)t * D + lane * EPT + e]) : 0.f;
        xr[e] = a.mode == 2 ? x - round_f16(x) : x;
      }
      exact_row<EPT>(a, xr, Ks, w * CD_ROWS + r, Bsh, Bsl, sg, qmax, lane, q, s);
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const float qq = fminf(fmaxf(q[e], -(float)qoff), (float)(qoff - 1));
      codes[w][lane * EPT + e] = (unsigned char)((int)qq + qoff);
    }
    __syncwarp();
    if (t < a.T) {
      const long long row = (long long)h * a.row_ld + a.row_off + t;
      unsigned char* cb = (unsigned char*)a.blob + a.off_codes + row * nbytes;
      const int per = 8 / b;
      for (int j = lane; j < nbytes; j += 32) {
        unsigned v = 0;
        for (int i = 0; i < per; ++i) v |= (unsigned)codes[w][j * per + i] << (i * b);
        cb[j] = (unsigned char)v;
      }
      if (lane == 0) ((__half*)(a.blob + a.off_scale))[row] = __float2half_rn(s);
    }
    __syncwarp();
  }
}

// Serialization of the header and the factor sections of a batch of units in
// one launch (grid y = unit): each unit lists up to three copies
// dst[a][b][c] = fp16(src[a*sa + b*sb + c]) (a < A, b < B, c < C) of a source
// in fp16, bf16 or fp32, and its 256-byte header.
struct CopyJob {
  const void* src;
  __half* dst;
  long long sa, sb;
  int A, B, C, type;   // type: 0 fp16, 1 bf16, 2 fp32
};
struct SecUnit {
  CopyJob job[3];
  int njobs;
  HeaderArgs ha;
  const int8_t* signs;
  char* blob;
};
struct SecBatch {
  SecUnit u[ENC_MAX_UNITS];
};

__global__ void sections_kernel(const __grid_constant__ SecBatch sb) {
  const SecUnit& su = sb.u[blockIdx.y];
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < 88; i += blockDim.x) su.blob[i] = (char)su.ha.fixed[i];
    for (int i = threadIdx.x; i < (su.ha.D + 7) / 8; i += blockDim.x) {
      unsigned char v = 0;
      for (int k = 0; k < 8; ++k) {
        const int d = i * 8 + k;
        if (d < su.ha.D && su.signs[d] < 0) v |= (unsigned char)(1u << k);
      }
      su.blob[88 + i] = (char)v;
    }
  }
  for (int j = 0; j < su.njobs; ++j) {
    const CopyJob& cj = su.job[j];
    const long long n = (long long)cj.A * cj.B * cj.C;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
      const int c = (int)(e % cj.C);
      const long long ab = e / cj.C;
      const int b = (int)(ab % cj.B), aa = (int)(ab / cj.B);
      const long long si = aa * cj.sa + b * cj.sb + c;
      float v;
      if (cj.type == 0) v = __half2float(((const __half*)cj.src)[si]);
      else if (cj.type == 1) v = __bfloat162float(((const __nv_bfloat16*)cj.src)[si]);
      else v = ((const float*)cj.src)[si];
      cj.dst[e] = __float2half_rn(v);
    }
  }
}

// Unrotated chain rows of a truncated core for a batch of units (grid z =
// unit; an entry with rT = 0 is skipped): B[h][k][:] = G16[h][k][:] U_d16^T,
// accumulated in double-float (fp16 x fp16 products are exact in fp32).
struct RowsUnit {
  const __half* G;
  long long g_hs;
  const __half* Ud;
  int ldu, rT, rd;
  float* Bhi;
  float* Blo;
};
struct RowsBatch {
  RowsUnit u[ENC_MAX_UNITS];
  int D;
};
__global__ void enc_rows_batch_kernel(const __grid_constant__ RowsBatch rb) {
  const RowsUnit& r = rb.u[blockIdx.z];
  const int D = rb.D;
  if (r.rT == 0) return;
  const int h = blockIdx.y;
  const __half* Gh = r.G + h * r.g_hs;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < r.rT * D; i += gridDim.x * blockDim.x) {
    const int k = i / D, d = i % D;
    float sh = 0.f, sl = 0.f;
    for (int j = 0; j < r.rd; ++j) {
      const float p = __half2float(Gh[k * r.rd + j]) * __half2float(r.Ud[(long long)d * r.ldu + j]);
      float s2, e;
      two_sum(sh, p, s2, e);
      sh = s2;
      sl += e;
    }
    const float hi = sh + sl;
    r.Bhi[(long long)h * r.rT * D + i] = hi;
    r.Blo[(long long)h * r.rT * D + i] = sl - (hi - sh);
  }
}

struct DecUnit {
  int rT, rd, b, pad;
  unsigned long long off_UT, off_Ud, off_G, off_scale, off_codes;
};
constexpr int DEC_MAX_UNITS = 32;
struct DecArgs {
  int H, T, D, out_dtype;
  const char* blob;
  unsigned long long stride;
  void* xhat;
  int u0;
  DecUnit un[DEC_MAX_UNITS];
};

// X^ = X~ + Q^T (s * codes), one tile of 64 rows of one head per CTA.
template <int EPT>
__global__ void __launch_bounds__(CD_THREADS) decode_kernel(DecArgs a) {
  constexpr int D = 32 * EPT;
  extern __shared__ __align__(16) float dsm[];
  float* Ks = dsm;                       // [64][CD_TILE]
  float* Bs = Ks + 64 * CD_TILE;         // [64][D]
  const int uz = blockIdx.z, h = blockIdx.y, t0 = blockIdx.x * CD_TILE;
  const int u = a.u0 + uz;
  const DecUnit du = a.un[uz];
  const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
  const char* blob = a.blob + (unsigned long long)u * a.stride;
  const int T = a.T, H = a.H;
  const int rT = du.rT, rd = du.rd, b = du.b;
  const bool fullT = (rT == T), fullD = (rd == D);
  const __half* G = (const __half*)(blob + du.off_G);
  float acc[CD_ROWS][EPT];
  int K = 0;
  if (fullT && fullD) {
#pragma unroll
    for (int r = 0; r < CD_ROWS; ++r) {
      const int t = t0 + w * CD_ROWS + r;
#pragma unroll
      for (int e = 0; e < EPT; ++e)
        acc[r][e] = (t < T) ? __half2float(G[((long long)h * T + t) * D + lane * EPT + e]) : 0.f;
    }
  } else {
    if (fullT) {
      // X~[t] = G[h][t][:rd] U_d^T
      K = rd;
      const __half* Ud = (const __half*)(blob + du.off_Ud);
      for (int i = threadIdx.x; i < CD_TILE * K; i += CD_THREADS) {
        const int row = i / K, j = i % K, t = t0 + row;
        Ks[j * CD_TILE + row] = (t < T) ? __half2float(G[((long long)h * T + t) * rd + j]) : 0.f;
      }
      for (int i = threadIdx.x; i < K * D; i += CD_THREADS) {
        const int j = i / D, d = i % D;
        Bs[i] = __half2float(Ud[(long long)d * rd + j]);
      }
    } else {
      // X~[t] = U_T[t] P_h, P_h = G[h] U_d^T (rT x D)
      K = rT;
      const __half* UT = (const __half*)(blob + du.off_UT);
      for (int i = threadIdx.x; i < CD_TILE * K; i += CD_THREADS) {
        const int row = i / K, k = i % K, t = t0 + row;
        Ks[k * CD_TILE + row] = (t < T) ? __half2float(UT[(long long)t * rT + k]) : 0.f;
      }
      const __half* Gh = G + (long long)h * rT * rd;
      if (fullD) {
        for (int i = threadIdx.x; i < K * D; i += CD_THREADS) Bs[i] = __half2float(Gh[i]);
      } else {
        const __half* Ud = (const __half*)(blob + du.off_Ud);
        for (int i = threadIdx.x; i < K * D; i += CD_THREADS) {
          const int k = i / D, d = i % D;
          float v = 0.f;
          for (int j = 0; j < rd; ++j)
            v = fmaf(__half2float(Gh[k * rd + j]), __half2float(Ud[(long long)d * rd + j]), v);
          Bs[i] = v;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < CD_ROWS; ++r)
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[r][e] = 0.f;
    for (int k = 0; k < K; ++k) {
      const float* kk = Ks + k * CD_TILE + w * CD_ROWS;
      float bv[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) bv[e] = Bs[k * D + lane * EPT + e];
#pragma unroll
      for (int r = 0; r < CD_ROWS; ++r)
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[r][e] = fmaf(kk[r], bv[e], acc[r][e]);
    }
  }
  if (b > 0) {
    const unsigned char* sbits = (const unsigned char*)blob + 88;
    float sg[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int d = lane * EPT + e;
      sg[e] = ((sbits[d >> 3] >> (d & 7)) & 1) ? -1.f : 1.f;
    }
    const float rs = rsqrtf((float)D);
    const unsigned char* cb = (const unsigned char*)blob + du.off_codes;
    const __half* sc = (const __half*)(blob + du.off_scale);
    const int qoff = 1 << (b - 1), mask = (1 << b) - 1;
#pragma unroll
    for (int r = 0; r < CD_ROWS; ++r) {
      const int t = t0 + w * CD_ROWS + r;
      const bool ok = t < T;
      const long long row = (long long)h * T + (ok ? t : 0);
      float q[EPT];
      const long long bit0 = (row * D + lane * EPT) * b;
      if (((EPT * b) & 7) == 0) {
        // this lane's EPT codes are EPT * b (8, 16 or 32) contiguous bits
        // starting on a byte boundary: one load
        unsigned word = 0;
        if (ok) {
          const unsigned char* p0 = cb + (bit0 >> 3);
          const int nbytes = (EPT * b) >> 3;
          if (nbytes == 4) word = *reinterpret_cast<const unsigned*>(p0);
          else if (nbytes == 2) word = *reinterpret_cast<const unsigned short*>(p0);
          else word = *p0;
        }
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          const int uu = ok ? (int)((word >> (e * b)) & mask) : qoff;
          q[e] = (float)(uu - qoff);
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          const long long bit = bit0 + (long long)e * b;
          const int uu = ok ? ((cb[bit >> 3] >> (bit & 7)) & mask) : qoff;
          q[e] = (float)(uu - qoff);
        }
      }
      fwht_row<EPT>(q, lane);
      const float cs = ok ? __half2float(sc[row]) * rs : 0.f;
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[r][e] = fmaf(sg[e] * cs, q[e], acc[r][e]);
    }
  }
#pragma unroll
  for (int r = 0; r < CD_ROWS; ++r) {
    const int t = t0 + w * CD_ROWS + r;
    if (t >= T) continue;
    const long long o = (((long long)u * H + h) * T + t) * D + lane * EPT;
    if (a.out_dtype == JOLT_BF16) {
      __nv_bfloat16* y = (__nv_bfloat16*)a.xhat + o;
      if constexpr (EPT == 4) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[r][0], acc[r][1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[r][2], acc[r][3]);
        uint2 pk;
        pk.x = *reinterpret_cast<unsigned*>(&p0);
        pk.y = *reinterpret_cast<unsigned*>(&p1);
        *reinterpret_cast<uint2*>(y) = pk;
      } else {
#pragma unroll
        for (int e = 0; e < EPT; ++e) y[e] = __float2bfloat16_rn(acc[r][e]);
      }
    } else {
      float* y = (float*)a.xhat + o;
#pragma unroll
      for (int e = 0; e < EPT; ++e) y[e] = acc[r][e];
    }
  }
}

template <typename TX, int EPT>
jolt_status launch_enc(dim3 grid, const EncBatch& ea, cudaStream_t st) {
  constexpr int D = 32 * EPT;
  const size_t smem = (64 * CD_TILE + 2 * 64 * D) * sizeof(float) + CD_WARPS * D;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(encode_codes_kernel<TX, EPT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  encode_codes_kernel<TX, EPT><<<grid, CD_THREADS, smem, st>>>(ea);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

template <int EPT>
jolt_status launch_dec(dim3 grid, const DecArgs& a, cudaStream_t st) {
  constexpr int D = 32 * EPT;
  const size_t smem = (64 * CD_TILE + 64 * D) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(decode_kernel<EPT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr = true;
  }
  decode_kernel<EPT><<<grid, CD_THREADS, smem, st>>>(a);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}



// ------------------------------------------------------------------ admission
// A block of tau new tokens joins an encoded unit whose candidate, factors,
// signs and bit width stay fixed.  ["Rotated Tucker residual for
// outlier-resistant KV quantization", Implementation notes: keep the Tucker
// factors, rebuild X~ for each incoming token block and code R = X - X~.]
// The stored rows of the new tokens are computed in double-float (fp16 x
// fp16 and bf16 x fp16 products are exact in fp32, the rest through
// TwoProduct) with the small normal-equation solve in f64, so that their
// fp16 rounding is the correctly rounded one except at exact ties.
constexpr int ADM_MAX_UNITS = 16;
constexpr int ADM_MAX_JOBS = 6;
constexpr int ADM_RT = 64;            // largest truncated token rank

// fp16 rounding (to nearest, ties to even) of the signed double-float zh + zl.
__device__ __forceinline__ __half round_f16_df_signed(float zh, float zl) {
  const __half h = __float2half_rn(zh);
  const float hf = __half2float(h);
  const float d = zh - hf;
  if (d == 0.f || zl == 0.f) return h;
  const unsigned short hb = __half_as_ushort(h);
  const bool neg = (hb & 0x8000u) != 0;
  unsigned short nb;   // the fp16 neighbour of hf on the side of zh
  if (d > 0.f) nb = neg ? (hb == 0x8000u ? 0x0001u : (unsigned short)(hb - 1)) : (unsigned short)(hb + 1);
  else nb = neg ? (unsigned short)(hb + 1) : (hb == 0 ? 0x8001u : (unsigned short)(hb - 1));
  const float nf = __half2float(__ushort_as_half(nb));
  if (zh == 0.5f * (hf + nf) && (d > 0.f) == (zl > 0.f)) return __ushort_as_half(nb);
  return h;
}

struct AdmJob {
  unsigned long long src, dst;        // byte offsets in the old / new blob
  long long nblk, blk, sstride, dstride;
};
struct AdmCopyUnit {
  const char* in;
  char* out;
  unsigned char hdr[88];
  int D, njobs;
  int8_t* signs;                      // the sign vector as int8 (workspace)
  AdmJob job[ADM_MAX_JOBS];
};
struct AdmCopyBatch {
  AdmCopyUnit u[ADM_MAX_UNITS];
};

// New header, the sign bits carried over, and every section of the old
// tokens moved to its place in the longer layout (grid y = unit).
__global__ void adm_copy_kernel(const __grid_constant__ AdmCopyBatch cb) {
  const AdmCopyUnit& u = cb.u[blockIdx.y];
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < 88; i += blockDim.x) u.out[i] = (char)u.hdr[i];
    for (int i = threadIdx.x; i < (u.D + 7) / 8; i += blockDim.x) u.out[88 + i] = u.in[88 + i];
    for (int d = threadIdx.x; d < u.D; d += blockDim.x)
      u.signs[d] = ((((const unsigned char*)u.in)[88 + (d >> 3)] >> (d & 7)) & 1) ? -1 : 1;
  }
  for (int j = 0; j < u.njobs; ++j) {
    const AdmJob& jb = u.job[j];
    const bool w4 = ((jb.src | jb.dst | (unsigned long long)jb.blk | (unsigned long long)jb.sstride |
                      (unsigned long long)jb.dstride) & 3) == 0;
    if (w4) {
      const long long per = jb.blk / 4, n = jb.nblk * per;
      for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
           e += (long long)gridDim.x * blockDim.x) {
        const long long bk = e / per, o = e % per;
        reinterpret_cast<uint32_t*>(u.out + jb.dst + bk * jb.dstride)[o] =
            reinterpret_cast<const uint32_t*>(u.in + jb.src + bk * jb.sstride)[o];
      }
    } else {
      const long long per = jb.blk / 2, n = jb.nblk * per;
      for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
           e += (long long)gridDim.x * blockDim.x) {
        const long long bk = e / per, o = e % per;
        reinterpret_cast<unsigned short*>(u.out + jb.dst + bk * jb.dstride)[o] =
            reinterpret_cast<const unsigned short*>(u.in + jb.src + bk * jb.sstride)[o];
      }
    }
  }
}

struct AdmUnit {
  const void* X;          // [H][tau][D] new tokens
  const __half* Ud;       // stored U_d [D][rd], or null for r_d = D
  const __half* G;        // stored core [H][rT][rd] (r_T < T)
  __half* Gout;           // r_T = T: new core rows at Gout + h * g_hs + t * rd
  long long g_hs;
  __half* UTout;          // r_T < T: new U_T rows [tau][rT]
  float* Yh;              // r_T < T: Y = X U_d as double-float [H][tau][rd]
  float* Yl;
  double* M;              // sum_h G_h G_h^T [rT][rT]
  int rT, rd, whole;      // whole: r_T = T (the core gains rows)
};
struct AdmBatch {
  AdmUnit u[ADM_MAX_UNITS];
  int H, tau, D, xdt;
};

// Y[h][t][j] = sum_d X[h][t][d] U_d[d][j] in double-float; for a whole
// token mode the core rows fp16(Y) go straight to the new blob.  Grid:
// (ceil(tau / 8), H, unit), 256 threads = 8 tokens x 32 lanes over j.
__global__ void adm_proj_kernel(const __grid_constant__ AdmBatch ab) {
  const AdmUnit& a = ab.u[blockIdx.z];
  const int D = ab.D, tau = ab.tau, h = blockIdx.y;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + w;
  __shared__ float xs[8][128];
  if (t < tau)
    for (int d = lane; d < D; d += 32) {
      const long long o = ((long long)h * tau + t) * D + d;
      xs[w][d] = ab.xdt == JOLT_BF16 ? __bfloat162float(((const __nv_bfloat16*)a.X)[o])
                                     : ((const float*)a.X)[o];
    }
  __syncwarp();
  if (t >= tau) return;
  for (int j = lane; j < a.rd; j += 32) {
    float sh, sl;
    if (!a.Ud) {
      sh = xs[w][j];
      sl = 0.f;
    } else {
      sh = 0.f; sl = 0.f;
      for (int d = 0; d < D; ++d) {
        const float u = __half2float(a.Ud[(long long)d * a.rd + j]);
        const float p = xs[w][d] * u;
        const float pe = fmaf(xs[w][d], u, -p);
        float s2, e;
        two_sum(sh, p, s2, e);
        sh = s2;
        sl += e + pe;
      }
      const float hi = sh + sl;
      sl = sl - (hi - sh);
      sh = hi;
    }
    if (a.whole) {
      a.Gout[(long long)h * a.g_hs + (long long)t * a.rd + j] = round_f16_df_signed(sh, sl);
    } else {
      const long long o = ((long long)h * tau + t) * a.rd + j;
      a.Yh[o] = sh;
      a.Yl[o] = sl;
    }
  }
}

// M[k][l] = sum_h sum_j G[h][k][j] G[h][l][j] (fp16 products exact in fp32,
// TwoSum accumulation), as f64.  Grid: (rT, unit), 64 threads over l.
__global__ void adm_gram_kernel(const __grid_constant__ AdmBatch ab) {
  const AdmUnit& a = ab.u[blockIdx.y];
  const int k = blockIdx.x, l = threadIdx.x;
  if (a.whole || k >= a.rT || l >= a.rT) return;
  float sh = 0.f, sl = 0.f;
  for (int h = 0; h < ab.H; ++h) {
    const __half* Gh = a.G + (long long)h * a.rT * a.rd;
    for (int j = 0; j < a.rd; ++j) {
      const float p = __half2float(Gh[k * a.rd + j]) * __half2float(Gh[l * a.rd + j]);
      float s2, e;
      two_sum(sh, p, s2, e);
      sh = s2;
      sl += e;
    }
  }
  a.M[k * a.rT + l] = (double)sh + (double)sl;
}

// The fold-in: for each new token t, u_t solves (sum_h G_h G_h^T) u =
// sum_h G_h Y[h][t]^T.  One CTA per (8 tokens, unit): the CTA factors M by
// Cholesky in f64 (pivots at most 2^-40 max diag(M) dropped: that
// coordinate is 0), a warp per token forms its right-hand side in
// double-float and substitutes in f64; u is rounded to fp16 into the blob.
__global__ void __launch_bounds__(256) adm_solve_kernel(const __grid_constant__ AdmBatch ab) {
  const AdmUnit& a = ab.u[blockIdx.y];
  if (a.whole) return;
  const int rT = a.rT, rd = a.rd, H = ab.H, tau = ab.tau;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  __shared__ double L[ADM_RT][ADM_RT + 1];
  __shared__ int keep[ADM_RT];
  __shared__ double tol;
  for (int e = tid; e < rT * rT; e += 256) L[e / rT][e % rT] = a.M[e];
  __syncthreads();
  if (tid == 0) {
    double mx = 0.0;
    for (int j = 0; j < rT; ++j) mx = fmax(mx, L[j][j]);
    tol = 0x1p-40 * mx;
  }
  __syncthreads();
  // right-looking Cholesky on the lower triangle
  for (int j = 0; j < rT; ++j) {
    const double d = L[j][j];
    const bool kj = d > tol;
    __syncthreads();
    if (tid == 0) {
      keep[j] = kj;
      L[j][j] = kj ? sqrt(d) : 0.0;
    }
    __syncthreads();
    for (int i = j + 1 + tid; i < rT; i += 256) L[i][j] = kj ? L[i][j] / L[j][j] : 0.0;
    __syncthreads();
    if (kj)
      for (int e = tid; e < (rT - j - 1) * (rT - j - 1); e += 256) {
        const int i = j + 1 + e / (rT - j - 1), c = j + 1 + e % (rT - j - 1);
        if (c <= i) L[i][c] -= L[i][j] * L[c][j];
      }
    __syncthreads();
  }
  const int t = blockIdx.x * 8 + w;
  if (t >= tau) return;
  // right-hand side: lanes over k (k = lane, lane + 32)
  double r[2];
  for (int q = 0; q < 2; ++q) {
    const int k = lane + 32 * q;
    float sh = 0.f, sl = 0.f;
    if (k < rT) {
      for (int h = 0; h < H; ++h) {
        const __half* Gk = a.G + ((long long)h * rT + k) * rd;
        const float* yh = a.Yh + ((long long)h * tau + t) * rd;
        const float* yl = a.Yl + ((long long)h * tau + t) * rd;
        for (int j = 0; j < rd; ++j) {
          const float g = __half2float(Gk[j]);
          const float p = yh[j] * g;
          const float pe = fmaf(yh[j], g, -p);
          float s2, e;
          two_sum(sh, p, s2, e);
          sh = s2;
          sl += e + fmaf(yl[j], g, pe);
        }
      }
    }
    r[q] = (double)sh + (double)sl;
  }
  // forward substitution L z = r, then back substitution L^T u = z
  for (int j = 0; j < rT; ++j) {
    const int owner = j & 31, q = j >> 5;
    double zj = __shfl_sync(0xffffffffu, q ? r[1] : r[0], owner);
    zj = keep[j] ? zj / L[j][j] : 0.0;
    if (lane == owner) { if (q) r[1] = zj; else r[0] = zj; }
    for (int qq = 0; qq < 2; ++qq) {
      const int i = lane + 32 * qq;
      if (i > j && i < rT) r[qq] -= L[i][j] * zj;
    }
  }
  for (int j = rT - 1; j >= 0; --j) {
    const int owner = j & 31, q = j >> 5;
    double uj = __shfl_sync(0xffffffffu, q ? r[1] : r[0], owner);
    uj = keep[j] ? uj / L[j][j] : 0.0;
    if (lane == owner) { if (q) r[1] = uj; else r[0] = uj; }
    for (int qq = 0; qq < 2; ++qq) {
      const int i = lane + 32 * qq;
      if (i < j) r[qq] -= L[j][i] * uj;
    }
  }
  for (int q = 0; q < 2; ++q) {
    const int k = lane + 32 * q;
    if (k < rT) a.UTout[(long long)t * rT + k] = __double2half(r[q]);
  }
}

}  // namespace

void blob_layout(int H, int T, int D, int rT, int rd, int b, int block, int align,
                 jolt_blob_desc* d) {
  const long long n = (long long)H * T * D;
  long long off = JOLT_HEADER_BYTES;
  uint64_t* offs[5] = {&d->off_UT, &d->off_Ud, &d->off_G, &d->off_scale, &d->off_codes};
  const long long sz[5] = {rT == T ? 0 : 2LL * T * rT, rd == D ? 0 : 2LL * D * rd,
                           2LL * H * rT * rd, b == 0 ? 0 : 2 * (n / block), b == 0 ? 0 : n * b / 8};
  for (int s = 0; s < 5; ++s) {
    off = (long long)align_up((size_t)off, (size_t)align);
    *offs[s] = sz[s] > 0 ? (uint64_t)off : (uint64_t)0;
    off += sz[s];
  }
  d->bytes = align_up((size_t)off, (size_t)align);
  d->H = H; d->T = T; d->D = D; d->rT = rT; d->rd = rd; d->b = b; d->block = block;
  d->flags = (rT == T ? 1 : 0) | (rd == D ? 2 : 0);
}

jolt_status encode_run(const Layout& L, int U, const void* X, const int8_t* signs, const char* ws,
                       const int32_t* choice, char* blob, size_t stride, jolt_blob_desc* desc,
                       cudaStream_t st) {
  const int H = L.H, T = L.T, D = L.D, RT = L.RT, RD = L.RD;
  const size_t xes = (L.dtype == JOLT_F32) ? 4 : 2;
  const long long xu = (long long)H * T * D;
  // validate and lay out every unit before launching anything
  for (int u = 0; u < U; ++u) {
    if (choice[u] < 0 || choice[u] >= L.ncand) return JOLT_ERR_INVALID;
    int iT, id, ib;
    cand_split(L, choice[u], &iT, &id, &ib);
    blob_layout(H, T, D, L.rT[iT], L.rd[id], L.b[ib], L.block, L.align, &desc[u]);
    if (desc[u].bytes > stride) return JOLT_ERR_INVALID;
  }
  // one zero fill for every blob slot (padding bytes are deterministic)
  JOLT_CUDA_TRY(cudaMemsetAsync(blob, 0, (size_t)U * stride, st));
  // per batch of up to ENC_MAX_UNITS units: one launch for the headers and
  // factor sections, one for the chain rows, one for the codes
  SecBatch secs;
  RowsBatch rows;
  EncBatch batch;
  int nsec = 0, nrows = 0, nbatch = 0;
  const bool bf = (L.dtype == JOLT_BF16);
  auto flush = [&]() -> jolt_status {
    if (nsec > 0) {
      sections_kernel<<<dim3(64, nsec), 256, 0, st>>>(secs);
      JOLT_LAUNCH_CHECK();
    }
    if (nrows > 0) {
      rows.D = D;
      enc_rows_batch_kernel<<<dim3((RT * D + 255) / 256, H, nrows), 256, 0, st>>>(rows);
      JOLT_LAUNCH_CHECK();
    }
    jolt_status ls = JOLT_OK;
    if (nbatch > 0) {
      dim3 grid((T + CD_TILE - 1) / CD_TILE, H, nbatch);
      switch (D) {
        case 128: ls = bf ? launch_enc<__nv_bfloat16, 4>(grid, batch, st) : launch_enc<float, 4>(grid, batch, st); break;
        case 64: ls = bf ? launch_enc<__nv_bfloat16, 2>(grid, batch, st) : launch_enc<float, 2>(grid, batch, st); break;
        default: ls = bf ? launch_enc<__nv_bfloat16, 1>(grid, batch, st) : launch_enc<float, 1>(grid, batch, st);
      }
    }
    nsec = nrows = nbatch = 0;
    return ls;
  };
  for (int u = 0; u < U; ++u) {
    int iT, id, ib;
    cand_split(L, choice[u], &iT, &id, &ib);
    const int rT = L.rT[iT], rd = L.rd[id], b = L.b[ib];
    const jolt_blob_desc& dsc = desc[u];
    char* bl = blob + (size_t)u * stride;
    const char* wu = ws + (size_t)u * L.unit_bytes;
    const void* Xu = (const char*)X + (size_t)u * xu * xes;
    SecUnit& su = secs.u[nsec++];
    memset(&su, 0, sizeof(su));
    const uint32_t hd32[10] = {MAGIC, VERSION, (uint32_t)H, (uint32_t)T, (uint32_t)D, (uint32_t)rT,
                               (uint32_t)rd, (uint32_t)b, (uint32_t)L.block, (uint32_t)dsc.flags};
    memcpy(su.ha.fixed, hd32, 40);
    const uint64_t hd64[6] = {dsc.off_UT, dsc.off_Ud, dsc.off_G, dsc.off_scale, dsc.off_codes,
                              dsc.bytes};
    memcpy(su.ha.fixed + 40, hd64, 48);
    su.ha.D = D;
    su.signs = signs + (size_t)u * D;
    su.blob = bl;
    auto job = [&](const void* src, int type, long long sa, long long sbv, size_t off, int A, int B,
                   int C) {
      CopyJob& j = su.job[su.njobs++];
      j.src = src; j.type = type; j.sa = sa; j.sb = sbv;
      j.dst = (__half*)(bl + off); j.A = A; j.B = B; j.C = C;
    };
    // factor sections
    if (rT < T) job(wu + L.o_UT16 + (size_t)id * T * RT * 2, 0, 0, RT, dsc.off_UT, 1, T, rT);
    if (rd < D) job(wu + L.o_Ud16, 0, 0, RD, dsc.off_Ud, 1, D, rd);
    if (rT < T) {
      job(wu + L.o_G16 + (size_t)id * H * RT * D * 2, 0, (long long)RT * rd, rd, dsc.off_G, H, rT, rd);
    } else if (rd < D) {
      job(wu + L.o_Y16, 0, (long long)T * RD, RD, dsc.off_G, H, T, rd);
    } else {
      job(Xu, L.dtype == JOLT_BF16 ? 1 : (L.dtype == JOLT_F16 ? 0 : 2), (long long)T * D, D,
          dsc.off_G, H, T, D);
    }
    if (b > 0) {
      EncArgs ea;
      memset(&ea, 0, sizeof(ea));
      ea.X = Xu; ea.signs = signs + (size_t)u * D;
      ea.H = H; ea.T = T; ea.D = D; ea.dtype = L.dtype; ea.b = b;
      ea.blob = bl; ea.off_scale = dsc.off_scale; ea.off_codes = dsc.off_codes;
      ea.row_ld = T; ea.row_off = 0;
      {
        const double rs = 1.0 / sqrt((double)D);
        ea.rs_hi = (float)rs;
        ea.rs_lo = (float)(rs - (double)ea.rs_hi);
      }
      const __half* Ud16 = (const __half*)(wu + L.o_Ud16);
      if (rT == T && rd == D) {
        ea.mode = 2;
      } else if (rT == T) {
        // X~_h = Y16_h U_d16^T
        ea.mode = 1; ea.K = rd;
        ea.Kg = (const __half*)(wu + L.o_Y16); ea.k_hs = (long long)T * RD; ea.k_ld = RD;
        ea.B16 = Ud16; ea.b_hs = 0; ea.b_ks = 1; ea.b_ds = RD;
      } else {
        // X~_h = U_T16 (G16_h U_d16^T)
        ea.mode = 0; ea.K = rT;
        ea.Kg = (const __half*)(wu + L.o_UT16) + (size_t)id * T * RT; ea.k_hs = 0; ea.k_ld = RT;
        const __half* G16 = (const __half*)(wu + L.o_G16) + (size_t)id * H * RT * D;
        if (rd == D) {
          ea.B16 = G16; ea.b_hs = (long long)RT * D; ea.b_ks = D; ea.b_ds = 1;
        } else {
          float* Bh = (float*)(ws + (size_t)u * L.unit_bytes + L.o_W);
          float* Blo = Bh + (size_t)H * rT * D;
          RowsUnit& ru = rows.u[nrows++];
          ru.G = G16; ru.g_hs = (long long)RT * rd; ru.Ud = Ud16; ru.ldu = RD;
          ru.rT = rT; ru.rd = rd; ru.Bhi = Bh; ru.Blo = Blo;
          ea.Bhi = Bh; ea.Blo = Blo; ea.b_hs = (long long)rT * D;
        }
      }
      batch.u[nbatch++] = ea;
    }
    if (nsec == ENC_MAX_UNITS) {
      jolt_status ls = flush();
      if (ls != JOLT_OK) return ls;
    }
  }
  {
    jolt_status ls = flush();
    if (ls != JOLT_OK) return ls;
  }
  return JOLT_OK;
}

jolt_status decode_run(int U, const jolt_blob_desc* desc, const char* blob, size_t stride,
                       void* xhat, int out_dtype, cudaStream_t st) {
  const int H = desc[0].H, T = desc[0].T, D = desc[0].D;
  // D = 128: the tensor-core decoder (16-byte vector loads of codes and
  // whole-mode cores, 16-byte stores)
  bool tc_ok = decode_tc_supported(D) && ((uintptr_t)xhat % 16) == 0 &&
               ((uintptr_t)blob % 16) == 0 && (stride % 16) == 0;
  for (int u = 0; u < U && tc_ok; ++u)
    tc_ok = (desc[u].off_codes % 16) == 0 && (desc[u].off_G % 16) == 0;
  if (tc_ok) return decode_tc_run(U, desc, blob, stride, xhat, out_dtype, st);
  for (int u0 = 0; u0 < U; u0 += DEC_MAX_UNITS) {
    const int nu = (U - u0) < DEC_MAX_UNITS ? (U - u0) : DEC_MAX_UNITS;
    DecArgs a;
    memset(&a, 0, sizeof(a));
    a.H = H; a.T = T; a.D = D; a.out_dtype = out_dtype; a.blob = blob; a.stride = stride;
    a.xhat = xhat; a.u0 = u0;
    for (int i = 0; i < nu; ++i) {
      const jolt_blob_desc& d = desc[u0 + i];
      a.un[i].rT = d.rT; a.un[i].rd = d.rd; a.un[i].b = d.b;
      a.un[i].off_UT = d.off_UT; a.un[i].off_Ud = d.off_Ud; a.un[i].off_G = d.off_G;
      a.un[i].off_scale = d.off_scale; a.un[i].off_codes = d.off_codes;
    }
    dim3 grid((T + CD_TILE - 1) / CD_TILE, H, nu);
    jolt_status ls;
    switch (D) {
      case 128: ls = launch_dec<4>(grid, a, st); break;
      case 64: ls = launch_dec<2>(grid, a, st); break;
      default: ls = launch_dec<1>(grid, a, st);
    }
    if (ls != JOLT_OK) return ls;
  }
  return JOLT_OK;
}

size_t admit_ws_unit_bytes(int H, int tau, int D) {
  // signs, Y (double-float), M (f64), chain rows (double-float)
  return align_up(256 + (size_t)H * tau * D * 8 + (size_t)ADM_RT * ADM_RT * 8 +
                      (size_t)H * ADM_RT * D * 8, 256);
}

jolt_status admit_run(int U, const jolt_blob_desc* din, const char* bin, size_t sin,
                      const void* Xn, int xdt, int tau, int align, char* ws, char* bout,
                      size_t sout, jolt_blob_desc* dout, cudaStream_t st) {
  const int H = din[0].H, T = din[0].T, D = din[0].D;
  const int Tn = T + tau;
  const size_t wub = admit_ws_unit_bytes(H, tau, D);
  const size_t xes = xdt == JOLT_BF16 ? 2 : 4;
  for (int u = 0; u < U; ++u) {
    const jolt_blob_desc& d = din[u];
    const int rTn = d.rT == T ? Tn : d.rT;
    blob_layout(H, Tn, D, rTn, d.rd, d.b, D, align, &dout[u]);
    if (dout[u].bytes > sout) return JOLT_ERR_INVALID;
  }
  JOLT_CUDA_TRY(cudaMemsetAsync(bout, 0, (size_t)U * sout, st));
  for (int u0 = 0; u0 < U; u0 += ADM_MAX_UNITS) {
    const int nu = (U - u0) < ADM_MAX_UNITS ? (U - u0) : ADM_MAX_UNITS;
    AdmCopyBatch cb;
    AdmBatch ab;
    RowsBatch rows;
    EncBatch eb;
    memset(&cb, 0, sizeof(cb));
    memset(&ab, 0, sizeof(ab));
    memset(&rows, 0, sizeof(rows));
    memset(&eb, 0, sizeof(eb));
    ab.H = H; ab.tau = tau; ab.D = D; ab.xdt = xdt;
    rows.D = D;
    int nrows = 0, nenc = 0, nsolve = 0;
    for (int i = 0; i < nu; ++i) {
      const int u = u0 + i;
      const jolt_blob_desc& di = din[u];
      const jolt_blob_desc& dn = dout[u];
      const char* bi = bin + (size_t)u * sin;
      char* bo = bout + (size_t)u * sout;
      char* wu = ws + (size_t)u * wub;
      const int rT = di.rT, rd = di.rd, b = di.b;
      const bool whole = (rT == T), fullD = (rd == D);
      // header and the old tokens' sections
      AdmCopyUnit& cu = cb.u[i];
      cu.in = bi; cu.out = bo; cu.D = D; cu.signs = (int8_t*)wu;
      const uint32_t hd32[10] = {MAGIC, VERSION, (uint32_t)H, (uint32_t)Tn, (uint32_t)D,
                                 (uint32_t)dn.rT, (uint32_t)rd, (uint32_t)b, (uint32_t)D,
                                 (uint32_t)dn.flags};
      memcpy(cu.hdr, hd32, 40);
      const uint64_t hd64[6] = {dn.off_UT, dn.off_Ud, dn.off_G, dn.off_scale, dn.off_codes,
                                dn.bytes};
      memcpy(cu.hdr + 40, hd64, 48);
      auto job = [&](unsigned long long src, unsigned long long dst, long long nblk, long long blk,
                     long long ss, long long ds) {
        AdmJob& j = cu.job[cu.njobs++];
        j.src = src; j.dst = dst; j.nblk = nblk; j.blk = blk; j.sstride = ss; j.dstride = ds;
      };
      if (!whole) job(di.off_UT, dn.off_UT, 1, 2LL * T * rT, 0, 0);
      if (!fullD) job(di.off_Ud, dn.off_Ud, 1, 2LL * D * rd, 0, 0);
      if (!whole) job(di.off_G, dn.off_G, 1, 2LL * H * rT * rd, 0, 0);
      else job(di.off_G, dn.off_G, H, 2LL * T * rd, 2LL * T * rd, 2LL * Tn * rd);
      if (b > 0) {
        job(di.off_scale, dn.off_scale, H, 2LL * T, 2LL * T, 2LL * Tn);
        const long long rb = (long long)T * D * b / 8, rbn = (long long)Tn * D * b / 8;
        job(di.off_codes, dn.off_codes, H, rb, rb, rbn);
      }
      // the new tokens' stored rows
      AdmUnit& au = ab.u[i];
      au.X = (const char*)Xn + (size_t)u * H * tau * D * xes;
      au.Ud = fullD ? nullptr : (const __half*)(bo + dn.off_Ud);
      au.G = (const __half*)(bo + dn.off_G);
      au.rT = whole ? 0 : rT; au.rd = rd; au.whole = whole;
      float* Y = (float*)(wu + 256);
      au.Yh = Y;
      au.Yl = Y + (size_t)H * tau * rd;
      au.M = (double*)(wu + 256 + (size_t)H * tau * D * 8);
      float* Bh = (float*)(wu + 256 + (size_t)H * tau * D * 8 + (size_t)ADM_RT * ADM_RT * 8);
      if (whole) {
        au.Gout = (__half*)(bo + dn.off_G) + (size_t)T * rd;
        au.g_hs = (long long)Tn * rd;
      } else {
        au.UTout = (__half*)(bo + dn.off_UT) + (size_t)T * rT;
        ++nsolve;
      }
      // the new tokens' codes, from the stored rows as in encode
      if (b > 0) {
        EncArgs& ea = eb.u[nenc++];
        ea.X = au.X; ea.signs = cu.signs;
        ea.H = H; ea.T = tau; ea.D = D; ea.dtype = xdt; ea.b = b;
        ea.blob = bo; ea.off_scale = dn.off_scale; ea.off_codes = dn.off_codes;
        ea.row_ld = Tn; ea.row_off = T;
        const double rs = 1.0 / sqrt((double)D);
        ea.rs_hi = (float)rs;
        ea.rs_lo = (float)(rs - (double)ea.rs_hi);
        if (whole && fullD) {
          ea.mode = 2;
        } else if (whole) {
          ea.mode = 1; ea.K = rd;
          ea.Kg = au.Gout; ea.k_hs = (long long)Tn * rd; ea.k_ld = rd;
          ea.B16 = au.Ud; ea.b_hs = 0; ea.b_ks = 1; ea.b_ds = rd;
        } else {
          ea.mode = 0; ea.K = rT;
          ea.Kg = au.UTout; ea.k_hs = 0; ea.k_ld = rT;
          if (fullD) {
            ea.B16 = au.G; ea.b_hs = (long long)rT * D; ea.b_ks = D; ea.b_ds = 1;
          } else {
            RowsUnit& ru = rows.u[nrows++];
            ru.G = au.G; ru.g_hs = (long long)rT * rd; ru.Ud = au.Ud; ru.ldu = rd;
            ru.rT = rT; ru.rd = rd; ru.Bhi = Bh; ru.Blo = Bh + (size_t)H * rT * D;
            ea.Bhi = ru.Bhi; ea.Blo = ru.Blo; ea.b_hs = (long long)rT * D;
          }
        }
      }
    }
    adm_copy_kernel<<<dim3(128, nu), 256, 0, st>>>(cb);
    JOLT_LAUNCH_CHECK();
    adm_proj_kernel<<<dim3((tau + 7) / 8, H, nu), 256, 0, st>>>(ab);
    JOLT_LAUNCH_CHECK();
    if (nsolve > 0) {
      adm_gram_kernel<<<dim3(ADM_RT, nu), 64, 0, st>>>(ab);
      JOLT_LAUNCH_CHECK();
      adm_solve_kernel<<<dim3((tau + 7) / 8, nu), 256, 0, st>>>(ab);
      JOLT_LAUNCH_CHECK();
    }
    if (nrows > 0) {
      enc_rows_batch_kernel<<<dim3((ADM_RT * D + 255) / 256, H, nrows), 256, 0, st>>>(rows);
      JOLT_LAUNCH_CHECK();
    }
    if (nenc > 0) {
      const dim3 grid((tau + CD_TILE - 1) / CD_TILE, H, nenc);
      jolt_status ls;
      const bool bf = (xdt == JOLT_BF16);
      switch (D) {
        case 128: ls = bf ? launch_enc<__nv_bfloat16, 4>(grid, eb, st) : launch_enc<float, 4>(grid, eb, st); break;
        case 64: ls = bf ? launch_enc<__nv_bfloat16, 2>(grid, eb, st) : launch_enc<float, 2>(grid, eb, st); break;
        default: ls = bf ? launch_enc<__nv_bfloat16, 1>(grid, eb, st) : launch_enc<float, 1>(grid, eb, st);
      }
      if (ls != JOLT_OK) return ls;
    }
  }
  return JOLT_OK;
}

}  // namespace jolt
