// Global byte-budget allocation by bisection on the Lagrange multiplier.
//
// ["Joint Tucker-rank and residual-bit KV allocator", Formulas: L(z, lambda)
//  = sum D(z) + lambda (sum C(z) - B), z*(lambda) = argmin_z D(z) + lambda C(z)
//  per group and cache type; Implementation notes: binary-search lambda until
//  total storage is within one alignment block of B; "Technical Summary: A
//  JOLT for the KV Cache", Methodology 3.]
//
// One thread block.  Each best response is taken per unit by one warp: the
// candidate with the least dist + lambda * cost (the product rounded before
// the sum, no fused multiply-add), ties to the smaller cost, then the lower
// candidate index.  The schedule of lambda values:
//   z(0) fits            -> return it, lambda = 0
//   cheapest misfits     -> return the cheapest allocation, INFEASIBLE
//   otherwise hi = 1, doubled until z(hi) fits, lo = the last misfit (0 at
//   first); then up to 200 bisection steps on mid = (lo + hi) / 2, keeping
//   z(hi) feasible, stopping once sum C(z(hi)) is within one alignment block
//   of the budget or hi - lo <= 2^-52 hi; return z(hi), hi.
#include "jolt_internal.cuh"

namespace jolt {

namespace {

constexpr int AL_THREADS = 512;
constexpr int AL_MAX_ITER = 200;

// Lexicographic key (k1, k2, index) on unsigned integers that order like the
// values they encode, so that no comparison needs the fp64 pipe: a double
// maps to its bit pattern with the sign bit set (>= +0) or all bits inverted
// (< 0), -0 first folded to +0; a signed cost to its value with the sign bit
// flipped.
__device__ __forceinline__ unsigned long long dkey(double x) {
  long long b = __double_as_longlong(x);
  if (b == (long long)0x8000000000000000ull) b = 0;
  return (unsigned long long)(b ^ ((b >> 63) | (long long)0x8000000000000000ull));
}
__device__ __forceinline__ unsigned long long ikey(long long k) {
  return (unsigned long long)k ^ 0x8000000000000000ull;
}

struct Key {
  unsigned long long k1, k2;
  int i;
};

__device__ __forceinline__ bool less_key(const Key& a, const Key& b) {
  if (a.k1 != b.k1) return a.k1 < b.k1;
  if (a.k2 != b.k2) return a.k2 < b.k2;
  return a.i < b.i;
}

// The tables as the best responses read them: dist, cost, and the cost
// converted to double once (exact for |cost| < 2^53; null when the tables
// stay in global memory, then converted on the fly).
struct Tabs {
  const double* dist;
  const int64_t* cost;
  const double* costd;
};

// mode 0: z(lambda), key (dist + lambda*cost, cost, index)
// mode 1: cheapest allocation, key (cost, dist, index)
// Writes out[u] and returns the total cost (the same in every thread).  One
// barrier per call: the warps' totals go to one of two buffers in turn
// (`parity`), and every warp sums them itself.
__device__ long long best_response(int U, int nc, const Tabs& tb, double lam, int mode, int* out,
                                   int& parity) {
  const int w = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  __shared__ long long part[2][AL_THREADS / 32];
  long long mine = 0;
  for (int u = w; u < U; u += nw) {
    Key b{~0ull, ~0ull, INT_MAX};
    for (int c = lane; c < nc; c += 32) {
      const long long i = (long long)u * nc + c;
      const double d = tb.dist[i];
      const long long k = tb.cost[i];
      Key x;
      if (mode == 0) {
        const double kd = tb.costd ? tb.costd[i] : (double)k;
        x.k1 = dkey(__dadd_rn(d, __dmul_rn(lam, kd)));
        x.k2 = ikey(k);
      } else {
        x.k1 = ikey(k);
        x.k2 = dkey(d);
      }
      x.i = c;
      if (less_key(x, b)) b = x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Key y;
      y.k1 = __shfl_xor_sync(0xffffffffu, b.k1, o);
      y.k2 = __shfl_xor_sync(0xffffffffu, b.k2, o);
      y.i = __shfl_xor_sync(0xffffffffu, b.i, o);
      if (less_key(y, b)) b = y;
    }
    if (lane == 0) {
      out[u] = b.i;
      mine += tb.cost[(long long)u * nc + b.i];
    }
  }
  if (lane == 0) part[parity][w] = mine;
  __syncthreads();
  long long s = lane < nw ? part[parity][lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  parity ^= 1;
  return s;
}

__global__ void __launch_bounds__(AL_THREADS)
alloc_kernel(int U, int nc, const double* __restrict__ gdist, const int64_t* __restrict__ gcost,
             long long budget, int align, int32_t* choice, double* lambda, int32_t* status,
             int cached) {
  extern __shared__ __align__(16) unsigned char asm_raw[];
  // tables copied into shared memory once when they fit (the bisection
  // evaluates best responses up to a few hundred times)
  Tabs tb{gdist, gcost, nullptr};
  int* zs;
  if (cached) {
    double* sd = (double*)asm_raw;
    double* scd = sd + (size_t)U * nc;
    int64_t* sc = (int64_t*)(scd + (size_t)U * nc);
    for (int i = threadIdx.x; i < U * nc; i += blockDim.x) {
      sd[i] = gdist[i];
      sc[i] = gcost[i];
      scd[i] = (double)gcost[i];
    }
    tb = Tabs{sd, sc, scd};
    zs = (int*)(sc + (size_t)U * nc);
  } else {
    zs = (int*)asm_raw;
  }
  __syncthreads();
  int* zhi = zs;            // [U], the last feasible best response
  int* zmid = zs + U;       // [U], the one being evaluated (the two swap roles)
  int parity = 0;
  long long tot = best_response(U, nc, tb, 0.0, 0, zhi, parity);
  if (tot <= budget) {
    for (int u = threadIdx.x; u < U; u += blockDim.x) choice[u] = zhi[u];
    if (threadIdx.x == 0) { *lambda = 0.0; *status = JOLT_OK; }
    return;
  }
  tot = best_response(U, nc, tb, 0.0, 1, zhi, parity);
  if (tot > budget) {
    for (int u = threadIdx.x; u < U; u += blockDim.x) choice[u] = zhi[u];
    if (threadIdx.x == 0) { *lambda = INFINITY; *status = JOLT_ERR_INFEASIBLE; }
    return;
  }
  double lo = 0.0, hi = 1.0;
  long long chi = best_response(U, nc, tb, hi, 0, zhi, parity);
  // z(lambda) reaches the cheapest allocation, which fits, as lambda grows;
  // the cap only guards non-finite tables
  while (chi > budget && hi < 1e300) {
    lo = hi;
    hi = hi * 2.0;
    chi = best_response(U, nc, tb, hi, 0, zhi, parity);
  }
  for (int it = 0; it < AL_MAX_ITER; ++it) {
    if ((budget - align < chi && chi <= budget) || hi - lo <= 0x1.0p-52 * hi) break;
    const double mid = 0.5 * (lo + hi);
    tot = best_response(U, nc, tb, mid, 0, zmid, parity);
    if (tot <= budget) {
      hi = mid;
      chi = tot;
      int* z = zhi;
      zhi = zmid;
      zmid = z;
    } else {
      lo = mid;
    }
  }
  for (int u = threadIdx.x; u < U; u += blockDim.x) choice[u] = zhi[u];
  if (threadIdx.x == 0) {
    *lambda = hi;
    *status = (chi <= budget) ? JOLT_OK : JOLT_ERR_INFEASIBLE;
  }
}

// Greedy improvement of a feasible allocation ["Joint Tucker-rank and
// residual-bit KV allocator", Implementation notes: swap candidates with the
// best distortion reduction per added byte].  A swap replaces unit u's
// candidate z by c with added bytes dc = C(c) - C(z) in (0, slack] and
// reduction dd = D(z) - D(c) > 0; its rate is dd / dc (f64, correctly
// rounded).  Every round applies the swap of highest rate (ties: smaller dc,
// then lower unit, then lower candidate), until none fits.  One thread block;
// each warp scans whole units, the block reduces the warps' bests.
struct SwapKey {
  unsigned long long k1, k2;   // ~rate key (higher rate first), dc
  int uc;                      // u * nc + c
};
__device__ __forceinline__ bool less_swap(const SwapKey& a, const SwapKey& b) {
  if (a.k1 != b.k1) return a.k1 < b.k1;
  if (a.k2 != b.k2) return a.k2 < b.k2;
  return a.uc < b.uc;
}

__global__ void __launch_bounds__(AL_THREADS)
refine_kernel(int U, int nc, const double* __restrict__ dist, const int64_t* __restrict__ cost,
              long long budget, int32_t* choice, int32_t* n_swaps) {
  extern __shared__ __align__(16) unsigned char rf_raw[];
  int* z = (int*)rf_raw;   // [U]
  __shared__ SwapKey wbest[AL_THREADS / 32];
  __shared__ long long slack;
  __shared__ int done;
  const int w = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  for (int u = threadIdx.x; u < U; u += blockDim.x) z[u] = choice[u];
  __syncthreads();
  if (threadIdx.x == 0) {
    long long c = 0;
    for (int u = 0; u < U; ++u) c += cost[(long long)u * nc + z[u]];
    slack = budget - c;
  }
  __syncthreads();
  const SwapKey none{~0ull, ~0ull, INT_MAX};
  int swaps = 0;
  for (int round = 0; round < U * nc; ++round) {
    SwapKey b = none;
    for (int u = w; u < U; u += nw) {
      const double d0 = dist[(long long)u * nc + z[u]];
      const long long c0 = cost[(long long)u * nc + z[u]];
      for (int c = lane; c < nc; c += 32) {
        const long long dc = cost[(long long)u * nc + c] - c0;
        const double dd = __dsub_rn(d0, dist[(long long)u * nc + c]);
        if (dc <= 0 || dc > slack || !(dd > 0.0)) continue;
        const double rate = __ddiv_rn(dd, (double)dc);
        const SwapKey k{~dkey(rate), ikey(dc), u * nc + c};
        if (less_swap(k, b)) b = k;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      SwapKey y;
      y.k1 = __shfl_xor_sync(0xffffffffu, b.k1, o);
      y.k2 = __shfl_xor_sync(0xffffffffu, b.k2, o);
      y.uc = __shfl_xor_sync(0xffffffffu, b.uc, o);
      if (less_swap(y, b)) b = y;
    }
    if (lane == 0) wbest[w] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
      SwapKey best = none;
      for (int i = 0; i < nw; ++i)
        if (less_swap(wbest[i], best)) best = wbest[i];
      done = (best.uc == INT_MAX);
      if (!done) {
        const int u = best.uc / nc, c = best.uc % nc;
        slack -= cost[(long long)u * nc + c] - cost[(long long)u * nc + z[u]];
        z[u] = c;
      }
    }
    __syncthreads();
    if (done) break;
    ++swaps;
  }
  for (int u = threadIdx.x; u < U; u += blockDim.x) choice[u] = z[u];
  if (threadIdx.x == 0 && n_swaps) *n_swaps = swaps;
}

struct UniformArgs {
  int n;                      // candidates in the list
  int cand[JOLT_MAX_CAND];    // flat indices
};

// The uniform baseline allocators ["Joint Tucker-rank and residual-bit KV
// allocator", Verification, Stage 1: every group on the same (r_T, r_d, b),
// fixed 4-bit]: every unit takes the same candidate of the list, the one of
// least total distortion (summed over units in order, f64) whose total cost
// fits (ties: lower index); with none fitting, the cheapest by total cost
// (ties: lower index) and JOLT_ERR_INFEASIBLE.  One thread per candidate,
// then one thread picks.
__global__ void __launch_bounds__(256)
uniform_kernel(int U, int nc, const double* __restrict__ dist, const int64_t* __restrict__ cost,
               long long budget, UniformArgs a, int32_t* choice, int32_t* status) {
  __shared__ double td[JOLT_MAX_CAND];
  __shared__ long long tc[JOLT_MAX_CAND];
  __shared__ int pick, st;
  for (int i = threadIdx.x; i < a.n; i += blockDim.x) {
    const int c = a.cand[i];
    double d = 0.0;
    long long k = 0;
    for (int u = 0; u < U; ++u) {
      d = __dadd_rn(d, dist[(long long)u * nc + c]);
      k += cost[(long long)u * nc + c];
    }
    td[i] = d;
    tc[i] = k;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = -1, cheap = -1;
    for (int i = 0; i < a.n; ++i) {
      const int c = a.cand[i];
      if (cheap < 0 || tc[i] < tc[cheap] || (tc[i] == tc[cheap] && c < a.cand[cheap])) cheap = i;
      if (tc[i] <= budget &&
          (best < 0 || td[i] < td[best] || (td[i] == td[best] && c < a.cand[best])))
        best = i;
    }
    pick = best >= 0 ? a.cand[best] : a.cand[cheap];
    st = best >= 0 ? JOLT_OK : JOLT_ERR_INFEASIBLE;
    *status = st;
  }
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) choice[u] = pick;
}

}  // namespace

jolt_status alloc_run(int U, int nc, const double* dist, const int64_t* cost, int64_t budget,
                      int align, int32_t* choice, double* lambda, int32_t* status,
                      cudaStream_t st) {
  const size_t ztab = (size_t)2 * U * sizeof(int);
  const size_t tabs = (size_t)U * nc * (2 * sizeof(double) + sizeof(int64_t));
  const int cached = (tabs + ztab <= 150 * 1024) ? 1 : 0;
  const size_t smem = cached ? tabs + ztab : ztab;
  if (smem > 160 * 1024) return JOLT_ERR_INVALID;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(alloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       160 * 1024));
    attr = true;
  }
  alloc_kernel<<<1, AL_THREADS, smem, st>>>(U, nc, dist, cost, (long long)budget, align, choice,
                                            lambda, status, cached);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace jolt

namespace jolt {

jolt_status refine_run(int U, int nc, const double* dist, const int64_t* cost, int64_t budget,
                       int32_t* choice, int32_t* n_swaps, cudaStream_t st) {
  const size_t smem = (size_t)U * sizeof(int);
  if (smem > 160 * 1024) return JOLT_ERR_INVALID;
  static bool attr = false;
  if (!attr) {
    JOLT_CUDA_TRY(cudaFuncSetAttribute(refine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       160 * 1024));
    attr = true;
  }
  refine_kernel<<<1, AL_THREADS, smem, st>>>(U, nc, dist, cost, (long long)budget, choice,
                                             n_swaps);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

jolt_status uniform_run(int U, int nc, const double* dist, const int64_t* cost, int64_t budget,
                        const int32_t* cand_host, int n_list, int32_t* choice, int32_t* status,
                        cudaStream_t st) {
  UniformArgs a;
  a.n = n_list;
  for (int i = 0; i < n_list; ++i) a.cand[i] = cand_host[i];
  uniform_kernel<<<1, 256, 0, st>>>(U, nc, dist, cost, (long long)budget, a, choice, status);
  JOLT_LAUNCH_CHECK();
  return JOLT_OK;
}

}  // namespace jolt
