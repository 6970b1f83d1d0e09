// C-ABI entry points of libjolt: argument validation, the per-unit workspace
// layout, and dispatch to the kernels of factor.cu, sweep.cu, alloc.cu and
// codec.cu.  Nothing here allocates device memory.
#include "jolt_internal.cuh"

#include <string.h>

namespace jolt {

unsigned long long g_launches = 0;

jolt_status make_layout(const jolt_config* cfg, Layout* Lp) {
  if (!cfg || !Lp) return JOLT_ERR_INVALID;
  Layout L;
  memset(&L, 0, sizeof(L));
  L.H = cfg->H; L.T = cfg->T; L.D = cfg->D; L.dtype = cfg->dtype;
  if (L.H <= 0 || L.T <= 0 || L.D <= 0) return JOLT_ERR_INVALID;
  if (!(L.D == 32 || L.D == 64 || L.D == 128)) return JOLT_ERR_INVALID;
  if (L.dtype != JOLT_F32 && L.dtype != JOLT_BF16) return JOLT_ERR_INVALID;
  if (cfg->quant_block != L.D) return JOLT_ERR_INVALID;
  if (cfg->n_rT < 1 || cfg->n_rT > JOLT_MAX_GRID || cfg->n_rd < 1 || cfg->n_rd > JOLT_MAX_GRID)
    return JOLT_ERR_INVALID;
  if (cfg->n_b < 1 || cfg->n_b > 4) return JOLT_ERR_INVALID;
  L.nT = cfg->n_rT; L.nd = cfg->n_rd; L.nb = cfg->n_b;
  // token ranks: ascending truncated ranks, then an optional FULL
  for (int i = 0; i < L.nT; ++i) {
    const int r = cfg->rT[i];
    if (r == JOLT_FULL) {
      if (i != L.nT - 1) return JOLT_ERR_INVALID;
      L.rT[i] = L.T;
      L.hasFullT = 1;
    } else {
      if (r < 1 || r > 64 || r >= L.T) return JOLT_ERR_INVALID;
      if (i > 0 && r <= cfg->rT[i - 1]) return JOLT_ERR_INVALID;
      L.rT[i] = r;
      L.nTt = i + 1;
      L.RT = r;
    }
  }
  for (int i = 0; i < L.nd; ++i) {
    const int r = cfg->rd[i];
    if (r == JOLT_FULL) {
      if (i != L.nd - 1) return JOLT_ERR_INVALID;
      L.rd[i] = L.D;
      L.hasFullD = 1;
    } else {
      if (r < 1 || r > 64 || r >= L.D) return JOLT_ERR_INVALID;
      if (i > 0 && r <= cfg->rd[i - 1]) return JOLT_ERR_INVALID;
      L.rd[i] = r;
      L.ndt = i + 1;
      L.RD = r;
    }
  }
  for (int i = 0; i < L.nb; ++i) {
    const int b = cfg->b[i];
    if (!(b == 0 || b == 2 || b == 4 || b == 8)) return JOLT_ERR_INVALID;
    if (i > 0 && b <= cfg->b[i - 1]) return JOLT_ERR_INVALID;
    L.b[i] = b;
  }
  L.token_mode = cfg->token_mode;
  if (L.token_mode != JOLT_TOKEN_EXACT && L.token_mode != JOLT_TOKEN_RANDOMIZED)
    return JOLT_ERR_INVALID;
  if (cfg->cost_model != JOLT_COST_FORMULA && cfg->cost_model != JOLT_COST_SERIALIZED)
    return JOLT_ERR_INVALID;
  if (cfg->align < 16 || cfg->align % 16) return JOLT_ERR_INVALID;
  L.cost_model = cfg->cost_model;
  L.align = cfg->align;
  L.block = cfg->quant_block;
  L.power_iters = cfg->power_iters;
  L.ncand = L.nT * L.nd * L.nb;

  const int RT = L.RT, RD = L.RD, H = L.H, T = L.T, D = L.D;
  if (RT > 0 && L.token_mode == JOLT_TOKEN_RANDOMIZED) {
    if (cfg->oversample < 0 || cfg->power_iters < 0 || cfg->power_iters > 16)
      return JOLT_ERR_INVALID;
    L.ell = RT + cfg->oversample;
    if (L.ell > 64 || L.ell > T) return JOLT_ERR_INVALID;
    if (!(L.ell == 32 || L.ell == 40 || L.ell == 48 || L.ell == 64)) return JOLT_ERR_INVALID;
    // the sketch Z = A Omega needs at least ell independent columns of A
    for (int i = 0; i < L.nd; ++i)
      if ((long long)H * L.rd[i] < L.ell) return JOLT_ERR_INVALID;
  }
  if (RT > 0 && L.token_mode == JOLT_TOKEN_EXACT) {
    if (T <= 128) {
      L.L = T;
    } else {
      // block width: twice the largest token rank, one of the widths the
      // row-parallel triangular solve is built for
      int w = 2 * RT < 32 ? 32 : (2 * RT <= 40 ? 40 : (2 * RT <= 48 ? 48 : 64));
      if (w < RT + 8) w = 64;
      if (w > T) return JOLT_ERR_INVALID;
      L.L = w;
    }
  }
  // feature Gram split: groups of hg heads with hg * T <= 4096 rows
  int hg = 1;
  for (int d = 1; d <= H; ++d)
    if (H % d == 0 && (long long)d * T <= 4096) hg = d;
  L.nsplit = H / hg;
  L.chunk = hg;
  L.ks = 1;
  for (int d = 1; d <= 4; ++d)
    if (T % d == 0 && T / d >= 32) L.ks = d;
  L.hs = 1;
  for (int d = 1; d <= 16; ++d)
    if (H % d == 0) L.hs = d;
  L.tile_rows = 8192 / D;     // sweep CTA rows: 8 warps x (32 / (D/16)) row groups x 2 rows
  L.ntiles = H * ((T + L.tile_rows - 1) / L.tile_rows);

  const int Lw = (L.token_mode == JOLT_TOKEN_EXACT) ? L.L : L.ell;
  const bool iter = RT > 0 && (L.token_mode == JOLT_TOKEN_RANDOMIZED || T > 128);
  const int Dmax = L.hasFullD ? D : RD;
  size_t off = 0;
  auto sect = [&](size_t bytes) {
    off = align_up(off, 256);
    const size_t o = off;
    off += bytes;
    return o;
  };
  L.o_status = sect(256);
  L.o_Sd = sect((size_t)D * D * 4);
  L.o_Sd64 = sect((size_t)D * D * 8);
  L.o_Sdp = sect((size_t)L.nsplit * D * D * 4);
  L.o_evd = sect((size_t)D * 4);
  L.o_Vd = sect((size_t)D * D * 4);
  L.o_Ud16 = sect((size_t)D * RD * 2);
  L.o_QUd = sect((size_t)RD * D * 4);
  L.o_Y = sect((size_t)H * T * RD * 4);
  L.o_Y16 = sect((size_t)H * T * RD * 2);
  const bool exact = RT > 0 && L.token_mode == JOLT_TOKEN_EXACT;
  const bool svtc = exact && T > 128 && L.L == 64;
  L.o_Yt = (svtc && RD > 0) ? sect((size_t)2 * T * RD * H * 4) : 0;
  L.o_Hs = (L.dtype == JOLT_BF16 && D == 128) ? sect((size_t)D * D * 2) : 0;
  L.o_Vs3 = (L.dtype == JOLT_BF16 && D == 128 && RD > 0 && RD <= 32) ? sect((size_t)3 * 32 * D * 2)
                                                                      : 0;
  L.o_Ub3 = (L.dtype == JOLT_BF16 && D == 128 && RT > 0 && RT <= 32 && L.nd * 96 <= 512)
                ? sect((size_t)T * 512 * 2)
                : 0;
  L.o_UT32 = sect((size_t)L.nd * T * RT * 4);
  L.o_UT16 = sect((size_t)L.nd * T * RT * 2);
  L.o_tokev = sect((size_t)L.nd * RT * 4);
  L.o_cap = sect((size_t)L.nd * RT * 8);
  {
    const bool fl = RT > 0 && L.token_mode == JOLT_TOKEN_RANDOMIZED && L.dtype == JOLT_BF16 &&
                    D == 128;
    L.o_Bx = fl ? sect((size_t)H * 512 * D * 2) : 0;
    L.o_Qs = fl ? sect((size_t)T * 512 * 2) : 0;
    L.o_C = fl ? sect((size_t)H * D * 160 * 4) : 0;
  }
  L.o_G32 = sect((size_t)L.nd * H * RT * D * 4);
  L.o_G16 = sect((size_t)L.nd * H * RT * D * 2);
  // rotated chain rows of the sweep; the encoder reuses the first two slots
  L.o_W = sect((size_t)(L.nd > 2 ? L.nd : 2) * H * RT * D * 4);
  L.o_part = sect((size_t)L.ntiles * (L.ncand + 1) * 4);
  L.o_P = sect((RT > 0 && L.token_mode == JOLT_TOKEN_RANDOMIZED) ? (size_t)H * Dmax * L.ell * 4 : 0);
  L.unit_bytes = align_up(off, 256);

  // one token problem per feature rank
  L.nprob = RT > 0 ? L.nd : 0;
  off = 0;
  L.p_status = sect(256);
  L.p_flag = sect(256);
  L.p_ST = exact ? sect((size_t)T * T * 4) : 0;
  L.p_STs = svtc ? sect((size_t)T * T * 4) : 0;
  L.p_Vs = svtc ? sect((size_t)2 * T * 64 * 4) : 0;   // V^T and its tf32 low part
  const size_t blk = iter ? (size_t)T * Lw * 4 : 0;
  L.p_V = sect(blk);
  L.p_Z = sect(blk);
  L.p_V2 = sect(blk);
  L.p_Z2 = sect(blk);
  const size_t sq = RT > 0 ? (size_t)Lw * Lw * 4 : 0;
  const int nparts = L.ks > L.hs ? L.ks : L.hs;
  L.p_Hm = sect(sq * nparts);
  L.p_Wm = sect(sq);
  L.p_Gram = sect(sq * L.ks);
  L.p_Rinv = sect(sq);
  L.p_theta = sect((size_t)(Lw > T ? Lw : T) * 4);
  L.p_UT = sect((size_t)T * RT * 4);
  L.p_ev = sect((size_t)RT * 4);
  L.prob_bytes = L.nprob > 0 ? align_up(off, 256) : 0;
  L.unit_total = L.unit_bytes + (size_t)L.nprob * L.prob_bytes;
  *Lp = L;
  return JOLT_OK;
}

int64_t cost_formula(int H, int T, int D, int rT, int rd, int b, int block, int align) {
  const long long n = (long long)H * T * D;
  long long c = (long long)align_up((size_t)(2LL * H * ((long long)rT * T + (long long)rd * rT + (long long)rd * D)), align);
  if (b > 0) c += (long long)align_up((size_t)(b * n / 8), align) + (long long)align_up((size_t)(2 * n / block), align);
  return c + JOLT_HEADER_BYTES;
}

}  // namespace jolt

using namespace jolt;

static cudaStream_t S(void* s) { return (cudaStream_t)s; }

static bool ws_ok(const Layout& L, int n, const void* ws, size_t ws_bytes) {
  return ws && ((uintptr_t)ws % 256 == 0) && ws_bytes >= (size_t)n * L.unit_total;
}

extern "C" {

int jolt_num_candidates(const jolt_config* cfg) {
  Layout L;
  if (make_layout(cfg, &L) != JOLT_OK) return 0;
  return L.ncand;
}

size_t jolt_workspace_size(const jolt_config* cfg) {
  Layout L;
  if (make_layout(cfg, &L) != JOLT_OK) return 0;
  return L.unit_total;
}

jolt_status jolt_factor_group(const jolt_config* cfg, int n_units, const void* X,
                              const float* sketch, void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  jolt_status s = make_layout(cfg, &L);
  if (s != JOLT_OK) return s;
  if (n_units < 1 || n_units > 65535 || !X) return JOLT_ERR_INVALID;
  if (L.token_mode == JOLT_TOKEN_RANDOMIZED && L.RT > 0 && !sketch) return JOLT_ERR_INVALID;
  if (!ws_ok(L, n_units, ws, ws_bytes)) return JOLT_ERR_WORKSPACE;
  return factor_run(L, n_units, X, sketch, (char*)ws, S(stream));
}

jolt_status jolt_sweep_candidates(const jolt_config* cfg, int n_units, const void* X,
                                  const int8_t* signs, void* ws, size_t ws_bytes, double* dist,
                                  int64_t* cost, void* stream) {
  Layout L;
  jolt_status s = make_layout(cfg, &L);
  if (s != JOLT_OK) return s;
  if (n_units < 1 || n_units > 65535 || !X || !signs || !dist || !cost) return JOLT_ERR_INVALID;
  if (!ws_ok(L, n_units, ws, ws_bytes)) return JOLT_ERR_WORKSPACE;
  return sweep_run(L, n_units, X, signs, (char*)ws, dist, cost, S(stream));
}

jolt_status jolt_allocate(int n_units, int n_cand, const double* dist, const int64_t* cost,
                          int64_t budget, int align, int32_t* choice, double* lambda,
                          int32_t* status, void* stream) {
  if (n_units < 1 || n_cand < 1 || !dist || !cost || !choice || !lambda || !status || align < 1)
    return JOLT_ERR_INVALID;
  return alloc_run(n_units, n_cand, dist, cost, budget, align, choice, lambda, status, S(stream));
}

jolt_status jolt_set_sweep_events(void* start, void* stop) {
  if ((start == nullptr) != (stop == nullptr)) return JOLT_ERR_INVALID;
  g_sweep_ev[0] = start;
  g_sweep_ev[1] = stop;
  return JOLT_OK;
}

jolt_status jolt_set_factor_events(void* const* events) {
  for (int i = 0; i < 5; ++i) g_factor_ev[i] = events ? events[i] : nullptr;
  return JOLT_OK;
}

jolt_status jolt_set_solver_limits(int max_sweeps, int max_subspace_blocks) {
  if (max_sweeps < 0 || max_subspace_blocks < 0) return JOLT_ERR_INVALID;
  set_max_sweeps(max_sweeps);
  set_subspace_blocks(max_subspace_blocks);
  return JOLT_OK;
}

jolt_status jolt_model_candidates(const jolt_config* cfg, int n_units, const void* ws,
                                  size_t ws_bytes, const double* eps2_host, double* dist,
                                  void* stream) {
  Layout L;
  jolt_status s = make_layout(cfg, &L);
  if (s != JOLT_OK) return s;
  if (n_units < 1 || n_units > 65535 || !eps2_host || !dist) return JOLT_ERR_INVALID;
  if (!ws_ok(L, n_units, ws, ws_bytes)) return JOLT_ERR_WORKSPACE;
  for (int i = 0; i < L.nb; ++i)
    if (L.b[i] > 0 && !(eps2_host[i] >= 0.0)) return JOLT_ERR_INVALID;
  return model_table_run(L, n_units, (const char*)ws, eps2_host, dist, S(stream));
}

jolt_status jolt_calibrate_eps2(const float* rows, int n_rows, int D, const int32_t* bits_host,
                                int n_b, double* scratch, double* eps2, void* stream) {
  if (!rows || n_rows < 1 || !(D == 32 || D == 64 || D == 128) || !bits_host || n_b < 1 ||
      n_b > 4 || !scratch || !eps2)
    return JOLT_ERR_INVALID;
  for (int i = 0; i < n_b; ++i)
    if (!(bits_host[i] == 0 || bits_host[i] == 2 || bits_host[i] == 4 || bits_host[i] == 8))
      return JOLT_ERR_INVALID;
  return eps2_run(rows, n_rows, D, bits_host, n_b, scratch, eps2, S(stream));
}

jolt_status jolt_refine(int n_units, int n_cand, const double* dist, const int64_t* cost,
                        int64_t budget, int32_t* choice, int32_t* n_swaps, void* stream) {
  if (n_units < 1 || n_cand < 1 || n_cand > JOLT_MAX_CAND || !dist || !cost || !choice)
    return JOLT_ERR_INVALID;
  if ((long long)n_units * n_cand > (1LL << 30)) return JOLT_ERR_INVALID;
  return refine_run(n_units, n_cand, dist, cost, budget, choice, n_swaps, S(stream));
}

jolt_status jolt_allocate_uniform(int n_units, int n_cand, const double* dist,
                                  const int64_t* cost, int64_t budget, const int32_t* cand_host,
                                  int n_list, int32_t* choice, int32_t* status, void* stream) {
  if (n_units < 1 || n_cand < 1 || n_cand > JOLT_MAX_CAND || !dist || !cost || !choice ||
      !status || !cand_host || n_list < 1 || n_list > JOLT_MAX_CAND)
    return JOLT_ERR_INVALID;
  for (int i = 0; i < n_list; ++i)
    if (cand_host[i] < 0 || cand_host[i] >= n_cand) return JOLT_ERR_INVALID;
  return uniform_run(n_units, n_cand, dist, cost, budget, cand_host, n_list, choice, status,
                     S(stream));
}

size_t jolt_blob_bytes(const jolt_config* cfg, int cand) {
  Layout L;
  if (make_layout(cfg, &L) != JOLT_OK || cand < 0 || cand >= L.ncand) return 0;
  int iT, id, ib;
  cand_split(L, cand, &iT, &id, &ib);
  jolt_blob_desc d;
  blob_layout(L.H, L.T, L.D, L.rT[iT], L.rd[id], L.b[ib], L.block, L.align, &d);
  return d.bytes;
}

jolt_status jolt_encode(const jolt_config* cfg, int n_units, const void* X, const int8_t* signs,
                        const void* ws, size_t ws_bytes, const int32_t* choice_host, void* blob,
                        size_t blob_stride, jolt_blob_desc* desc_out, void* stream) {
  Layout L;
  jolt_status s = make_layout(cfg, &L);
  if (s != JOLT_OK) return s;
  if (n_units < 1 || !X || !signs || !choice_host || !blob || !desc_out) return JOLT_ERR_INVALID;
  if (((uintptr_t)blob % 256) || (blob_stride % 256)) return JOLT_ERR_INVALID;
  if (!ws_ok(L, n_units, ws, ws_bytes)) return JOLT_ERR_WORKSPACE;
  return encode_run(L, n_units, X, signs, (const char*)ws, choice_host, (char*)blob, blob_stride,
                    desc_out, S(stream));
}

jolt_status jolt_decode(int n_units, const jolt_blob_desc* desc, const void* blob,
                        size_t blob_stride, void* xhat, jolt_dtype out_dtype, void* stream) {
  if (n_units < 1 || !desc || !blob || !xhat) return JOLT_ERR_INVALID;
  if (out_dtype != JOLT_F32 && out_dtype != JOLT_BF16) return JOLT_ERR_INVALID;
  if (((uintptr_t)blob % 256) || (blob_stride % 256)) return JOLT_ERR_INVALID;
  const int H = desc[0].H, T = desc[0].T, D = desc[0].D;
  if (H <= 0 || T <= 0 || !(D == 32 || D == 64 || D == 128)) return JOLT_ERR_INVALID;
  for (int u = 0; u < n_units; ++u) {
    const jolt_blob_desc& d = desc[u];
    if (d.H != H || d.T != T || d.D != D || d.block != D) return JOLT_ERR_INVALID;
    if (!(d.rT == T || (d.rT >= 1 && d.rT <= 64 && d.rT < T))) return JOLT_ERR_INVALID;
    if (!(d.rd == D || (d.rd >= 1 && d.rd <= 64 && d.rd < D))) return JOLT_ERR_INVALID;
    if (!(d.b == 0 || d.b == 2 || d.b == 4 || d.b == 8)) return JOLT_ERR_INVALID;
    if (d.bytes > blob_stride) return JOLT_ERR_INVALID;
    if (d.off_G + 2ull * H * d.rT * d.rd > d.bytes) return JOLT_ERR_INVALID;
    if (d.b > 0 && d.off_codes + (unsigned long long)H * T * D * d.b / 8 > d.bytes)
      return JOLT_ERR_INVALID;
  }
  return decode_run(n_units, desc, (const char*)blob, blob_stride, xhat, out_dtype, S(stream));
}

jolt_status jolt_decode_status(void* stream) {
  int v = 0;
  const jolt_status s = decode_tc_status(&v, S(stream));
  if (s != JOLT_OK) return s;
  return (v & ST_TIMEOUT) ? JOLT_ERR_CUDA : JOLT_OK;
}

size_t jolt_attend_workspace_size(int n_groups, int H, int T, int D, int nq) {
  if (n_groups < 1 || H < 1 || T < 1 || D < 1 || nq < 1 || nq > JOLT_ATTN_MAX_Q) return 0;
  return attend_ws_bytes(n_groups, H, T, D, nq);
}

jolt_status jolt_attend(int n_groups, const jolt_blob_desc* desc, const void* blob,
                        size_t blob_stride, const float* q, int nq, float scale, void* ws,
                        size_t ws_bytes, float* out, void* stream) {
  if (n_groups < 1 || !desc || !blob || !q || !ws || !out) return JOLT_ERR_INVALID;
  if (nq < 1 || nq > JOLT_ATTN_MAX_Q || !(scale == scale) || scale > 3.4e38f || scale < -3.4e38f)
    return JOLT_ERR_INVALID;
  if (((uintptr_t)blob % 256) || (blob_stride % 256) || ((uintptr_t)q % 16) ||
      ((uintptr_t)out % 16) || ((uintptr_t)ws % 16))
    return JOLT_ERR_INVALID;
  const int H = desc[0].H, T = desc[0].T, D = desc[0].D;
  if (H <= 0 || H > 65535 || T <= 0 || !(D == 32 || D == 64 || D == 128)) return JOLT_ERR_INVALID;
  for (int u = 0; u < 2 * n_groups; ++u) {
    const jolt_blob_desc& d = desc[u];
    if (d.H != H || d.T != T || d.D != D || d.block != D) return JOLT_ERR_INVALID;
    if (!(d.rT == T || (d.rT >= 1 && d.rT <= 64 && d.rT < T))) return JOLT_ERR_INVALID;
    if (!(d.rd == D || (d.rd >= 1 && d.rd <= 64 && d.rd < D))) return JOLT_ERR_INVALID;
    if (!(d.b == 0 || d.b == 2 || d.b == 4 || d.b == 8)) return JOLT_ERR_INVALID;
    if (d.bytes > blob_stride) return JOLT_ERR_INVALID;
    if (d.off_G + 2ull * H * d.rT * d.rd > d.bytes) return JOLT_ERR_INVALID;
    if (d.rT < T && d.off_UT + 2ull * T * d.rT > d.bytes) return JOLT_ERR_INVALID;
    if (d.rd < D && d.off_Ud + 2ull * D * d.rd > d.bytes) return JOLT_ERR_INVALID;
    if ((d.off_UT % 4) || (d.off_Ud % 4) || (d.off_G % 4)) return JOLT_ERR_INVALID;
    if (d.b > 0) {
      if (d.off_scale + 2ull * H * T > d.bytes) return JOLT_ERR_INVALID;
      if (d.off_codes + (unsigned long long)H * T * D * d.b / 8 > d.bytes) return JOLT_ERR_INVALID;
      if ((d.off_scale % 2) || (d.off_codes % 16)) return JOLT_ERR_INVALID;
    }
  }
  if (ws_bytes < attend_ws_bytes(n_groups, H, T, D, nq)) return JOLT_ERR_WORKSPACE;
  return attend_run(n_groups, desc, (const char*)blob, blob_stride, q, nq, scale, (float*)ws, out,
                    S(stream));
}

size_t jolt_admit_workspace_size(int n_units, int H, int tau, int D) {
  if (n_units < 1 || H < 1 || tau < 1 || !(D == 32 || D == 64 || D == 128)) return 0;
  return (size_t)n_units * admit_ws_unit_bytes(H, tau, D);
}

jolt_status jolt_admit(int n_units, const jolt_blob_desc* desc_in, const void* blob_in,
                       size_t stride_in, const void* X_new, jolt_dtype x_dtype, int tau,
                       int align, void* ws, size_t ws_bytes, void* blob_out, size_t stride_out,
                       jolt_blob_desc* desc_out, void* stream) {
  if (n_units < 1 || !desc_in || !blob_in || !X_new || !ws || !blob_out || !desc_out)
    return JOLT_ERR_INVALID;
  if (x_dtype != JOLT_F32 && x_dtype != JOLT_BF16) return JOLT_ERR_INVALID;
  if (tau < 1 || align < 16 || align > 4096 || (align & (align - 1))) return JOLT_ERR_INVALID;
  if (((uintptr_t)blob_in % 256) || (stride_in % 256) || ((uintptr_t)blob_out % 256) ||
      (stride_out % 256) || ((uintptr_t)ws % 256) ||
      ((uintptr_t)X_new % (x_dtype == JOLT_BF16 ? 2 : 4)))
    return JOLT_ERR_INVALID;
  const uintptr_t i0 = (uintptr_t)blob_in, i1 = i0 + (uintptr_t)n_units * stride_in;
  const uintptr_t o0 = (uintptr_t)blob_out, o1 = o0 + (uintptr_t)n_units * stride_out;
  if (i0 < o1 && o0 < i1) return JOLT_ERR_INVALID;
  const int H = desc_in[0].H, T = desc_in[0].T, D = desc_in[0].D;
  if (H <= 0 || H > 65535 || T <= 0 || !(D == 32 || D == 64 || D == 128)) return JOLT_ERR_INVALID;
  if ((long long)T + tau > (1LL << 30)) return JOLT_ERR_INVALID;
  for (int u = 0; u < n_units; ++u) {
    const jolt_blob_desc& d = desc_in[u];
    if (d.H != H || d.T != T || d.D != D || d.block != D) return JOLT_ERR_INVALID;
    if (!(d.rT == T || (d.rT >= 1 && d.rT <= 64 && d.rT < T))) return JOLT_ERR_INVALID;
    if (!(d.rd == D || (d.rd >= 1 && d.rd <= 64 && d.rd < D))) return JOLT_ERR_INVALID;
    if (!(d.b == 0 || d.b == 2 || d.b == 4 || d.b == 8)) return JOLT_ERR_INVALID;
    if (d.bytes > stride_in) return JOLT_ERR_INVALID;
    if (d.off_G + 2ull * H * d.rT * d.rd > d.bytes) return JOLT_ERR_INVALID;
    if (d.rT < T && d.off_UT + 2ull * T * d.rT > d.bytes) return JOLT_ERR_INVALID;
    if (d.rd < D && d.off_Ud + 2ull * D * d.rd > d.bytes) return JOLT_ERR_INVALID;
    if ((d.off_UT % 4) || (d.off_Ud % 4) || (d.off_G % 4)) return JOLT_ERR_INVALID;
    if (d.b > 0) {
      if (d.off_scale + 2ull * H * T > d.bytes) return JOLT_ERR_INVALID;
      if (d.off_codes + (unsigned long long)H * T * D * d.b / 8 > d.bytes) return JOLT_ERR_INVALID;
      if ((d.off_scale % 4) || (d.off_codes % 4)) return JOLT_ERR_INVALID;
    }
  }
  if (ws_bytes < (size_t)n_units * admit_ws_unit_bytes(H, tau, D)) return JOLT_ERR_WORKSPACE;
  return admit_run(n_units, desc_in, (const char*)blob_in, stride_in, X_new, x_dtype, tau, align,
                   (char*)ws, (char*)blob_out, stride_out, desc_out, S(stream));
}

jolt_status jolt_read_status(const jolt_config* cfg, int n_units, void* ws, void* stream) {
  Layout L;
  jolt_status s = make_layout(cfg, &L);
  if (s != JOLT_OK) return s;
  if (n_units < 1 || !ws) return JOLT_ERR_INVALID;
  cudaStream_t st = S(stream);
  JOLT_CUDA_TRY(cudaStreamSynchronize(st));
  int worst = 0;
  for (int u = 0; u < n_units; ++u) {
    int v = 0;
    JOLT_CUDA_TRY(cudaMemcpy(&v, (char*)ws + (size_t)u * L.unit_bytes + L.o_status, sizeof(int),
                             cudaMemcpyDeviceToHost));
    worst |= v;
  }
  JOLT_CUDA_TRY(cudaMemset2DAsync((char*)ws + L.o_status, L.unit_bytes, 0, sizeof(int), n_units, st));
  JOLT_CUDA_TRY(cudaStreamSynchronize(st));
  if (worst & ST_TIMEOUT) return JOLT_ERR_CUDA;
  if (worst & ST_NONFINITE) return JOLT_ERR_NONFINITE;
  if (worst & (ST_NOCONVERGE | ST_NOTPD)) return JOLT_ERR_NOCONVERGE;
  return JOLT_OK;
}

const char* jolt_status_string(jolt_status s) {
  switch (s) {
    case JOLT_OK: return "ok";
    case JOLT_ERR_INVALID: return "invalid argument";
    case JOLT_ERR_INFEASIBLE: return "budget below the cheapest allocation";
    case JOLT_ERR_NONFINITE: return "non-finite value in the input";
    case JOLT_ERR_NOCONVERGE: return "eigensolver did not converge";
    case JOLT_ERR_WORKSPACE: return "workspace missing or too small";
    case JOLT_ERR_CUDA: return "CUDA runtime error";
    case JOLT_ERR_TOO_LARGE: return "batch beyond the static scratch of the no-allocation call";
  }
  return "unknown status";
}

uint64_t jolt_launch_count(void) { return (uint64_t)g_launches; }

}  // extern "C"
