// kvq_host.cu -- the C ABI of libkvq (include/kvq.h): argument validation,
// the byte layout of a layer buffer, the decode split plan, and launches.
// Host code only; every step of the method runs in the kernels.
#include <cmath>
#include <cstring>

#include "kvq_internal.cuh"

using namespace kvq;

namespace {

constexpr uint64_t kAlign = 256;
// The host-only split plan (kvq_layout_query / kvq_decode_plan run without a
// device) aims at this many CTAs, about two waves of 3 resident CTAs on 152
// SMs; a decode then widens it to the SM count and occupancy of the device
// it runs on (fill_waves below).
constexpr int kTargetCtas = 152 * 6;

uint64_t align_up(uint64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool valid_lut(const float* lut) {
  for (int i = 0; i < 8; ++i) {
    if (!std::isfinite(lut[i])) return false;
    if (i && !(lut[i] > lut[i - 1])) return false;
  }
  return true;
}

kvq_status make_geometry(const kvq_config* c, Geometry* g) {
  if (!c || !g) return KVQ_ERR_INVALID_ARG;
  if (c->batch < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1 || c->head_dim < 1 || c->max_tokens < 1)
    return KVQ_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (c->n_sink < 0 || c->n_recent < 0 || c->split_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if ((c->v_hadamard != 0 && c->v_hadamard != 1) || (c->k_pre_rope != 0 && c->k_pre_rope != 1))
    return KVQ_ERR_INVALID_ARG;
  if (!(c->softmax_scale >= 0.0f) || !std::isfinite(c->softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (c->k_pre_rope && !(c->rope_theta > 0.0f && std::isfinite(c->rope_theta))) return KVQ_ERR_INVALID_ARG;
  if (c->position_offset < 0 || (int64_t)c->position_offset + c->max_tokens >= (int64_t)1 << 31)
    return KVQ_ERR_INVALID_ARG;
  if ((c->hybrid_groups != 0 && c->hybrid_groups != 1) || (c->k_channel_norm != 0 && c->k_channel_norm != 1) ||
      c->k_group_channels < 0)
    return KVQ_ERR_INVALID_ARG;
  if (c->k_channel_norm && !c->k_group_channels) return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (c->n_q_heads / c->n_kv_heads > kMaxGQA) return KVQ_ERR_UNSUPPORTED;
  const int64_t ns = (int64_t)c->batch * c->n_kv_heads;
  if (ns > 65535) return KVQ_ERR_UNSUPPORTED;

  const bool fp16 = c->k_bits == 16 || c->v_bits == 16;
  auto uni = [](int b) { return b == 2 || b == 4 || b == 8; };
  if (fp16) {
    if (c->k_bits != 16 || c->v_bits != 16) return KVQ_ERR_UNSUPPORTED;
    if (c->v_hadamard) return KVQ_ERR_UNSUPPORTED;
  } else if (c->k_bits == 3 || c->v_bits == 3) {
    if (c->k_bits != 3 || c->v_bits != 3) return KVQ_ERR_UNSUPPORTED;
    if (c->outliers_per_vector < 0 || c->outliers_per_vector > kMaxOutliers) return KVQ_ERR_INVALID_ARG;
    if (!valid_lut(c->k_lut) || !valid_lut(c->v_lut)) return KVQ_ERR_INVALID_ARG;
  } else if (!uni(c->k_bits) || !uni(c->v_bits)) {
    return KVQ_ERR_UNSUPPORTED;
  }
  const bool uniform = !fp16 && c->k_bits != 3;
  if (c->hybrid_groups && !uniform) return KVQ_ERR_UNSUPPORTED;
  if (c->k_group_channels) {
    // InnerQ K: 64-channel per-token groups, served by the persistent decode
    if (c->k_group_channels != 64 || !uniform || c->v_group_channels != 64 || c->k_pre_rope)
      return KVQ_ERR_UNSUPPORTED;
  }
  if (!fp16) {
    if (c->k_group_tokens != kGroupTokens) return KVQ_ERR_UNSUPPORTED;
    if (c->v_bits != 3 && c->v_group_channels != 32 && c->v_group_channels != 64 &&
        c->v_group_channels != 128)
      return KVQ_ERR_UNSUPPORTED;
    if (c->split_tokens % kGroupTokens) return KVQ_ERR_INVALID_ARG;
  } else if (c->split_tokens % kGroupTokens) {
    return KVQ_ERR_INVALID_ARG;
  }

  const int32_t tot = c->kv_heads_total ? c->kv_heads_total : c->n_kv_heads;
  if (tot < c->n_kv_heads || (int64_t)c->batch * tot > 65535) return KVQ_ERR_INVALID_ARG;
  if (c->kv_head_index) {
    if (c->n_kv_heads > 256) return KVQ_ERR_UNSUPPORTED;
    for (int i = 0; i < c->n_kv_heads; ++i) {
      const int32_t h = c->kv_head_index[i];
      if (h < 0 || h >= tot) return KVQ_ERR_INVALID_ARG;
      for (int j = 0; j < i; ++j)
        if (c->kv_head_index[j] == h) return KVQ_ERR_INVALID_ARG;
    }
  }
  if (c->sm_budget < 0) return KVQ_ERR_INVALID_ARG;
  g->sm_budget = c->sm_budget;
  g->Hkv_tot = tot;
  g->Hq_tot = tot * (c->n_q_heads / c->n_kv_heads);
  g->has_map = c->kv_head_index ? 1 : 0;
  for (int i = 0; i < 256; ++i) g->kvmap[i] = (int16_t)(c->kv_head_index && i < c->n_kv_heads ? c->kv_head_index[i] : i);
  g->B = c->batch;
  g->Hq = c->n_q_heads;
  g->Hkv = c->n_kv_heads;
  g->g = c->n_q_heads / c->n_kv_heads;
  g->NS = (int)ns;
  g->d = c->head_dim;
  g->fp16_mode = fp16 ? 1 : 0;
  g->kb = c->k_bits;
  g->vb = c->v_bits;
  g->gk = kGroupTokens;
  g->gv = (c->v_bits == 3 || fp16) ? kHeadDim : c->v_group_channels;
  g->nvg = kHeadDim / g->gv;
  g->hadamard = c->v_hadamard;
  g->pre_rope = c->k_pre_rope;
  g->nout = (c->k_bits == 3) ? c->outliers_per_vector : 0;
  g->rope_theta = c->rope_theta;
  g->pos_offset = c->position_offset;
  g->gkc = c->k_group_channels;
  g->nkg = c->k_group_channels ? kHeadDim / c->k_group_channels : 0;
  g->hybrid = c->hybrid_groups;
  g->knorm = c->k_channel_norm;
  if (fp16) {
    g->S = 0;
    g->R = 0;
    g->ring = c->max_tokens;
    g->qcap = 0;
    g->krow = g->vrow = 0;
  } else {
    g->S = c->n_sink;
    g->R = c->n_recent;
    g->ring = c->n_recent + kGroupTokens;
    const int64_t rest = (int64_t)c->max_tokens - c->n_sink - c->n_recent;
    g->qcap = rest > 0 ? (int)(kGroupTokens * (rest / kGroupTokens)) : 0;
    g->krow = kHeadDim * c->k_bits / 8;
    g->vrow = kHeadDim * c->v_bits / 8;
  }
  g->gcap = g->qcap / kGroupTokens;
  return KVQ_OK;
}

// Sink tokens present, quantized tokens and window tokens at T tokens.
void counts(const Geometry& g, int T, int* S_eff, int* Nq, int* W) { window_counts(g, T, S_eff, Nq, W); }

kvq_status build_layout(const kvq_config* c, const Geometry& g, kvq_layout* L) {
  std::memset(L, 0, sizeof(*L));
  uint64_t off = 0;
  auto put = [&](kvq_region& r, uint64_t bytes) {
    r.offset = off;
    r.bytes = bytes;
    off = align_up(off + bytes);
  };
  const uint64_t NS = (uint64_t)g.NS, Q = (uint64_t)g.qcap, d = kHeadDim;
  put(L->k_codes, NS * Q * g.krow);
  put(L->k_scales, g.kb == 3 ? NS * Q * 4 : g.gkc ? NS * Q * g.nkg * 4 : NS * (uint64_t)g.gcap * d * 4);
  put(L->v_codes, NS * Q * g.vrow);
  put(L->v_scales, g.vb == 3 ? NS * Q * 4 : NS * Q * g.nvg * 4);
  put(L->k_sink, NS * g.S * d * 2);
  put(L->v_sink, NS * g.S * d * 2);
  put(L->k_ring, NS * (uint64_t)g.ring * d * 2);
  put(L->v_ring, NS * (uint64_t)g.ring * d * 2);
  const uint64_t k = (uint64_t)g.nout;
  const bool nuq = g.kb == 3;
  put(L->k_csr_rowptr, nuq ? NS * (Q + 1) * 4 : 0);
  put(L->k_csr_col, nuq ? NS * Q * k : 0);
  put(L->k_csr_val, nuq ? NS * Q * k * 2 : 0);
  put(L->v_csr_rowptr, nuq ? NS * (Q + 1) * 4 : 0);
  put(L->v_csr_col, nuq ? NS * Q * k : 0);
  put(L->v_csr_val, nuq ? NS * Q * k * 2 : 0);
  put(L->k_norm, g.knorm ? NS * d * 4 : 0);
  put(L->rows, 2 * kMaxRaggedRows * 4);  // a ragged append's per-row counts
  L->layer_bytes = off;
  L->max_splits = kMaxQSplits + 1;
  L->ring_slots = g.ring;
  L->q_cap = g.qcap;
  // split counters, partial (m, l) and accumulators, then a ragged decode's row tables
  const uint64_t ws = align_up(align_up(NS * 4) + align_up(NS * (uint64_t)L->max_splits * g.g * 2 * 4) +
                               NS * (uint64_t)L->max_splits * g.g * d * 4) +
                      kRaggedTableBytes;
  L->workspace_bytes = ws;
  (void)c;
  return KVQ_OK;
}

void layer_ptrs(const kvq_layout& L, void* base, LayerPtrs* P) {
  auto at = [&](const kvq_region& r) { return (void*)((char*)base + r.offset); };
  P->k_codes = (uint8_t*)at(L.k_codes);
  P->k_scales = (uint32_t*)at(L.k_scales);
  P->v_codes = (uint8_t*)at(L.v_codes);
  P->v_scales = (uint32_t*)at(L.v_scales);
  P->k_sink = (uint16_t*)at(L.k_sink);
  P->v_sink = (uint16_t*)at(L.v_sink);
  P->k_ring = (uint16_t*)at(L.k_ring);
  P->v_ring = (uint16_t*)at(L.v_ring);
  P->k_rowptr = (int32_t*)at(L.k_csr_rowptr);
  P->k_col = (uint8_t*)at(L.k_csr_col);
  P->k_val = (uint16_t*)at(L.k_csr_val);
  P->v_rowptr = (int32_t*)at(L.v_csr_rowptr);
  P->v_col = (uint8_t*)at(L.v_csr_col);
  P->v_val = (uint16_t*)at(L.v_csr_val);
  P->k_norm = (float*)at(L.k_norm);
  P->rows = (int*)at(L.rows);
}

// Split plan: how many splits cover `ngroups` 32-token groups of NS streams.
void split_groups(int ngroups, int NS, int split_tokens, int* n_split, int* gps) {
  if (ngroups <= 0) {
    *n_split = 0;
    *gps = 1;
    return;
  }
  int per;
  if (split_tokens > 0) {
    per = split_tokens / kGroupTokens;
  } else {
    int want = (kTargetCtas + NS - 1) / NS;
    if (want < 1) want = 1;
    if (want > kMaxQSplits) want = kMaxQSplits;
    if (want > ngroups) want = ngroups;
    per = (ngroups + want - 1) / want;
  }
  if (per < 1) per = 1;
  if ((ngroups + per - 1) / per > kMaxQSplits) per = (ngroups + kMaxQSplits - 1) / kMaxQSplits;
  *gps = per;
  *n_split = (ngroups + per - 1) / per;
}

struct Plan {
  int S_eff, Nq, W, n_qsplit, n_split, gps, fp16_tps;
};

Plan make_plan(const Geometry& g, int T, int split_tokens) {
  Plan p{};
  counts(g, T, &p.S_eff, &p.Nq, &p.W);
  if (g.fp16_mode) {
    int n, per;
    split_groups((T + kGroupTokens - 1) / kGroupTokens, g.NS, split_tokens, &n, &per);
    p.n_qsplit = 0;
    p.n_split = n;
    p.gps = per;
    p.fp16_tps = per * kGroupTokens;
  } else {
    int n, per;
    split_groups(p.Nq / kGroupTokens, g.NS, split_tokens, &n, &per);
    p.n_qsplit = n;
    p.gps = per;
    p.n_split = n + ((p.S_eff + p.W) > 0 ? 1 : 0);
    p.fp16_tps = p.S_eff + p.W;
  }
  return p;
}

}  // namespace

namespace kvq {

kvq_status make_geometry_for(const kvq_config* cfg, Geometry* g) { return make_geometry(cfg, g); }

kvq_status decode_setup(const kvq_config* cfg, const void* layer_buf, int32_t tokens, const uint16_t* q,
                        uint16_t* out, float* lse, DecodeParams* pp, bool* persistent, uint64_t* layout_ws) {
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (!layer_buf || !q || !out) return KVQ_ERR_INVALID_ARG;
  if (tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (tokens > cfg->max_tokens) return KVQ_ERR_CAPACITY;
  if (((uintptr_t)layer_buf | (uintptr_t)q | (uintptr_t)out) % 16) return KVQ_ERR_INVALID_ARG;
  kvq_layout L;
  build_layout(cfg, g, &L);
  Plan pl = make_plan(g, tokens, cfg->split_tokens);
  DecodeParams& p = *pp;
  std::memset(&p, 0, sizeof(p));
  p.geo = g;
  layer_ptrs(L, const_cast<void*>(layer_buf), &p.L);
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.T = tokens;
  p.S_eff = pl.S_eff;
  p.Nq = pl.Nq;
  p.W = pl.W;
  p.n_qsplit = pl.n_qsplit;
  p.n_split = pl.n_split;
  p.auto_split = cfg->split_tokens <= 0 ? 1 : 0;
  p.gps = pl.gps;
  p.fp16_tokens_per_split = pl.fp16_tps;
  const double sm = cfg->softmax_scale > 0.0f ? (double)cfg->softmax_scale : 1.0 / std::sqrt((double)kHeadDim);
  p.q_scale = (float)(sm * 1.4426950408889634);  // log2(e): softmax in base 2
  p.hadamard_c = (float)(1.0 / std::sqrt((double)kHeadDim));
  for (int i = 0; i < 8; ++i) {
    p.k_lut_off[i] = cfg->k_lut[i] - cfg->k_lut[0];
    p.v_lut_off[i] = cfg->v_lut[i] - cfg->v_lut[0];
  }
  if (g.pre_rope)  // RoPE frequencies (only the pre-RoPE paths read them)
    for (int i = 0; i < kHeadDim / 2; ++i)
      p.theta[i] = std::pow((double)cfg->rope_theta, -2.0 * i / (double)kHeadDim);
  *persistent = persist_eligible(g);
  *layout_ws = L.workspace_bytes;
  return KVQ_OK;
}

// Scratch of one decode: split counters [NS], then (m, l) and accumulators
// of every partial result (NS x splits for the split kernel; one per
// (warp, stream) piece for the persistent kernel).
static uint64_t scratch_bytes(const Geometry& g, uint64_t slots, uint64_t* cnt_bytes, uint64_t* ml_bytes) {
  *cnt_bytes = align_up((uint64_t)g.NS * 4);
  *ml_bytes = align_up(slots * g.g * 2 * 4);
  return *cnt_bytes + *ml_bytes + slots * g.g * kHeadDim * 4;
}

static uint64_t slots_of(const DecodeParams& p, bool persistent) {
  return persistent ? (uint64_t)p.nwarps + p.geo.NS : (uint64_t)p.geo.NS * p.n_split;
}

// Split kernel: with the split count left to the library, raise the
// quantized splits so that the grid (NS x splits CTAs) fills whole waves of
// the kernel's resident CTAs -- a grid of 1.5 waves leaves half the GPU idle
// during its last wave, and every CTA streams the same number of groups.
static cudaError_t fill_waves(DecodeParams* p) {
  if (!p->auto_split || p->n_qsplit <= 0) return cudaSuccess;
  int sms = 0, occ = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  if (p->geo.sm_budget > 0 && p->geo.sm_budget < sms) sms = p->geo.sm_budget;
  e = launch_decode(*p, nullptr, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaSuccess;
  p->gps = fill_waves_plan(p->geo.NS, (long long)sms * occ, p->Nq / kGroupTokens, p->gps, &p->n_qsplit,
                           &p->n_split);
  return cudaSuccess;
}

kvq_status decode_plan_device(DecodeParams* p, bool persistent, uint64_t* need, bool widen) {
  *need = 0;
  if (persistent) {
    uint64_t ignored;
    if (plan_persist(*p, &ignored) != cudaSuccess) return KVQ_ERR_CUDA;
  } else {
    if (widen && fill_waves(p) != cudaSuccess) return KVQ_ERR_CUDA;
    if (p->n_split <= 1) return KVQ_OK;
  }
  uint64_t c, m;
  *need = scratch_bytes(p->geo, slots_of(*p, persistent), &c, &m);
  return KVQ_OK;
}

kvq_status decode_launch(DecodeParams* p, bool persistent, void* ws, cudaStream_t st) {
  uint64_t c, m;
  if (persistent || p->n_split > 1) {
    scratch_bytes(p->geo, slots_of(*p, persistent), &c, &m);
    p->counters = (uint32_t*)ws;
    p->part_ml = (float*)((char*)ws + c);
    p->part_acc = (float*)((char*)ws + c + m);
  }
  const cudaError_t e = persistent ? launch_decode_persist(*p, st) : launch_decode(*p, st);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "token count exceeds capacity";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

kvq_status kvq_layout_query(const kvq_config* cfg, kvq_layout* out) {
  if (!cfg || !out) return KVQ_ERR_INVALID_ARG;
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  return build_layout(cfg, g, out);
}

kvq_status kvq_decode_plan(const kvq_config* cfg, int32_t tokens, int32_t* splits_per_stream,
                           int32_t* quantized_splits) {
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (tokens > cfg->max_tokens) return KVQ_ERR_CAPACITY;
  Plan p = make_plan(g, tokens, cfg->split_tokens);
  if (splits_per_stream) *splits_per_stream = p.n_split;
  if (quantized_splits) *quantized_splits = p.n_qsplit;
  return KVQ_OK;
}

kvq_status kvq_decode_path(const kvq_config* cfg, int32_t tokens, int32_t* persistent, int32_t* gq_slots) {
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (tokens > cfg->max_tokens) return KVQ_ERR_CAPACITY;
  if (persistent) *persistent = persist_eligible(g) ? 1 : 0;
  if (gq_slots) *gq_slots = g.g <= 1 ? 1 : g.g <= 2 ? 2 : g.g <= 4 ? 4 : 8;
  return KVQ_OK;
}

kvq_status kvq_context_shard(const kvq_config* cfg, int32_t tokens, int32_t n_shards, int32_t shard,
                             kvq_config* shard_cfg, int32_t* first_token, int32_t* shard_tokens) {
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (!shard_cfg || !first_token || !shard_tokens) return KVQ_ERR_INVALID_ARG;
  if (n_shards < 1 || n_shards > 65536 || shard < 0 || shard >= n_shards || tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (tokens > cfg->max_tokens) return KVQ_ERR_CAPACITY;
  // shard r starts at the quantized-group boundary S + 32 floor(r ng / n)
  // (fp16 cache: the 32-token block boundary), shard 0 at token 0
  int S_eff, Nq, W;
  counts(g, tokens, &S_eff, &Nq, &W);
  const int64_t ng = g.fp16_mode ? tokens / kGroupTokens : Nq / kGroupTokens;
  const int64_t base = g.fp16_mode ? 0 : g.S;
  auto bound = [&](int64_t r) -> int64_t {
    if (r <= 0) return 0;
    if (r >= n_shards) return tokens;
    const int64_t b = base + kGroupTokens * (r * ng / n_shards);
    return b < tokens ? b : tokens;
  };
  const int64_t a = bound(shard), b = bound(shard + 1);
  const bool last = shard == n_shards - 1;
  *shard_cfg = *cfg;
  shard_cfg->n_sink = shard == 0 ? cfg->n_sink : 0;
  shard_cfg->n_recent = last ? cfg->n_recent : 0;
  shard_cfg->position_offset = cfg->position_offset + (int32_t)a;
  const int64_t cap = last ? (int64_t)cfg->max_tokens - a : b - a;
  shard_cfg->max_tokens = (int32_t)(cap > 0 ? cap : 1);
  *first_token = (int32_t)a;
  *shard_tokens = (int32_t)(b - a);
  return KVQ_OK;
}

kvq_status kvq_fit_nuq_lut(const uint16_t* x, int64_t n_vectors, int32_t head_dim, int32_t outliers,
                           int32_t hadamard, int32_t max_iters, void* workspace, uint64_t ws_bytes, float* lut_out,
                           int32_t* info_out, kvq_stream_t stream) {
  if (head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (!x || !lut_out || n_vectors < 1 || outliers < 0 || outliers > kMaxOutliers || (hadamard != 0 && hadamard != 1) ||
      max_iters < 1 || max_iters > 1000000)
    return KVQ_ERR_INVALID_ARG;
  if (((uintptr_t)x % 8) || ((uintptr_t)lut_out % 4) || ((uintptr_t)info_out % 4)) return KVQ_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < KVQ_NUQ_FIT_WORKSPACE_BYTES || ((uintptr_t)workspace % 8)) return KVQ_ERR_WORKSPACE;
  const cudaError_t e = launch_nuq_fit(x, n_vectors, outliers, hadamard, max_iters, workspace, lut_out, info_out,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_merge_attn(int32_t n_parts, int64_t rows, int32_t head_dim, const uint16_t* outs,
                          const float* lses, uint16_t* out, float* lse_out, kvq_stream_t stream) {
  if (n_parts < 1 || rows < 0) return KVQ_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (rows == 0) return KVQ_OK;
  if (!outs || !lses || !out) return KVQ_ERR_INVALID_ARG;
  if (((uintptr_t)outs | (uintptr_t)out) % 8 || ((uintptr_t)lses | (uintptr_t)lse_out) % 4) return KVQ_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_merge_attn(n_parts, rows, outs, lses, out, lse_out, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_append(const kvq_config* cfg, void* layer_buf, int32_t tokens_before,
                      const uint16_t* k_new, const uint16_t* v_new, int32_t n_new,
                      kvq_stream_t stream) {
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (!layer_buf || !k_new || !v_new) return KVQ_ERR_INVALID_ARG;
  if (tokens_before < 0 || n_new < 1) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)tokens_before + n_new > cfg->max_tokens) return KVQ_ERR_CAPACITY;
  if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)layer_buf) % 16) return KVQ_ERR_INVALID_ARG;
  kvq_layout L;
  build_layout(cfg, g, &L);

  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.geo = g;
  layer_ptrs(L, layer_buf, &p.L);
  p.k_new = k_new;
  p.v_new = v_new;
  p.tokens_before = tokens_before;
  p.n_new = n_new;
  int s0, w0, s1, w1;
  counts(g, tokens_before, &s0, &p.nq_before, &w0);
  counts(g, tokens_before + n_new, &s1, &p.nq_after, &w1);
  p.first_group = p.nq_before / kGroupTokens;
  p.hadamard_c = (float)(1.0 / std::sqrt((double)kHeadDim));
  for (int i = 0; i < 8; ++i) {
    p.k_lut[i] = cfg->k_lut[i];
    p.v_lut[i] = cfg->v_lut[i];
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // InnerQ key normalisation: fixed by the first append into an empty cache
  if (g.knorm && tokens_before == 0 && launch_key_norm(p, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  const int n_groups = (p.nq_after - p.nq_before) / kGroupTokens;
  if (n_groups > 0) {
    if (launch_append_quantize(p, n_groups, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  if (launch_append_window(p, window_copies_max(p), cs) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_append_ragged(const kvq_config* cfg, void* layer_buf, const int32_t* tokens_before,
                             const int32_t* n_new, const uint16_t* k_new, const uint16_t* v_new, int32_t n_stride,
                             kvq_stream_t stream) {
  Geometry g;
  kvq_status st = make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (!layer_buf || !k_new || !v_new || !tokens_before || !n_new) return KVQ_ERR_INVALID_ARG;
  if (g.B > kMaxRaggedRows) return KVQ_ERR_UNSUPPORTED;
  if (n_stride < 1) return KVQ_ERR_INVALID_ARG;
  int most = 0;
  for (int b = 0; b < g.B; ++b) {
    if (tokens_before[b] < 0 || n_new[b] < 0 || n_new[b] > n_stride) return KVQ_ERR_INVALID_ARG;
    if ((int64_t)tokens_before[b] + n_new[b] > cfg->max_tokens) return KVQ_ERR_CAPACITY;
    most = n_new[b] > most ? n_new[b] : most;
  }
  if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)layer_buf) % 16) return KVQ_ERR_INVALID_ARG;
  kvq_layout L;
  build_layout(cfg, g, &L);

  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.geo = g;
  layer_ptrs(L, layer_buf, &p.L);
  p.k_new = k_new;
  p.v_new = v_new;
  p.n_new = n_stride;
  p.ragged = 1;
  // plan on the host arrays, launch on their device copy in the layer buffer
  p.row_before = tokens_before;
  p.row_new = n_new;
  bool any_first = false;
  int n_groups = 0;
  for (int b = 0; b < g.B; ++b) {
    any_first = any_first || tokens_before[b] == 0;
    const RowAppend ra = row_append(p, b * g.Hkv);
    const int ng = (ra.nq_after - ra.nq_before) / kGroupTokens;
    n_groups = ng > n_groups ? ng : n_groups;
  }
  const int ncopy = window_copies_max(p);
  p.hadamard_c = (float)(1.0 / std::sqrt((double)kHeadDim));
  for (int i = 0; i < 8; ++i) {
    p.k_lut[i] = cfg->k_lut[i];
    p.v_lut[i] = cfg->v_lut[i];
  }
  if (most == 0) return KVQ_OK;  // no row appends anything
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (launch_append_rows(tokens_before, n_new, g.B, p.L.rows, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  p.row_before = p.L.rows;
  p.row_new = p.L.rows + kMaxRaggedRows;
  // InnerQ key normalisation of the rows that append into an empty cache
  if (g.knorm && any_first && launch_key_norm(p, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  if (n_groups > 0 && launch_append_quantize(p, n_groups, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  if (launch_append_window(p, ncopy, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_decode_attn_ragged(const kvq_config* cfg, const void* layer_buf, const int32_t* tokens,
                                  const uint16_t* q, uint16_t* out, float* lse, void* workspace, uint64_t ws_bytes,
                                  kvq_stream_t stream) {
  if (!cfg || !tokens) return KVQ_ERR_INVALID_ARG;
  if (cfg->batch < 1) return KVQ_ERR_INVALID_ARG;
  if (cfg->batch > kMaxRaggedRows) return KVQ_ERR_UNSUPPORTED;
  int T = 0;
  for (int b = 0; b < cfg->batch; ++b) {
    if (tokens[b] < 1) return KVQ_ERR_INVALID_ARG;
    if (tokens[b] > cfg->max_tokens) return KVQ_ERR_CAPACITY;
    T = tokens[b] > T ? tokens[b] : T;
  }
  DecodeParams p;
  bool persistent = false;
  uint64_t layout_ws = 0;
  kvq_status st = decode_setup(cfg, layer_buf, T, q, out, lse, &p, &persistent, &layout_ws);
  if (st != KVQ_OK) return st;
  // the same kernel as kvq_decode_attn: the persistent schedule lays every
  // stream's own items end to end; the split kernel is planned for the
  // longest row and every stream takes its row's counts
  // plan on host tables, launch on their copy in the workspace (behind the
  // scratch the plan needs)
  RaggedTables ht;
  std::memset(&ht, 0, sizeof(ht));
  for (int b = 0; b < cfg->batch; ++b) ht.tokens[b] = tokens[b];
  p.ragged = 1;
  p.row_tokens = ht.tokens;
  p.row_j0 = ht.j0;
  p.row_x0 = ht.x0;
  if (!workspace || ws_bytes < layout_ws || ((uintptr_t)workspace % 16)) return KVQ_ERR_WORKSPACE;
  uint64_t need = 0;
  st = decode_plan_device(&p, persistent, &need);
  if (st != KVQ_OK) return st;
  const uint64_t tab_off = align_up(need);
  if (ws_bytes < tab_off + kRaggedTableBytes) return KVQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->batch <= kInlineRows) {
    // few rows: the tables travel in the launch parameters
    for (int b = 0; b <= cfg->batch; ++b) {
      if (b < cfg->batch) p.in_tokens[b] = ht.tokens[b];
      p.in_j0[b] = ht.j0[b];
      p.in_x0[b] = ht.x0[b];
    }
    p.rows_inline = 1;
  } else {
    RaggedTables* dt = reinterpret_cast<RaggedTables*>(static_cast<char*>(workspace) + tab_off);
    if (launch_ragged_tables(ht, dt, cs) != cudaSuccess) return KVQ_ERR_CUDA;
    p.row_tokens = dt->tokens;
    p.row_j0 = dt->j0;
    p.row_x0 = dt->x0;
  }
  return decode_launch(&p, persistent, workspace, cs);
}

kvq_status kvq_decode_attn(const kvq_config* cfg, const void* layer_buf, int32_t tokens,
                           const uint16_t* q, uint16_t* out, float* lse, void* workspace,
                           uint64_t ws_bytes, kvq_stream_t stream) {
  DecodeParams p;
  bool persistent = false;
  uint64_t layout_ws = 0;
  kvq_status st = decode_setup(cfg, layer_buf, tokens, q, out, lse, &p, &persistent, &layout_ws);
  if (st != KVQ_OK) return st;
  // the persistent kernel always needs scratch; ask for the layout's bound
  // before touching the device
  if (persistent && (!workspace || ws_bytes < layout_ws || ((uintptr_t)workspace % 16))) return KVQ_ERR_WORKSPACE;
  uint64_t need = 0;
  st = decode_plan_device(&p, persistent, &need);
  if (st != KVQ_OK) return st;
  if (need > 0 && (!workspace || ws_bytes < need || ((uintptr_t)workspace % 16))) return KVQ_ERR_WORKSPACE;
  return decode_launch(&p, persistent, workspace, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
