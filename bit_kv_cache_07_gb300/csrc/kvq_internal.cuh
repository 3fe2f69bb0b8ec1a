// kvq_internal.cuh -- geometry, parameter blocks and small device helpers
// shared by the host layer (kvq_host.cu) and the kernels (kvq_append.cu,
// kvq_decode*.cu).  Not part of the public ABI (that is include/kvq.h).
#pragma once

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;      // d supported by the kernels
constexpr int kGroupTokens = 32;   // G_K supported by the kernels (one warp lane per token)
constexpr int kMaxQSplits = 64;    // quantized split-K chunks per stream (decode)
constexpr int kMaxOutliers = 8;    // non-uniform outliers per vector
constexpr int kMaxGQA = 8;         // query heads per KV head
constexpr int kThreads = 128;      // threads per CTA of the append and split-decode kernels
// Sequences of different lengths in one call (kvq_decode_attn_ragged,
// kvq_append_ragged): at most this many batch rows.
constexpr int kMaxRaggedRows = 256;
// Ragged decodes of at most this many rows carry their row tables in the
// launch parameters (no copy kernel ahead of the decode).
constexpr int kInlineRows = 16;

// Geometry derived once on the host from a kvq_config.
struct Geometry {
  int B, Hq, Hkv, g, NS, d;
  int kb, vb, gk, gv, nvg;
  int S, R, ring, qcap, gcap;
  int krow, vrow;
  int hadamard, pre_rope, nout, fp16_mode;
  int pos_offset;  // absolute position of the cache's first token (RoPE)
  int gkc, nkg;    // InnerQ K: channels per per-token K group (0: per-channel K), groups per token
  int hybrid;      // InnerQ: symmetric / asymmetric choice per uniform group
  int knorm;       // InnerQ: per-channel key normalisation
  float rope_theta;
  // per-head pairs: this cache holds Hkv of the layer's Hkv_tot KV heads
  // (kvmap[h] = the layer head of cache head h when has_map)
  int Hkv_tot, Hq_tot, has_map;
  int16_t kvmap[256];
  int sm_budget;  // decode: SMs this cache's work may use (0: all)
};

// The layer's KV head of this cache's head h.
__host__ __device__ inline int layer_head(const Geometry& G, int h) { return G.has_map ? G.kvmap[h] : h; }
// Row block of cache stream s in the layer's [B][Hkv_tot] inputs (k_new, v_new).
__host__ __device__ inline size_t in_stream(const Geometry& G, int s) {
  const int b = s / G.Hkv, h = s - b * G.Hkv;
  return (size_t)b * G.Hkv_tot + layer_head(G, h);
}
// Row of query head r of cache KV head hk, batch row b, in q / out / lse.
__host__ __device__ inline size_t q_row(const Geometry& G, int b, int hk, int r) {
  return (size_t)b * G.Hq_tot + (size_t)layer_head(G, hk) * G.g + r;
}

// Typed pointers into one layer buffer.
struct LayerPtrs {
  uint8_t* k_codes;
  uint32_t* k_scales;   // half2 {min, scale} words
  uint8_t* v_codes;
  uint32_t* v_scales;
  uint16_t* k_sink;
  uint16_t* v_sink;
  uint16_t* k_ring;
  uint16_t* v_ring;
  int32_t* k_rowptr;
  uint8_t* k_col;
  uint16_t* k_val;
  int32_t* v_rowptr;
  uint8_t* v_col;
  uint16_t* v_val;
  float* k_norm;        // [NS][d] InnerQ key normalisation
  int* rows;            // [2][kMaxRaggedRows] a ragged append's per-row tokens before / appended
};

// Window rule at T tokens (host and device): sinks present, quantized
// tokens (whole 32-token groups past the sinks, leaving at least R), and the
// fp16 window; an fp16 cache keeps every token in its window.
__host__ __device__ inline void window_counts(const Geometry& g, int T, int* S_eff, int* Nq, int* W) {
  if (g.fp16_mode) {
    *S_eff = 0;
    *Nq = 0;
    *W = T;
    return;
  }
  *S_eff = T < g.S ? T : g.S;
  const int rest = T - g.S - g.R;
  *Nq = rest > 0 ? kGroupTokens * (rest / kGroupTokens) : 0;
  *W = T - *S_eff - *Nq;
}


struct AppendParams {
  Geometry geo;
  LayerPtrs L;
  const uint16_t* k_new;  // [NS][n_new][d]
  const uint16_t* v_new;
  int tokens_before;      // T0
  int n_new;
  int nq_before;          // quantized tokens before the call
  int nq_after;           // quantized tokens after the call
  int first_group;        // first group flushed by this call
  float hadamard_c;       // fp32(1/sqrt(d))
  float k_lut[8];
  float v_lut[8];
  // ragged append: batch row b appends row_new[b] tokens (the first of its
  // n_new input rows) after row_before[b] (device copies in the layer
  // buffer at launch; host arrays while the host plans); n_new is then the
  // inputs' token stride
  int ragged;
  const int* row_before;
  const int* row_new;
};

// The append of batch row b (stream s = b Hkv + h): tokens before, tokens
// appended, quantized tokens before and after, first group flushed.
struct RowAppend {
  int before, n, nq_before, nq_after, first_group;
};
__host__ __device__ inline RowAppend row_append(const AppendParams& p, int s) {
  RowAppend r;
  if (!p.ragged) {
    r.before = p.tokens_before;
    r.n = p.n_new;
    r.nq_before = p.nq_before;
    r.nq_after = p.nq_after;
    r.first_group = p.first_group;
    return r;
  }
  const int b = s / p.geo.Hkv;
  r.before = p.row_before[b];
  r.n = p.row_new[b];
  int se, w;
  window_counts(p.geo, r.before, &se, &r.nq_before, &w);
  window_counts(p.geo, r.before + r.n, &se, &r.nq_after, &w);
  r.first_group = r.nq_before / kGroupTokens;
  return r;
}

// fp16 tokens a stream's append copies into sink / window slots: the call's
// tokens j < a (sinks; every token of an fp16 cache) and j >= b (past the
// quantized part).
__host__ __device__ inline void window_split(const AppendParams& p, const RowAppend& ra, int* a, int* b) {
  const Geometry& G = p.geo;
  if (G.fp16_mode) {
    *a = *b = ra.n;
    return;
  }
  auto clamp = [](int x, int lo, int hi) { return x < lo ? lo : x > hi ? hi : x; };
  *a = clamp(G.S - ra.before, 0, ra.n);
  *b = clamp(G.S + ra.nq_after - ra.before, *a, ra.n);
}
// The most tokens any stream copies (the grid's token extent).
__host__ __device__ inline int window_copies_max(const AppendParams& p) {
  int most = 0;
  const int rows = p.ragged ? p.geo.B : 1;
  for (int r = 0; r < rows; ++r) {
    const RowAppend ra = row_append(p, r * p.geo.Hkv);
    int a, b;
    window_split(p, ra, &a, &b);
    most = max(most, a + (ra.n - b));
  }
  return most;
}

// Division by a divisor that is fixed for a launch, without a hardware
// divide: floor(x / d) = (x * m) >> sh for 0 <= x < 2^56, where
// sh = 56 + ceil(log2 d) and m = ceil(2^sh / d) (< 2^57).  Writing
// m = (2^sh + e) / d with 0 <= e < d <= 2^(sh - 56), the product is
// x / d + x e / (d 2^sh) and x e < 2^sh keeps the excess below 1 / d, which
// is less than the distance from x / d to the next integer: the floor is
// exact.  (Round-up reciprocal multiplication, Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994.)
struct FastDiv {
  unsigned long long m;
  int sh;
};
inline FastDiv make_fastdiv(long long d) {  // host; d >= 1
  int l = 0;
  while ((1ull << l) < (unsigned long long)d) ++l;
  const int sh = 56 + l;
  const unsigned __int128 num = (unsigned __int128)1 << sh;
  return FastDiv{(unsigned long long)((num + (unsigned __int128)(d - 1)) / (unsigned __int128)d), sh};
}
__host__ __device__ inline long long fastdiv_mulshift(long long x, const FastDiv& f) {
  const unsigned long long ux = (unsigned long long)x;
#ifdef __CUDA_ARCH__
  const unsigned long long hi = __umul64hi(ux, f.m), lo = ux * f.m;
#else
  const unsigned __int128 pr = (unsigned __int128)ux * f.m;
  const unsigned long long hi = (unsigned long long)(pr >> 64), lo = (unsigned long long)pr;
#endif
  return (long long)(f.sh >= 64 ? hi >> (f.sh - 64) : (hi << (64 - f.sh)) | (lo >> f.sh));
}
constexpr long long kFastDivLimit = 1ll << 56;  // dividends must stay below this

struct DecodeParams {
  Geometry geo;
  LayerPtrs L;
  const uint16_t* q;      // [B][Hq][d]
  uint16_t* out;          // [B][Hq][d]
  float* lse;             // [B][Hq] or null
  uint32_t* counters;     // [NS] split tickets (workspace)
  float* part_ml;         // [NS][n_split][g][2]   (m in log2 units, l)
  float* part_acc;        // [NS][n_split][g][d]
  int T;                  // tokens attended
  int S_eff;              // sink tokens present
  int Nq;                 // quantized tokens
  int W;                  // window tokens
  int n_qsplit;           // splits over quantized groups
  int n_split;            // total splits per stream (quantized + fp16)
  int gps;                // quantized groups per split
  int auto_split;         // 1: split count chosen by the library (config split_tokens = 0)
  int fp16_tokens_per_split;
  float q_scale;          // softmax_scale * log2(e)
  float hadamard_c;       // fp32(1/sqrt(d))
  float k_lut_off[8];     // L_i - L_0 (fp32)
  float v_lut_off[8];
  double theta[kHeadDim / 2];  // RoPE frequencies rope_theta^(-2i/d), fp64
  // persistent schedule (tensor-core / fp16 kernels): the streams' work items
  // -- ng quantized 32-token groups, then nt fp16 items of a few tokens each --
  // laid end to end, weighted (wq, wt: see plan_persist), cut into nwarps
  // equal ranges.
  int ng, nt, n_items;
  int nwarps;
  long long wq, wt, wstream, wtot;
  FastDiv fd_n_items, fd_wq, fd_wt, fd_wstream, fd_wtot, fd_nwarps;  // for idiv
  // ragged decode: tokens of batch row b (T = their maximum); for the
  // persistent schedule, the first item and the first weight position of
  // row b's first stream (entry B: the totals).  Device copies in the
  // workspace at launch (RaggedTables), host arrays while the host plans.
  int ragged;
  const int* row_tokens;
  long long* row_j0;
  long long* row_x0;
  // ragged decode of at most kInlineRows rows: the same tables inline (the
  // kernels read them from the parameters; the pointers above stay the
  // host's)
  int rows_inline;
  int in_tokens[kInlineRows];
  long long in_j0[kInlineRows + 1], in_x0[kInlineRows + 1];
};

// The row tables a ragged decode reads: inline or through the pointers.
__host__ __device__ inline const int* rows_tokens(const DecodeParams& p) {
  return p.rows_inline ? p.in_tokens : p.row_tokens;
}
__host__ __device__ inline const long long* rows_j0(const DecodeParams& p) {
  return p.rows_inline ? p.in_j0 : p.row_j0;
}
__host__ __device__ inline const long long* rows_x0(const DecodeParams& p) {
  return p.rows_inline ? p.in_x0 : p.row_x0;
}

// A ragged decode's per-row tables, as the host builds them and as a copy
// kernel writes them into the workspace (behind the split counters and
// partial results).
struct RaggedTables {
  int tokens[kMaxRaggedRows];
  long long j0[kMaxRaggedRows + 1];
  long long x0[kMaxRaggedRows + 1];
};
constexpr uint64_t kRaggedTableBytes = (sizeof(RaggedTables) + 255) / 256 * 256;

constexpr int kPersistF16Tokens = 8;  // fp16 tokens per item of the persistent schedule

// One stream's part of the persistent schedule: its first item and weight
// position, quantized groups, fp16 items and tokens, and the window counts
// its fp16 tokens are addressed with.  Uniform calls: the same for every
// stream; ragged ones: from the stream's batch row.
struct StreamSpan {
  long long first, x0, wstream;
  int ng, nt, n_items, k1, S_eff, Nq;
};
__host__ __device__ inline StreamSpan row_span(const DecodeParams& p, int b) {
  StreamSpan r;
  int W;
  window_counts(p.geo, rows_tokens(p)[b], &r.S_eff, &r.Nq, &W);
  r.k1 = r.S_eff + W;
  r.ng = p.geo.fp16_mode ? 0 : r.Nq / kGroupTokens;
  r.nt = (r.k1 + kPersistF16Tokens - 1) / kPersistF16Tokens;
  r.n_items = r.ng + r.nt;
  r.wstream = (long long)r.ng * p.wq + (long long)r.nt * p.wt;
  r.first = rows_j0(p)[b];
  r.x0 = rows_x0(p)[b];
  return r;
}
// RG: the ragged schedule (compile-time in the kernel, p.ragged on the host)
template <bool RG>
__host__ __device__ inline StreamSpan stream_span_t(const DecodeParams& p, int s) {
  if constexpr (!RG) {
    StreamSpan r;
    r.first = (long long)s * p.n_items;
    r.x0 = (long long)s * p.wstream;
    r.wstream = p.wstream;
    r.ng = p.ng;
    r.nt = p.nt;
    r.n_items = p.n_items;
    r.k1 = p.S_eff + p.W;
    r.S_eff = p.S_eff;
    r.Nq = p.Nq;
    return r;
  }
  const int b = s / p.geo.Hkv, h = s - b * p.geo.Hkv;
  StreamSpan r = row_span(p, b);
  r.first += (long long)h * r.n_items;
  r.x0 += (long long)h * r.wstream;
  return r;
}
__host__ __device__ inline StreamSpan stream_span(const DecodeParams& p, int s) {
  return p.ragged ? stream_span_t<true>(p, s) : stream_span_t<false>(p, s);
}
// Ragged schedule: the last row whose first entry in `tab` (row_j0 or
// row_x0) is <= v (rows of a ragged call hold at least one item each).
__host__ __device__ inline int row_at(const long long* tab, int rows, long long v) {
  int lo = 0, hi = rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

#ifdef __CUDACC__
// row_at by a whole warp (every lane calls it with the same arguments): each
// lane tests up to 8 rows (rows <= 256) with independent loads, and the rows
// at or below v are counted by ballot (the entries increase strictly).
__device__ __forceinline__ int row_at_warp(const long long* tab, int rows, long long v, int lane) {
  int cnt = 0;
  for (int r0 = 0; r0 < rows; r0 += 32) {
    const int r = r0 + lane;
    cnt += __popc(__ballot_sync(0xffffffffu, r < rows && tab[r] <= v));
  }
  return cnt - 1;
}
#endif

// floor(x / d) for 0 <= x < 2^56: the device multiplies and shifts (a
// 64-bit integer division is a long serial emulation there, and fp64 is a
// narrow pipe on this GPU); the host divides exactly.
__host__ __device__ inline long long idiv(long long x, long long d, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  (void)d;
  return fastdiv_mulshift(x, f);
#else
  (void)f;
  return x / d;
#endif
}

// floor(x / d) for 0 <= x, 0 < d: in 32 bits when both fit (the usual case;
// a 64-bit integer division is a long serial emulation on the device).
__host__ __device__ inline long long udiv(long long x, long long d) {
  if (((unsigned long long)x | (unsigned long long)d) >> 32 == 0) return (long long)((unsigned)x / (unsigned)d);
  return x / d;
}

// Ragged persistent schedule (host): every row's first item and weight
// position, the totals, and whether any stream holds quantized groups.
inline void plan_rows(DecodeParams& p, long long* items, bool* any_groups) {
  p.row_j0[0] = p.row_x0[0] = 0;
  *any_groups = false;
  for (int b = 0; b < p.geo.B; ++b) {
    const StreamSpan r = row_span(p, b);
    p.row_j0[b + 1] = p.row_j0[b] + (long long)p.geo.Hkv * r.n_items;
    p.row_x0[b + 1] = p.row_x0[b] + (long long)p.geo.Hkv * r.wstream;
    *any_groups = *any_groups || r.ng > 0;
  }
  *items = p.row_j0[p.geo.B];
  p.wtot = p.row_x0[p.geo.B];
}

// Persistent-schedule arithmetic shared by host and device: items laid
// stream after stream, weighted by wq and wt; RG selects the ragged
// schedule at compile time (the wrappers below take p.ragged).
// (Dividends stay below 2^56: plan_persist checks (wtot + 1) (nwarps + 1) < 2^56.)
// Ragged schedule, item j of batch row b: its stream s and index k.
__host__ __device__ inline void locate_in_row(const DecodeParams& p, long long j, int b, int* s, int* k) {
  const StreamSpan r = row_span(p, b);
  const long long h = udiv(j - r.first, r.n_items);
  *s = b * p.geo.Hkv + (int)h;
  *k = (int)(j - r.first - h * r.n_items);
}
// Item j's stream s and index k within it.
template <bool RG>
__host__ __device__ inline void locate_item_t(const DecodeParams& p, long long j, int* s, int* k) {
  if constexpr (!RG) {
    const long long ss = idiv(j, p.n_items, p.fd_n_items);
    *s = (int)ss;
    *k = (int)(j - ss * p.n_items);
  } else {
    locate_in_row(p, j, row_at(rows_j0(p), p.geo.B, j), s, k);
  }
}
template <bool RG>
__host__ __device__ inline long long item_pos_t(const DecodeParams& p, long long j) {
  if constexpr (RG) {
    int s, k;
    locate_item_t<true>(p, j, &s, &k);
    const StreamSpan r = stream_span_t<true>(p, s);
    return r.x0 + (k <= r.ng ? k * p.wq : r.ng * p.wq + (k - r.ng) * p.wt);
  } else {
    const long long s = idiv(j, p.n_items, p.fd_n_items), k = j - s * p.n_items;
    return s * p.wstream + (k <= p.ng ? k * p.wq : p.ng * p.wq + (k - p.ng) * p.wt);
  }
}
// Start weight of item k of the stream whose span is r (item_pos_t of the
// stream's first item + k, without locating the stream).
__host__ __device__ inline long long item_pos_in(const DecodeParams& p, const StreamSpan& r, int k) {
  return r.x0 + (k <= r.ng ? (long long)k * p.wq : (long long)r.ng * p.wq + (long long)(k - r.ng) * p.wt);
}
// Ragged schedule: the first item whose start weight is >= x, for x in
// batch row b's weights [row_x0[b], row_x0[b + 1]).
__host__ __device__ inline long long first_item_in_row(const DecodeParams& p, long long x, int b) {
  const StreamSpan r = row_span(p, b);
  const long long h = udiv(x - r.x0, r.wstream), rem = x - r.x0 - h * r.wstream;
  const long long f = r.first + h * r.n_items;  // the stream's first item
  if (rem == 0) return f;
  long long k;
  if (rem <= (long long)r.ng * p.wq) k = udiv(rem + p.wq - 1, p.wq);
  else k = r.ng + udiv(rem - (long long)r.ng * p.wq + p.wt - 1, p.wt);
  return f + k;  // k == n_items: the next stream's first item
}
// First item whose start weight is >= x (x in [0, wtot]).
template <bool RG>
__host__ __device__ inline long long first_item_at_t(const DecodeParams& p, long long x) {
  if constexpr (RG) {
    if (x >= p.wtot) return rows_j0(p)[p.geo.B];
    return first_item_in_row(p, x, row_at(rows_x0(p), p.geo.B, x));
  } else {
    long long s = idiv(x, p.wstream, p.fd_wstream), rem = x - s * p.wstream, k;
    if (rem == 0) return s * p.n_items;
    if (rem <= p.ng * p.wq) k = idiv(rem + p.wq - 1, p.wq, p.fd_wq);
    else k = p.ng + idiv(rem - p.ng * p.wq + p.wt - 1, p.wt, p.fd_wt);
    if (k >= p.n_items) return (s + 1) * p.n_items;
    return s * p.n_items + k;
  }
}
__host__ __device__ inline void locate_item(const DecodeParams& p, long long j, int* s, int* k) {
  if (p.ragged) locate_item_t<true>(p, j, s, k);
  else locate_item_t<false>(p, j, s, k);
}
__host__ __device__ inline long long item_pos(const DecodeParams& p, long long j) {
  return p.ragged ? item_pos_t<true>(p, j) : item_pos_t<false>(p, j);
}
__host__ __device__ inline long long first_item_at(const DecodeParams& p, long long x) {
  return p.ragged ? first_item_at_t<true>(p, x) : first_item_at_t<false>(p, x);
}
// Warp i covers weight [x_i, x_{i+1}), x_i = floor(i * wtot / nwarps).
__host__ __device__ inline long long warp_x(const DecodeParams& p, long long i) {
  return idiv(i * p.wtot, p.nwarps, p.fd_nwarps);
}
__host__ __device__ inline int owner_of(const DecodeParams& p, long long pos) {
  return (int)(idiv((pos + 1) * p.nwarps + p.wtot - 1, p.wtot, p.fd_wtot) - 1);
}

// ----------------------------------------------------- RoPE group anchors
// For RoPE frequency theta (radians per position) and the absolute position
// S of the first quantized token: the per-group angle step 32 theta / (2 pi)
// in turns, split into three parts of at most 8 significant bits (exact
// products with a group index below 2^16) and the rest (below 2^-21 of the
// step), and the anchor of group 0 (position S) in turns.  fp64, once per
// CTA on the device.
__host__ __device__ inline void anchor_step(double theta, long long S, float4* v4, float* c0) {
  const double turns = theta / (2.0 * 3.14159265358979323846);
  double v = turns * kGroupTokens, parts[3];
  for (int i = 0; i < 3; ++i) {
    parts[i] = 0.0;
    if (v > 0.0) {
      const double q = ldexp(1.0, ilogb(v) - 7);  // unit in the 8th significant bit
      parts[i] = floor(v / q) * q;
      v -= parts[i];
    }
  }
  *v4 = make_float4((float)parts[0], (float)parts[1], (float)parts[2], (float)v);
  const double a = turns * (double)S;
  *c0 = (float)(a - floor(a));
}
// The anchor angle of a channel pair (step parts v, start c0) in group
// g (< 2^16) in turns, in [0, 1): frac(c0 + g v.x + g v.y + g v.z + g v.w) in
// fp32; g v.x .. g v.z are exact and reduced exactly, g v.w stays below 0.2
// turns, so the result is off by a few fp32 units of one turn (checked
// against fp64 on the host).
__host__ __device__ inline float anchor_turns(const float4& v, float c0, int g) {
  const float gf = (float)g;
  const float a = gf * v.x, b = gf * v.y, c = gf * v.z;
  float t = (a - floorf(a)) + (b - floorf(b));
  t = (t - floorf(t)) + (c - floorf(c));
  t += fmaf(gf, v.w, c0);
  return t - floorf(t);
}

// ------------------------------------------------ dependent launch (PDL)
// Kernels launched with launch_dependent() may start while the previous
// kernel in the stream is still running (their CTAs set up shared memory and
// the schedule meanwhile); grid_dep_wait() returns once every earlier grid
// has completed and its memory writes are visible, so a kernel calls it
// before its first access to memory that earlier work writes or reads.
// grid_dep_trigger() lets the next such kernel launch early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" :::); }

template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Split kernel: raise the quantized splits (n_qsplit of n_split per stream,
// the rest covering the fp16 tokens) so that NS x splits CTAs fill whole
// waves of `resident` CTAs, at most kMaxQSplits and one group per split.
// Returns the new groups per split (or the old one when nothing changes)
// and updates the split counts.
inline int fill_waves_plan(long long NS, long long resident, int ngroups, int gps, int* n_qsplit, int* n_split) {
  if (*n_qsplit <= 0 || resident < 1) return gps;
  const int fp16_split = *n_split - *n_qsplit;
  const long long waves = (NS * *n_split + resident - 1) / resident;
  long long q = waves * resident / NS - fp16_split;
  if (q > kMaxQSplits) q = kMaxQSplits;
  if (q > ngroups) q = ngroups;
  if (q <= *n_qsplit) return gps;
  const int per = (ngroups + (int)q - 1) / (int)q;
  *n_qsplit = (ngroups + per - 1) / per;
  *n_split = *n_qsplit + fp16_split;
  return per;
}

// ----------------------------------------------- per-device launch memos
// Facts that do not change within a process -- a device's SM count, a
// kernel's raised shared-memory limit, its resident CTAs at a shared-memory
// size -- are remembered per device (0 = not known yet; a race only repeats
// a query), so that a decode call does not pay the runtime queries each time.
constexpr int kMemoDevices = 64;

inline int memo_slot() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMemoDevices) return -1;
  return d;
}

inline cudaError_t device_sm_count(int* sms) {
  static std::atomic<long long> memo[kMemoDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < kMemoDevices;
  if (slot) {
    const long long v = memo[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *sms = (int)v;
      return cudaSuccess;
    }
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && slot) memo[dev].store(*sms, std::memory_order_relaxed);
  return e;
}

// Raise a kernel's dynamic shared-memory limit to at least smem (memo: the
// largest limit set per device).
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kernel, std::atomic<long long>* memo, int smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  const int d = memo_slot();
  if (d >= 0 && memo[d].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && d >= 0) {
    long long cur = memo[d].load(std::memory_order_relaxed);
    while (cur < smem && !memo[d].compare_exchange_weak(cur, smem, std::memory_order_relaxed)) {
    }
  }
  return e;
}

// Resident CTAs per SM of a kernel at (threads, smem) (memo: the last size
// asked per device; call after ensure_smem_limit).
template <typename Kernel>
inline cudaError_t occupancy_memo(Kernel kernel, std::atomic<long long>* memo, int threads, int smem, int* ctas) {
  const int d = memo_slot();
  if (d >= 0) {
    const long long v = memo[d].load(std::memory_order_relaxed);
    if (v > 0 && (v >> 16) == smem) {
      *ctas = (int)(v & 0xFFFF) - 1;
      return cudaSuccess;
    }
  }
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, threads, smem);
  if (e == cudaSuccess && d >= 0 && *ctas >= 0 && *ctas < 0xFFFF)
    memo[d].store(((long long)smem << 16) | (*ctas + 1), std::memory_order_relaxed);
  return e;
}

// ------------------------------------------------------------ host hooks
cudaError_t launch_distortion(const AppendParams& p, int n_tokens, int bits, float* knorm, double* mse,
                              cudaStream_t st);
cudaError_t launch_nuq_fit(const uint16_t* x, long long nvec, int k, int hadamard, int max_iters, void* ws,
                           float* lut_out, int* info_out, cudaStream_t st);
cudaError_t launch_merge_attn(int n_parts, long long rows, const uint16_t* outs, const float* lses,
                              uint16_t* out, float* lse_out, cudaStream_t st);
cudaError_t launch_append_quantize(const AppendParams& p, int n_groups, cudaStream_t st);
cudaError_t launch_key_norm(const AppendParams& p, cudaStream_t st);
cudaError_t launch_append_window(const AppendParams& p, int ncopy, cudaStream_t st);
cudaError_t launch_append_rows(const int32_t* before, const int32_t* n, int rows, int* dst, cudaStream_t st);
cudaError_t launch_ragged_tables(const RaggedTables& t, RaggedTables* dst, cudaStream_t st);
// Split-K decode; with occ != nullptr it only reports the kernel's resident
// CTAs per SM (for sizing the grid) and launches nothing.
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st, int* occ = nullptr);
// Persistent decode (uniform K/V with 64-channel V groups, no RoPE; or an fp16
// cache).  Fills the schedule fields of p (nwarps from the device's SM count
// and the kernel's occupancy) and reports the workspace it needs.
bool persist_eligible(const Geometry& g);
cudaError_t plan_persist(DecodeParams& p, uint64_t* ws_need);
cudaError_t launch_decode_persist(const DecodeParams& p, cudaStream_t st);
// Geometry of a config (validation included), for the other host units.
kvq_status make_geometry_for(const kvq_config* cfg, Geometry* g);
// One decode in three steps (kvq_decode_attn and the no-allocation entry
// point share them): validate and plan on the host; size the scratch (the
// persistent plan asks the device for its SM count and occupancy); launch.
kvq_status decode_setup(const kvq_config* cfg, const void* layer_buf, int32_t tokens, const uint16_t* q,
                        uint16_t* out, float* lse, DecodeParams* p, bool* persistent, uint64_t* layout_ws);
// widen: with automatic splits, raise the split kernel's split count so its
// grid fills whole waves of resident CTAs (more scratch; the fixed-scratch
// entry point passes false when the widened plan would not fit its array).
kvq_status decode_plan_device(DecodeParams* p, bool persistent, uint64_t* need, bool widen = true);
kvq_status decode_launch(DecodeParams* p, bool persistent, void* ws, cudaStream_t st);

// --------------------------------------------------------- device helpers
#ifdef __CUDACC__

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t float_to_half_bits(float f) {
  return __half_as_ushort(__float2half_rn(f));
}

// {min, scale} pair stored as two fp16 in one 32-bit word (min in the low half).
__device__ __forceinline__ float2 unpack_min_scale(uint32_t w) {
  return make_float2(half_bits_to_float((uint16_t)(w & 0xffffu)),
                     half_bits_to_float((uint16_t)(w >> 16)));
}

// An integer 0 <= u < 2^23 as fp32, exactly: build the float 2^23 + u by
// bit pattern and subtract 2^23 (both exact).
__device__ __forceinline__ float small_uint_to_float(uint32_t u) {
  return __uint_as_float(0x4B000000u | u) - 8388608.0f;
}

// Code c (b bits) of a packed little-endian bitstream held in 32-bit words.
template <int B>
__device__ __forceinline__ uint32_t code_at(const uint32_t* w, int c) {
  const int bit = c * B;
  const int wi = bit >> 5, sh = bit & 31;
  if (sh + B <= 32) return (w[wi] >> sh) & ((1u << B) - 1u);
  return __funnelshift_r(w[wi], w[wi + 1], sh) & ((1u << B) - 1u);
}

#endif  // __CUDACC__

}  // namespace kvq
