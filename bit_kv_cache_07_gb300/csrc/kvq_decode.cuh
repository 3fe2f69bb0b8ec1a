// kvq_decode.cuh -- fused dequantize-and-attend decode kernel (split-K over
// the context, last-CTA log-sum-exp merge), CUDA-core fp32 version.
//
// Method (page title, section):
//  * InnerQ, Methodology 3 and 5: dequantization fused with the GEMV in one
//    pass; a group's scale is loaded once and reused by every element of
//    the group.  Here the per-channel K scales of a 32-token group are folded
//    into the query once per group (q'_c = q_c * scale_c, bias = q . min),
//    and the per-token V scales are folded into the softmax weight
//    (p'_t = p_t * scale_t), so codes are used as plain small integers.
//  * InnerQ, Methodology 4: fp16 sink and recent tokens attended in the
//    same launch.
//  * KVQuant, technical approach: pre-RoPE K -- RoPE is applied to each
//    dequantized key at its position; non-uniform codes index a per-layer
//    level table; per-vector fp16 outliers are added back from CSR rows.
//  * Hadamard write-up, "section details": the quantized part of the
//    attention sum stays in the rotated domain and is rotated back once, in
//    the merge, after the sum.
//
// Work decomposition: grid = (splits per stream, NS streams), 4 warps per
// CTA.  Splits [0, n_qsplit) each own a run of 32-token quantized groups;
// the last split (quantized mode) owns the fp16 sinks + window.  In fp16
// mode every split owns a run of fp16 tokens.  Inside a CTA, warp w takes
// every 4th group/chunk.  For K, lane l computes the logits of token l of
// the group for every query head of the GQA group (no cross-lane reduction
// per token); for V, lane l owns channels 4l..4l+3 and accumulates over the
// group's tokens.  Softmax is online, in base 2 (q carries log2(e)).
#pragma once

#include <cstddef>

#include "kvq_internal.cuh"

namespace kvq {

template <int GQ>
struct DecodeSmem {
  // every member starts on a 16-byte boundary: several are read as float4
  alignas(16) float q[GQ][kHeadDim];     // q * softmax_scale * log2(e); heads >= g are 0
  alignas(16) float qsum[GQ];            // sum_c q[r][c]
  alignas(16) float p[4][kGroupTokens][GQ];              // per warp: softmax weights of the current chunk
  alignas(16) float pv[4][kGroupTokens][GQ];             // per warp: NUQ weights times the token's V scale
  alignas(16) float2 anchor[4][kHeadDim / 2];  // per warp: e^{i t0 theta_j} of the group
  alignas(16) float4 anc_v[kHeadDim / 2];      // RoPE group-anchor steps and starts (anchor_step),
  alignas(16) float anc_c0[kHeadDim / 2];      // in shared memory: lanes index them by pair
  alignas(16) float ml[4][GQ][2];              // per warp (m, l)
  alignas(16) float comb_ml[GQ][2];            // CTA-combined (m, l)
  alignas(16) float lut_k[8];
  alignas(16) float lut_v[8];
  int is_last;
  // used by the uniform-code paths only (a non-uniform launch leaves them out
  // of its shared memory: decode_smem_fixed)
  alignas(16) float work[4][GQ > 2 ? GQ : 2][kHeadDim];  // per warp: folded q' / K min+scale; merge staging
  alignas(16) uint32_t vs[4][kGroupTokens][4];           // per warp: V {min, scale} words of the group
  alignas(16) uint8_t ocol[4][kGroupTokens][kMaxOutliers];  // per warp: V outlier columns
  alignas(16) float oval[4][kGroupTokens][kMaxOutliers];    // per warp: V outlier values
  alignas(16) int ocnt[4][kGroupTokens];
};

// Bytes of DecodeSmem a launch uses: the non-uniform (KB = 3) kernel stops
// before `work` (its merge staging goes to its free NUQ stages instead).
template <int KB, int GQ>
__host__ __device__ constexpr size_t decode_smem_fixed() {
  return ((KB == 3 ? offsetof(DecodeSmem<GQ>, work) : sizeof(DecodeSmem<GQ>)) + 15) / 16 * 16;
}

// RoPE offset table e^{i l theta_j} (or the query-folded W_{j,l}), l = token
// offset in a 32-token group: entries of pairs 2i and 2i+1 for one l are
// adjacent (a lane reads both with one 16-byte load), lanes l consecutive.
__host__ __device__ __forceinline__ int rope_tab_index(int j, int l) { return (((j >> 1) * 32 + l) << 1) | (j & 1); }

// RoPE region of the dynamic shared memory: the offset table over 32 token
// offsets, or, for non-uniform codes with one query head, the query-folded
// table over 16 offsets followed by each warp's second anchor set (the
// anchors of offsets 16..31, see k_logits_nuq_st).
template <int KB, int GQ>
__host__ __device__ constexpr int rope_region_bytes() {
  return (KB == 3 && GQ == 1) ? 16 * (kHeadDim / 2) * 8 + 4 * (kHeadDim / 2) * 8
                              : kGroupTokens * (kHeadDim / 2) * 8;
}

// 16-byte asynchronous global -> shared copies (cp.async, completion by group)
__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y);
}

// e^{i x} for an fp64 angle: reduce modulo 2 pi in fp64, then fp32 sincos.
__device__ __forceinline__ float2 expi(double x) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;  // n only needs to be the nearest integer or next to it
  const double r = x - two_pi * rint(x * inv_two_pi);
  float sn, cs;
  sincosf((float)r, &sn, &cs);
  return make_float2(cs, sn);
}

// Anchor e^{i theta_j (S + 32 g)} of group g without fp64 (a narrow pipe
// on this GPU, and every lane needs two anchors per group): the angle in
// turns from anchor_turns (a few 1e-7 turns off), reduced to [-1/2, 1/2]
// turns, then the hardware sine and cosine (absolute error below 1e-6).
// Groups from 2^16 on take the fp64 reduction.
template <int GQ>
__device__ __forceinline__ float2 anchor_expi(const DecodeParams& p, const DecodeSmem<GQ>& sm, int j, int g) {
  if (g >= (1 << 16))
    return expi(((double)p.geo.pos_offset + (double)p.geo.S + (double)g * kGroupTokens) * p.theta[j]);
  float t = anchor_turns(sm.anc_v[j], sm.anc_c0[j], g);
  t -= rintf(t);
  float sn, cs;
  __sincosf(6.28318530717958648f * t, &sn, &cs);
  return make_float2(cs, sn);
}

// Online-softmax update of one warp for one 32-token chunk: z[r] is the
// base-2 logit of this lane's token (-inf when masked).
template <int GQ>
__device__ __forceinline__ void softmax_update(float (&z)[GQ], float (&m)[GQ], float (&lsum)[GQ],
                                               float (&acc)[GQ][4], float (&macc)[GQ],
                                               float (*p_out)[GQ], int lane) {
#pragma unroll
  for (int r = 0; r < GQ; ++r) {
    const float cmax = warp_max(z[r]);
    const float mnew = fmaxf(m[r], cmax);
    float alpha, pl;
    if (mnew == -INFINITY) {
      alpha = 1.0f;
      pl = 0.0f;
    } else {
      alpha = exp2f(m[r] - mnew);
      pl = exp2f(z[r] - mnew);
    }
    lsum[r] = lsum[r] * alpha + pl;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[r][k] *= alpha;
    macc[r] *= alpha;
    m[r] = mnew;
    p_out[lane][r] = pl;
  }
  __syncwarp();
}

// ---------------------------------------------------------------- K logits

// Uniform per-channel K, no RoPE: z[r] = bias_r + sum_c q'_rc * code_c.
template <int KB, int GQ>
__device__ __forceinline__ void k_logits_uniform(const DecodeParams& p, DecodeSmem<GQ>& sm,
                                                 int s, int grp, int lane, int w, float (&z)[GQ]) {
  const Geometry& G = p.geo;
  {
    const uint4 sc = *reinterpret_cast<const uint4*>(p.L.k_scales +
                                                     ((size_t)s * G.gcap + grp) * kHeadDim + 4 * lane);
    const uint32_t wv[4] = {sc.x, sc.y, sc.z, sc.w};
    float bpart[GQ];
#pragma unroll
    for (int r = 0; r < GQ; ++r) bpart[r] = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 ms = unpack_min_scale(wv[k]);
      const int c = 4 * lane + k;
#pragma unroll
      for (int r = 0; r < GQ; ++r) {
        const float qv = sm.q[r][c];
        sm.work[w][r][c] = qv * ms.y;
        bpart[r] = fmaf(qv, ms.x, bpart[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < GQ; ++r) z[r] = warp_sum(bpart[r]);
  }
  __syncwarp();
  constexpr int KROW = kHeadDim * KB / 8;
  constexpr int PER_WORD = 32 / KB;
  const uint4* row = reinterpret_cast<const uint4*>(p.L.k_codes + ((size_t)s * G.qcap +
                                                                   (size_t)grp * kGroupTokens + lane) * KROW);
#pragma unroll
  for (int ch = 0; ch < KROW / 16; ++ch) {
    const uint4 u = __ldg(row + ch);
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
      for (int m0 = 0; m0 < PER_WORD; m0 += 4) {
        const int c = (ch * 4 + wi) * PER_WORD + m0;
        float x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = small_uint_to_float((wd[wi] >> ((m0 + k) * KB)) & ((1u << KB) - 1u));
#pragma unroll
        for (int r = 0; r < GQ; ++r) {
          const float4 qp = *reinterpret_cast<const float4*>(&sm.work[w][r][c]);
          z[r] = fmaf(qp.x, x[0], z[r]);
          z[r] = fmaf(qp.y, x[1], z[r]);
          z[r] = fmaf(qp.z, x[2], z[r]);
          z[r] = fmaf(qp.w, x[3], z[r]);
        }
      }
    }
  }
}

// Any quantized K with RoPE after dequantization: reconstruct k^ for each
// channel pair (j, j + 64), rotate by the angle of this lane's position
// (anchor of the group times e^{i lane theta_j}), dot with q.
template <int KB, int GQ>
__device__ __forceinline__ void k_logits_rope(const DecodeParams& p, DecodeSmem<GQ>& sm,
                                              const float2* __restrict__ rope_e, int s, int grp,
                                              int lane, int w, float (&z)[GQ]) {
  const Geometry& G = p.geo;
  // group anchor e^{i (S + 32 grp) theta_j}
  for (int j = lane; j < kHeadDim / 2; j += 32) sm.anchor[w][j] = anchor_expi<GQ>(p, sm, j, grp);
  const size_t i = (size_t)grp * kGroupTokens + lane;
  float nmin = 0.0f, nsc = 0.0f;
  if (KB == 3) {
    const float2 ms = unpack_min_scale(__ldg(p.L.k_scales + (size_t)s * G.qcap + i));
    nmin = ms.x;
    nsc = ms.y;
  } else {
    const uint4 sc = *reinterpret_cast<const uint4*>(p.L.k_scales +
                                                     ((size_t)s * G.gcap + grp) * kHeadDim + 4 * lane);
    const uint32_t wv[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 ms = unpack_min_scale(wv[k]);
      sm.work[w][0][4 * lane + k] = ms.x;
      sm.work[w][1][4 * lane + k] = ms.y;
    }
  }
  __syncwarp();
  constexpr int KROW = kHeadDim * KB / 8;
  constexpr int NW = KROW / 4;
  uint32_t wd[NW + 1];
  const uint4* row = reinterpret_cast<const uint4*>(p.L.k_codes + ((size_t)s * G.qcap + i) * KROW);
#pragma unroll
  for (int k = 0; k < KROW / 16; ++k) {
    const uint4 u = __ldg(row + k);
    wd[4 * k] = u.x; wd[4 * k + 1] = u.y; wd[4 * k + 2] = u.z; wd[4 * k + 3] = u.w;
  }
  wd[NW] = 0;
#pragma unroll
  for (int r = 0; r < GQ; ++r) z[r] = 0.0f;
#pragma unroll
  for (int j = 0; j < kHeadDim / 2; ++j) {
    float a, b;
    const uint32_t ca = code_at<KB>(wd, j), cb = code_at<KB>(wd, j + kHeadDim / 2);
    if (KB == 3) {
      a = fmaf(nsc, sm.lut_k[ca], nmin);
      b = fmaf(nsc, sm.lut_k[cb], nmin);
    } else {
      a = fmaf(small_uint_to_float(ca), sm.work[w][1][j], sm.work[w][0][j]);
      b = fmaf(small_uint_to_float(cb), sm.work[w][1][j + kHeadDim / 2], sm.work[w][0][j + kHeadDim / 2]);
    }
    const float2 e = cmul(sm.anchor[w][j], rope_e[rope_tab_index(j, lane)]);
    const float ra = a * e.x - b * e.y;
    const float rb = b * e.x + a * e.y;
#pragma unroll
    for (int r = 0; r < GQ; ++r) z[r] = fmaf(sm.q[r][j], ra, fmaf(sm.q[r][j + kHeadDim / 2], rb, z[r]));
  }
  if (KB == 3) {
    const int32_t* rp = p.L.k_rowptr + (size_t)s * (G.qcap + 1);
    const int jcap = G.qcap * G.nout;
    const int j0 = max(0, __ldg(rp + i)), j1 = min(jcap, __ldg(rp + i + 1));
    const size_t base = (size_t)s * jcap;
    for (int j = j0; j < j1; ++j) {
      const int col = __ldg(p.L.k_col + base + j);
      const float dv = half_bits_to_float(__ldg(p.L.k_val + base + j)) - nmin;
      const int f = col & (kHeadDim / 2 - 1);
      const float2 e = cmul(sm.anchor[w][f], rope_e[rope_tab_index(f, lane)]);
      // rotated unit vector of channel col, times dv, dotted with q
#pragma unroll
      for (int r = 0; r < GQ; ++r) {
        const float qa = sm.q[r][f], qb = sm.q[r][f + kHeadDim / 2];
        const float dotu = (col < kHeadDim / 2) ? (qa * e.x + qb * e.y) : (-qa * e.y + qb * e.x);
        z[r] = fmaf(dv, dotu, z[r]);
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ V part

template <int VB, int GQ>
__device__ __forceinline__ void v_accumulate(const DecodeParams& p, DecodeSmem<GQ>& sm, int s, int grp,
                                             int lane, int w, float (&acc)[GQ][4], float (&macc)[GQ]) {
  const Geometry& G = p.geo;
  const size_t i0 = (size_t)grp * kGroupTokens;
  // stage this group's V scales (and, for non-uniform V, its outliers)
  if (VB == 3) {
    const size_t i = i0 + lane;
    sm.vs[w][lane][0] = __ldg(p.L.v_scales + (size_t)s * G.qcap + i);
    const int32_t* rp = p.L.v_rowptr + (size_t)s * (G.qcap + 1);
    const int jcap = G.qcap * G.nout;
    const int j0 = max(0, __ldg(rp + i)), j1 = min(jcap, __ldg(rp + i + 1));
    const size_t base = (size_t)s * jcap;
    const float mn = unpack_min_scale(sm.vs[w][lane][0]).x;
    int n = 0;
    for (int j = j0; j < j1 && n < kMaxOutliers; ++j, ++n) {
      sm.ocol[w][lane][n] = __ldg(p.L.v_col + base + j);
      sm.oval[w][lane][n] = half_bits_to_float(__ldg(p.L.v_val + base + j)) - mn;
    }
    sm.ocnt[w][lane] = n;
  } else {
    const uint32_t* src = p.L.v_scales + ((size_t)s * G.qcap + i0 + lane) * G.nvg;
    for (int k = 0; k < G.nvg; ++k) sm.vs[w][lane][k] = __ldg(src + k);
  }
  __syncwarp();
  const int jg = (VB == 3) ? 0 : (4 * lane) / G.gv;
  constexpr int VROW = kHeadDim * VB / 8;
  const uint8_t* vbase = p.L.v_codes + ((size_t)s * G.qcap + i0) * VROW;
#pragma unroll 4
  for (int t = 0; t < kGroupTokens; ++t) {
    const float2 ms = unpack_min_scale(sm.vs[w][t][jg]);
    float cv[4];
    if (VB == 8) {
      const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(vbase + (size_t)t * VROW) + lane);
#pragma unroll
      for (int k = 0; k < 4; ++k) cv[k] = small_uint_to_float((u >> (8 * k)) & 0xffu);
    } else if (VB == 4) {
      const uint32_t u = __ldg(reinterpret_cast<const uint16_t*>(vbase + (size_t)t * VROW) + lane);
#pragma unroll
      for (int k = 0; k < 4; ++k) cv[k] = small_uint_to_float((u >> (4 * k)) & 0xfu);
    } else if (VB == 2) {
      const uint32_t u = __ldg(vbase + (size_t)t * VROW + lane);
#pragma unroll
      for (int k = 0; k < 4; ++k) cv[k] = small_uint_to_float((u >> (2 * k)) & 0x3u);
    } else {  // 3-bit: channels 4l..4l+3 at bits 12l..12l+11
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(vbase + (size_t)t * VROW);
      const int bit = 12 * lane, wi = bit >> 5, sh = bit & 31;
      uint32_t u = __ldg(rw + wi) >> sh;
      if (sh > 20) u |= __ldg(rw + wi + 1) << (32 - sh);
#pragma unroll
      for (int k = 0; k < 4; ++k) cv[k] = sm.lut_v[(u >> (3 * k)) & 7u];
    }
#pragma unroll
    for (int r = 0; r < GQ; ++r) {
      const float pr = sm.p[w][t][r];
      const float pp = pr * ms.y;
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[r][k] = fmaf(pp, cv[k], acc[r][k]);
      macc[r] = fmaf(pr, ms.x, macc[r]);
    }
    if (VB == 3) {
      const int n = sm.ocnt[w][t];
      for (int j = 0; j < n; ++j) {
        const int col = sm.ocol[w][t][j];
        if ((col >> 2) == lane) {
          const float dv = sm.oval[w][t][j];
#pragma unroll
          for (int r = 0; r < GQ; ++r) {
            const float a = sm.p[w][t][r] * dv;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if ((col & 3) == k) acc[r][k] += a;
          }
        }
      }
    }
  }
  __syncwarp();
}

// fp16 token of index k in this split's fp16 token list -> (row pointer
// offset in halves, absolute position).
// S_eff, Nq: the stream's sinks present and quantized tokens.
__device__ __forceinline__ size_t fp16_row_at(const DecodeParams& p, int s, int k, int S_eff, int Nq, bool* in_sink,
                                              int* pos) {
  const Geometry& G = p.geo;
  if (G.fp16_mode) {
    *in_sink = false;
    *pos = k;
    return ((size_t)s * G.ring + k) * kHeadDim;
  }
  if (k < S_eff) {
    *in_sink = true;
    *pos = k;
    return ((size_t)s * G.S + k) * kHeadDim;
  }
  const int ps = G.S + Nq + (k - S_eff);
  *in_sink = false;
  *pos = ps;
  return ((size_t)s * G.ring + (ps - G.S) % G.ring) * kHeadDim;
}

// One 32-token chunk of fp16 tokens (sinks / window, or an fp16 cache) for
// one warp: lane = token for q.k, lane = 4 channels for p.v.  sq is the
// scaled query [GQ][d] in shared memory, pbuf this warp's [32][GQ] buffer.
// KBATCH / VBATCH: independent loads in flight per batch (K: 16-byte pieces
// of the lane's row; V: rows), traded against registers.  ROPE = false
// compiles the RoPE path out (callers that never see pre-RoPE keys).
template <int GQ, int KBATCH = 8, int VBATCH = 8, bool ROPE = true>
__device__ __forceinline__ void fp16_chunk(const DecodeParams& p, const float (*sq)[kHeadDim],
                                           float (*pbuf)[GQ], int s, int k0, int k1, int se, int nq, int lane,
                                           float (&m)[GQ], float (&lsum)[GQ], float (&acc)[GQ][4],
                                           float (&macc)[GQ]) {
  const Geometry& G = p.geo;
  float z[GQ];
  const int k = k0 + lane;
#pragma unroll
  for (int r = 0; r < GQ; ++r) z[r] = -INFINITY;
  if (k < k1) {
    bool sink;
    int pos;
    const size_t off = fp16_row_at(p, s, k, se, nq, &sink, &pos);
    const uint4* krow = reinterpret_cast<const uint4*>((sink ? p.L.k_sink : p.L.k_ring) + off);
#pragma unroll
    for (int r = 0; r < GQ; ++r) z[r] = 0.0f;
    if (!ROPE || !G.pre_rope) {
      // the row in batches of KBATCH independent 16-byte loads
#pragma unroll
      for (int half = 0; half < 16 / KBATCH; ++half) {
        uint4 u[KBATCH];
#pragma unroll
        for (int i = 0; i < KBATCH; ++i) u[i] = __ldg(krow + KBATCH * half + i);
#pragma unroll
        for (int i = 0; i < KBATCH; ++i) {
          const uint32_t wd[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 kv = __half22float2(*reinterpret_cast<const __half2*>(&wd[h]));
            const int c = (KBATCH * half + i) * 8 + 2 * h;
#pragma unroll
            for (int r = 0; r < GQ; ++r) z[r] = fmaf(sq[r][c], kv.x, fmaf(sq[r][c + 1], kv.y, z[r]));
          }
        }
      }
    } else if constexpr (ROPE) {
      // RoPE pairs (j, j + d/2): the row's first half holds channel j, the second j + d/2
      uint4 ua[8], ub[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ua[i] = __ldg(krow + i);
        ub[i] = __ldg(krow + 8 + i);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t wa[4] = {ua[i].x, ua[i].y, ua[i].z, ua[i].w};
        const uint32_t wb[4] = {ub[i].x, ub[i].y, ub[i].z, ub[i].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 a2 = __half22float2(*reinterpret_cast<const __half2*>(&wa[h]));
          const float2 b2 = __half22float2(*reinterpret_cast<const __half2*>(&wb[h]));
          const int j = i * 8 + 2 * h;
          const double apos = (double)G.pos_offset + (double)pos;  // absolute position
          const float2 e0 = expi(apos * p.theta[j]);
          const float2 e1 = expi(apos * p.theta[j + 1]);
          const float ra0 = a2.x * e0.x - b2.x * e0.y, rb0 = b2.x * e0.x + a2.x * e0.y;
          const float ra1 = a2.y * e1.x - b2.y * e1.y, rb1 = b2.y * e1.x + a2.y * e1.y;
#pragma unroll
          for (int r = 0; r < GQ; ++r) {
            z[r] = fmaf(sq[r][j], ra0, fmaf(sq[r][j + kHeadDim / 2], rb0, z[r]));
            z[r] = fmaf(sq[r][j + 1], ra1, fmaf(sq[r][j + 1 + kHeadDim / 2], rb1, z[r]));
          }
        }
      }
    }
  }
  softmax_update<GQ>(z, m, lsum, acc, macc, pbuf, lane);
  const int n = min(32, k1 - k0);
  // V rows in batches of VBATCH tokens: the loads of a batch are independent
  for (int t0 = 0; t0 < n; t0 += VBATCH) {
    uint2 u[VBATCH];
#pragma unroll
    for (int i = 0; i < VBATCH; ++i) {
      u[i] = make_uint2(0u, 0u);
      if (t0 + i < n) {
        bool sink;
        int pos;
        const size_t off = fp16_row_at(p, s, k0 + t0 + i, se, nq, &sink, &pos);
        u[i] = __ldg(reinterpret_cast<const uint2*>((sink ? p.L.v_sink : p.L.v_ring) + off) + lane);
      }
    }
#pragma unroll
    for (int i = 0; i < VBATCH; ++i) {
      if (t0 + i >= n) break;
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&u[i].x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&u[i].y));
#pragma unroll
      for (int r = 0; r < GQ; ++r) {
        const float pr = pbuf[t0 + i][r];
        acc[r][0] = fmaf(pr, v01.x, acc[r][0]);
        acc[r][1] = fmaf(pr, v01.y, acc[r][1]);
        acc[r][2] = fmaf(pr, v23.x, acc[r][2]);
        acc[r][3] = fmaf(pr, v23.y, acc[r][3]);
      }
    }
  }
  __syncwarp();
}

// In-warp FWHT of a 128-vector (lane l holds elements 4l..4l+3), then * c.
__device__ __forceinline__ void warp_fwht(float (&v)[4], float c, int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float o = __shfl_xor_sync(0xffffffffu, v[q], m);
      v[q] = upper ? (o - v[q]) : (v[q] + o);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] *= c;
}

// ------------------------------------------------------ staged NUQ groups
// For the non-uniform (3-bit) cache every warp streams its groups into
// shared memory with cp.async: while it computes group i, group i + 4 (its
// next one) streams in.  The K code rows (48 bytes per token) go to one
// buffer per warp: the lanes take their rows into registers before the
// next group's rows are issued into it.  Everything else is double-buffered
// in stages: V code rows, the per-token {min, s} words, and the group's CSR
// outlier entries -- exactly k per row (the append writes k entries for
// every row), so a group's entries are the k*32 consecutive ones starting
// at row * k and the row pointers are not needed here.
struct NuqStage {
  static constexpr int KBUF = kGroupTokens * 48;  // the per-warp K code buffer
  static constexpr int VC = 0, KMS = kGroupTokens * 48;
  static constexpr int VMS = KMS + kGroupTokens * 4, CSR = VMS + kGroupTokens * 4;
  static __host__ __device__ constexpr int kcol(int k) { return CSR; }
  static __host__ __device__ constexpr int kval(int k) { return CSR + 32 * k; }
  static __host__ __device__ constexpr int vcol(int k) { return CSR + 96 * k; }
  static __host__ __device__ constexpr int vval(int k) { return CSR + 128 * k; }
  static __host__ __device__ constexpr int bytes(int k) { return (CSR + 192 * k + 127) / 128 * 128; }
  // one warp's K buffer and two stages
  static __host__ __device__ constexpr int warp_bytes(int k) { return KBUF + 2 * bytes(k); }
};

__device__ __forceinline__ void issue_nuq(const DecodeParams& p, int s, int grp, uint32_t kdst, uint32_t dst,
                                          int lane) {
  const Geometry& G = p.geo;
  const int k = G.nout;
  const size_t i0 = (size_t)s * G.qcap + (size_t)grp * kGroupTokens;  // first row of the group
  const uint8_t* kc = p.L.k_codes + i0 * 48;
  const uint8_t* vc = p.L.v_codes + i0 * 48;
  for (int c = lane; c < kGroupTokens * 48 / 16; c += 32) {
    cp_async16(kdst + 16 * c, kc + 16 * c);
    cp_async16(dst + NuqStage::VC + 16 * c, vc + 16 * c);
  }
  if (lane < 8) {
    cp_async16(dst + NuqStage::KMS + 16 * lane, p.L.k_scales + i0 + 4 * lane);
    cp_async16(dst + NuqStage::VMS + 16 * lane, p.L.v_scales + i0 + 4 * lane);
  }
  // CSR: 32k column bytes and 64k value bytes per side (multiples of 16)
  for (int c = lane; c < 2 * k; c += 32) {
    cp_async16(dst + NuqStage::kcol(k) + 16 * c, p.L.k_col + i0 * k + 16 * c);
    cp_async16(dst + NuqStage::vcol(k) + 16 * c, p.L.v_col + i0 * k + 16 * c);
  }
  for (int c = lane; c < 4 * k; c += 32) {
    cp_async16(dst + NuqStage::kval(k) + 16 * c, reinterpret_cast<const uint8_t*>(p.L.k_val + i0 * k) + 16 * c);
    cp_async16(dst + NuqStage::vval(k) + 16 * c, reinterpret_cast<const uint8_t*>(p.L.v_val + i0 * k) + 16 * c);
  }
}

// 3-bit code c of a 48-byte row held in 12 (+1 zero) registers.
__device__ __forceinline__ uint32_t code3(const uint32_t (&w)[13], int c) { return code_at<3>(w, c); }

// Pair tables: the level values of two adjacent 3-bit codes with one 8-byte
// load.  Entry f = c0 | c1 << 3 holds (L[c0], L[c1]); each entry is stored
// 16 times, copy i at bank pair i, and lane l reads copy l & 15, so the
// 16 lanes of a half-warp never meet in a bank whatever their codes.
// Byte offset of entry f, copy i: f * 128 + i * 8.
constexpr int kPairEntries = 64, kPairCopies = 16;
constexpr int kPairTableBytes = kPairEntries * kPairCopies * 8;

// Dynamic shared memory of a split-kernel launch: DecodeSmem (up to `work`
// for non-uniform codes), for non-uniform codes the K and V pair tables (at
// a fixed offset, so their loads take it as an immediate), the RoPE region,
// and for non-uniform codes the warps' K buffers and stages and their
// outlier buffers.
template <int KB, int GQ>
__host__ __device__ constexpr size_t decode_smem_bytes(bool pre_rope, int nout) {
  return decode_smem_fixed<KB, GQ>() + (KB == 3 ? 2 * kPairTableBytes : 0) +
         (pre_rope ? rope_region_bytes<KB, GQ>() : 0) +
         (KB == 3 ? 4 * (size_t)NuqStage::warp_bytes(nout) + 4 * GQ * kHeadDim * sizeof(float) : 0);
}

// (L[c], L[c+1]) for codes c, c+1 (c even) of a 48-byte row in registers;
// loff = (lane & 15) * 8.  The 6-bit field at bit 3c is shifted to bits
// 7..12 of x, which makes it the entry's byte offset.
__device__ __forceinline__ float2 pair_levels(const unsigned char* tab, const uint32_t (&w)[13], int c, uint32_t loff) {
  const int bp = 3 * c;
  uint32_t x;
  if (bp < 7) {
    x = w[0] << (7 - bp);
  } else {
    const int sft = bp - 7, w0 = sft >> 5, sh = sft & 31;
    x = sh <= 19 ? (w[w0] >> sh) : __funnelshift_r(w[w0], w[w0 + 1], sh);
  }
  return *reinterpret_cast<const float2*>(tab + ((x & 0x1F80u) | loff));
}

// K logits of one staged NUQ group, lane = token.
//  no RoPE:    z = min * sum(q) + s * sum_c q_c L'_code, plus outlier terms
//  RoPE, GQ=1: z = sum_j Re[W_{j,d} * A_j * (k_j + i k_{j+64})] for the
//              lane's offset lane = 16 h + d, with
//              W_{j,d} = conj(q_j + i q_{j+64}) e^{i theta_j d}, d < 16
//              (table, per CTA) and A_j = e^{i theta_j (t0 + 16 h)} (anchor
//              set h of the group): two complex products per channel pair
//              instead of rotating q or k; lanes d and 16 + d read the same
//              table entry
//  RoPE, GQ>1: rotate each key pair once by A_j e^{i theta_j lane}, dot with
//              every head
// Group anchors of a warp that visits groups g, g + 4, g + 8, ...: lane j
// keeps pairs j and j + 32; the anchor moves by e^{i theta_j 128} per visit
// (`step`, from an fp64 angle) and is recomputed exactly (anchor_expi) every
// kAnchorEvery visits, so fp32 rounding of the products stays within that
// many complex multiplications.  The second set is the first times
// e^{i theta_j 16} (`half`, from an fp64 angle).
constexpr int kAnchorEvery = 16;
struct AnchorWalk {
  float2 a[2], step[2], half[2];
  int left;  // visits before the next exact anchor
};

// A lane's K code row (48 bytes, token = lane) from the warp's K buffer.
__device__ __forceinline__ void load_code_row(const unsigned char* kbuf, int lane, uint32_t (&wd)[13]) {
  const uint4* row = reinterpret_cast<const uint4*>(kbuf + 48 * lane);
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint4 u = row[i];
    wd[4 * i] = u.x; wd[4 * i + 1] = u.y; wd[4 * i + 2] = u.z; wd[4 * i + 3] = u.w;
  }
  wd[12] = 0;
}

// tab: the RoPE region (for GQ = 1 the folded 16-offset table, then the
// second anchor sets of the 4 warps)
template <int GQ>
__device__ __forceinline__ void k_logits_nuq_st(const DecodeParams& p, DecodeSmem<GQ>& sm,
                                                const float2* tab, const unsigned char* ptab_k,
                                                const uint32_t (&wd)[13], const unsigned char* st, int grp,
                                                int lane, int w, float (&z)[GQ], AnchorWalk& aw) {
  const Geometry& G = p.geo;
  const int k = G.nout;
  const float2 ms = unpack_min_scale(reinterpret_cast<const uint32_t*>(st + NuqStage::KMS)[lane]);
  const uint8_t* ocol = st + NuqStage::kcol(k) + k * lane;
  const uint16_t* oval = reinterpret_cast<const uint16_t*>(st + NuqStage::kval(k)) + k * lane;
#pragma unroll
  for (int r = 0; r < GQ; ++r) z[r] = 0.0f;
  if (!G.pre_rope) {
    float zl[GQ];
#pragma unroll
    for (int r = 0; r < GQ; ++r) zl[r] = 0.0f;
#pragma unroll
    for (int c = 0; c < kHeadDim; c += 4) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = sm.lut_k[code3(wd, c + e)];
#pragma unroll
      for (int r = 0; r < GQ; ++r) {
        const float4 qv = *reinterpret_cast<const float4*>(&sm.q[r][c]);
        zl[r] = fmaf(qv.x, x[0], fmaf(qv.y, x[1], fmaf(qv.z, x[2], fmaf(qv.w, x[3], zl[r]))));
      }
    }
#pragma unroll
    for (int r = 0; r < GQ; ++r) z[r] = fmaf(ms.x, sm.qsum[r], ms.y * zl[r]);
    for (int e = 0; e < k; ++e) {
      const int col = ocol[e];
      const float dv = half_bits_to_float(oval[e]) - ms.x;
#pragma unroll
      for (int r = 0; r < GQ; ++r) z[r] = fmaf(sm.q[r][col], dv, z[r]);
    }
    return;
  }
  // group anchor e^{i t0 theta_j}
  if constexpr (GQ == 1) {
    // anchors of pairs 2i, 2i+1 as (x_2i, x_2i+1, y_2i, y_2i+1): fp32x2
    // operands without shuffling; set 0 (offsets 0..15) in sm.anchor, set 1
    // (offsets 16..31) after the folded table
    float* ap0 = reinterpret_cast<float*>(&sm.anchor[w][0]);
    float* ap1 = reinterpret_cast<float*>(const_cast<float2*>(tab) + 16 * (kHeadDim / 2) + w * (kHeadDim / 2));
    if (aw.left == 0) {
      aw.a[0] = anchor_expi<GQ>(p, sm, lane, grp);
      aw.a[1] = anchor_expi<GQ>(p, sm, lane + 32, grp);
      aw.left = kAnchorEvery;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      const float2 a1 = cmul(aw.a[h], aw.half[h]);
      ap0[(j >> 1) * 4 + (j & 1)] = aw.a[h].x;
      ap0[(j >> 1) * 4 + 2 + (j & 1)] = aw.a[h].y;
      ap1[(j >> 1) * 4 + (j & 1)] = a1.x;
      ap1[(j >> 1) * 4 + 2 + (j & 1)] = a1.y;
      aw.a[h] = cmul(aw.a[h], aw.step[h]);  // the anchor of this warp's next group
    }
    --aw.left;
    __syncwarp();
    // two channel pairs at a time in packed fp32x2 arithmetic (W laid out like the anchors)
    const float4* tab4 = reinterpret_cast<const float4*>(tab) + (lane & 15);
    const float4* anc4 = reinterpret_cast<const float4*>(lane < 16 ? ap0 : ap1);
    const float2 S2 = make_float2(ms.y, ms.y), M2 = make_float2(ms.x, ms.x);
    const uint32_t loff = (uint32_t)(lane & 15) * 8u;
    float2 z2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kHeadDim / 2; j += 2) {
      const float4 A4 = anc4[j >> 1];
      const float4 W4 = tab4[(j >> 1) * 16];
      const float2 Ax = make_float2(A4.x, A4.y), Ay = make_float2(A4.z, A4.w);
      const float2 Wx = make_float2(W4.x, W4.y), Wy = make_float2(W4.z, W4.w);
      const float2 a2 = __ffma2_rn(S2, pair_levels(ptab_k, wd, j, loff), M2);
      const float2 b2 = __ffma2_rn(S2, pair_levels(ptab_k, wd, j + kHeadDim / 2, loff), M2);
      const float2 cx = __ffma2_rn(Ax, a2, __fmul2_rn(make_float2(-Ay.x, -Ay.y), b2));  // ax a - ay b
      const float2 cy = __ffma2_rn(Ax, b2, __fmul2_rn(Ay, a2));                          // ax b + ay a
      z2 = __ffma2_rn(Wx, cx, __ffma2_rn(make_float2(-Wy.x, -Wy.y), cy, z2));           // Re[W c]
    }
    float zr = z2.x + z2.y;
    for (int e = 0; e < k; ++e) {
      const int col = ocol[e];
      const float dv = half_bits_to_float(oval[e]) - ms.x;
      const int j = col & (kHeadDim / 2 - 1);
      // W and the anchor of pair j as 16-byte loads: the W rows of a lane are
      // 16 bytes apart from its neighbours' whatever their columns (no bank
      // conflicts); pick the pair's components
      const float4 W4 = tab4[(j >> 1) * 16];
      const float4 A4 = anc4[j >> 1];
      const bool odd = (j & 1) != 0;
      const float2 WA = cmul(make_float2(odd ? W4.y : W4.x, odd ? W4.w : W4.z),
                             make_float2(odd ? A4.y : A4.x, odd ? A4.w : A4.z));
      zr = fmaf(dv, (col < kHeadDim / 2) ? WA.x : -WA.y, zr);  // Re[WA dv] or Re[WA i dv]
    }
    z[0] = zr;
  } else {
    for (int j = lane; j < kHeadDim / 2; j += 32) sm.anchor[w][j] = anchor_expi<GQ>(p, sm, j, grp);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kHeadDim / 2; ++j) {
      const float a = fmaf(ms.y, sm.lut_k[code3(wd, j)], ms.x);
      const float b = fmaf(ms.y, sm.lut_k[code3(wd, j + kHeadDim / 2)], ms.x);
      const float2 e = cmul(sm.anchor[w][j], tab[rope_tab_index(j, lane)]);
      const float ra = a * e.x - b * e.y, rb = b * e.x + a * e.y;
#pragma unroll
      for (int r = 0; r < GQ; ++r) z[r] = fmaf(sm.q[r][j], ra, fmaf(sm.q[r][j + kHeadDim / 2], rb, z[r]));
    }
    for (int e = 0; e < k; ++e) {
      const int col = ocol[e];
      const float dv = half_bits_to_float(oval[e]) - ms.x;
      const int f = col & (kHeadDim / 2 - 1);
      const float2 ee = cmul(sm.anchor[w][f], tab[rope_tab_index(f, lane)]);
#pragma unroll
      for (int r = 0; r < GQ; ++r) {
        const float qa = sm.q[r][f], qb = sm.q[r][f + kHeadDim / 2];
        const float dotu = (col < kHeadDim / 2) ? (qa * ee.x + qb * ee.y) : (-qa * ee.y + qb * ee.x);
        z[r] = fmaf(dv, dotu, z[r]);
      }
    }
  }
  __syncwarp();
}

// V part of one staged NUQ group: lane = channels 4l..4l+3; the group's
// outlier corrections go through a per-warp shared buffer (lane = entry,
// shared-memory atomics), folded into the accumulators afterwards.
template <int GQ>
__device__ __forceinline__ void v_accumulate_nuq_st(const DecodeParams& p, DecodeSmem<GQ>& sm,
                                                    const unsigned char* st, const unsigned char* ptab_v,
                                                    float* obuf, int lane, int w,
                                                    float (&acc)[GQ][4], float (&macc)[GQ]) {
  const int k = p.geo.nout;
  const uint32_t* vms = reinterpret_cast<const uint32_t*>(st + NuqStage::VMS);
  const int bit = 12 * lane, wi = bit >> 5, sh = bit & 31;
  {
    // this lane's token: p * scale for the loop below; the V-min term
    // sum_t p_t min_t once for the warp
    const float2 ms = unpack_min_scale(vms[lane]);
#pragma unroll
    for (int r = 0; r < GQ; ++r) {
      const float pr = sm.p[w][lane][r];
      sm.pv[w][lane][r] = pr * ms.y;
      macc[r] += warp_sum(pr * ms.x);
    }
    __syncwarp();
  }
  const uint32_t loff = (uint32_t)(lane & 15) * 8u;
#pragma unroll 4
  for (int t = 0; t < kGroupTokens; ++t) {
    // this lane's 12 bits (word wi + 1 of the last row is the next region's
    // first word: in the stage, and shifted out)
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(st + NuqStage::VC + 48 * t);
    const uint32_t u = __funnelshift_r(rw[wi], rw[wi + 1], sh);
    const float2 c01 = *reinterpret_cast<const float2*>(ptab_v + (((u << 7) & 0x1F80u) | loff));
    const float2 c23 = *reinterpret_cast<const float2*>(ptab_v + (((u << 1) & 0x1F80u) | loff));
#pragma unroll
    for (int r = 0; r < GQ; ++r) {
      const float pp = sm.pv[w][t][r];
      const float2 pp2 = make_float2(pp, pp);
      const float2 a01 = __ffma2_rn(pp2, c01, make_float2(acc[r][0], acc[r][1]));
      const float2 a23 = __ffma2_rn(pp2, c23, make_float2(acc[r][2], acc[r][3]));
      acc[r][0] = a01.x;
      acc[r][1] = a01.y;
      acc[r][2] = a23.x;
      acc[r][3] = a23.y;
    }
  }
  if (k == 0) return;
  // outliers: lane t adds its own token's k entries (rows hold exactly k,
  // at entries t k .. t k + k - 1); columns of different tokens may meet
  const uint8_t* ocol = st + NuqStage::vcol(k) + k * lane;
  const uint16_t* oval = reinterpret_cast<const uint16_t*>(st + NuqStage::vval(k)) + k * lane;
  const float vmin = unpack_min_scale(vms[lane]).x;
  for (int e = 0; e < k; ++e) {
    const int col = ocol[e];
    const float dv = half_bits_to_float(oval[e]) - vmin;
#pragma unroll
    for (int r = 0; r < GQ; ++r) atomicAdd(&obuf[r * kHeadDim + col], sm.p[w][lane][r] * dv);
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < GQ; ++r) {
    float4* b4 = reinterpret_cast<float4*>(&obuf[r * kHeadDim + 4 * lane]);
    const float4 o = *b4;
    acc[r][0] += o.x;
    acc[r][1] += o.y;
    acc[r][2] += o.z;
    acc[r][3] += o.w;
    *b4 = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncwarp();
}

template <int KB, int VB, int GQ>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  DecodeSmem<GQ>& sm = *reinterpret_cast<DecodeSmem<GQ>*>(smem_raw);
  // NUQ: K and V pair tables first
  unsigned char* nuq_ptab = smem_raw + decode_smem_fixed<KB, GQ>();
  float2* rope_e = reinterpret_cast<float2*>(nuq_ptab + (KB == 3 ? 2 * kPairTableBytes : 0));
  const Geometry& G = p.geo;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int sp = blockIdx.x, s = blockIdx.y;
  const int b = s / G.Hkv, hk = s % G.Hkv, g = G.g;
  // this stream's tokens: the call's T, or its batch row's in a ragged call
  int T_s = p.T, S_eff = p.S_eff, Nq = p.Nq, Wn = p.W;
  if (p.ragged) {
    T_s = rows_tokens(p)[b];
    window_counts(G, T_s, &S_eff, &Nq, &Wn);
  }

  for (int idx = tid; idx < GQ * kHeadDim; idx += kThreads) {
    const int r = idx / kHeadDim, c = idx % kHeadDim;
    float v = 0.0f;
    if (r < g) v = half_bits_to_float(p.q[q_row(G, b, hk, r) * kHeadDim + c]) * p.q_scale;
    sm.q[r][c] = v;
  }
  if (tid < 8) {
    sm.lut_k[tid] = p.k_lut_off[tid];
    sm.lut_v[tid] = p.v_lut_off[tid];
  }
  if (G.pre_rope)
    for (int j = tid; j < kHeadDim / 2; j += kThreads)
      anchor_step(p.theta[j], (long long)G.pos_offset + G.S, &sm.anc_v[j], &sm.anc_c0[j]);
  const bool quant_split = sp < p.n_qsplit;
  constexpr bool kFolded = KB == 3 && GQ == 1;  // query-folded 16-offset table (built below)
  if (!kFolded && G.pre_rope && quant_split) {
    // e^{i l theta_j} at [j][l]: a warp reads one j for its 32 token offsets l,
    // 32 consecutive entries (no bank conflicts)
    for (int idx = tid; idx < kGroupTokens * (kHeadDim / 2); idx += kThreads) {
      const int j = idx / kGroupTokens, l = idx % kGroupTokens;
      rope_e[rope_tab_index(j, l)] = expi((double)l * p.theta[j]);
    }
  }
  // NUQ: per-warp K buffers and stages, then per-warp outlier buffers (zeroed)
  unsigned char* nuq_stages = reinterpret_cast<unsigned char*>(rope_e) +
                              (G.pre_rope ? rope_region_bytes<KB, GQ>() : 0);
  float* nuq_obuf = reinterpret_cast<float*>(nuq_stages + (KB == 3 ? 4 * NuqStage::warp_bytes(G.nout) : 0));
  if constexpr (KB == 3) {
    for (int idx = tid; idx < 4 * GQ * kHeadDim; idx += kThreads) nuq_obuf[idx] = 0.0f;
    for (int idx = tid; idx < 2 * kPairEntries * kPairCopies; idx += kThreads) {
      const int f = (idx / kPairCopies) % kPairEntries;
      const float* L = idx < kPairEntries * kPairCopies ? p.k_lut_off : p.v_lut_off;
      reinterpret_cast<float2*>(nuq_ptab)[idx] = make_float2(L[f & 7], L[f >> 3]);
    }
  }
  __syncthreads();
  if constexpr (KB == 3 && GQ == 1) {
    // one query head: the offset table with the query folded in,
    // W_{j,l} = conj(q_j + i q_{j+64}) e^{i l theta_j}, offsets l < 16
    if (G.pre_rope && quant_split) {
      // W of pairs 2i, 2i+1 for offset l as (x_2i, x_2i+1, y_2i, y_2i+1)
      float4* tab4 = reinterpret_cast<float4*>(rope_e);
      for (int idx = tid; idx < 16 * (kHeadDim / 4); idx += kThreads) {
        const int jp = idx / 16, l = idx % 16, j = 2 * jp;
        const float2 w0 = cmul(make_float2(sm.q[0][j], -sm.q[0][j + kHeadDim / 2]), expi((double)l * p.theta[j]));
        const float2 w1 =
            cmul(make_float2(sm.q[0][j + 1], -sm.q[0][j + 1 + kHeadDim / 2]), expi((double)l * p.theta[j + 1]));
        tab4[jp * 16 + l] = make_float4(w0.x, w1.x, w0.y, w1.y);
      }
      __syncthreads();
    }
  }
  if (tid < GQ) {
    float a = 0.0f;
    for (int c = 0; c < kHeadDim; ++c) a += sm.q[tid][c];
    sm.qsum[tid] = a;
  }
  __syncthreads();

  float m[GQ], lsum[GQ], acc[GQ][4], macc[GQ];
#pragma unroll
  for (int r = 0; r < GQ; ++r) {
    m[r] = -INFINITY;
    lsum[r] = 0.0f;
    macc[r] = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[r][k] = 0.0f;
  }

  if constexpr (KB == 3) if (quant_split) {
    // staged: group grp + 4 (this warp's next) streams in while grp is computed
    const int ngroups = Nq / kGroupTokens;
    const int g0 = sp * p.gps;
    const int g1 = min(ngroups, g0 + p.gps);
    const int sb = NuqStage::bytes(G.nout);
    unsigned char* kbw = nuq_stages + w * NuqStage::warp_bytes(G.nout);  // this warp's K buffer
    unsigned char* stw = kbw + NuqStage::KBUF;                           // and its two stages
    const uint32_t kbw_s = smem_u32(kbw), stw_s = smem_u32(stw);
    float* obuf = nuq_obuf + w * GQ * kHeadDim;
    int cur = 0;
    AnchorWalk aw;
    aw.left = 0;
    if (G.pre_rope) {
      // e^{i theta_j 4 G_K}: a warp's consecutive groups are 4 apart
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        aw.step[h] = expi(4.0 * kGroupTokens * p.theta[lane + 32 * h]);
        aw.half[h] = expi(16.0 * p.theta[lane + 32 * h]);
      }
    }
    if (g0 + w < g1) issue_nuq(p, s, g0 + w, kbw_s, stw_s, lane);
    cp_async_commit();
    for (int grp = g0 + w; grp < g1; grp += 4) {
      cp_async_wait<0>();
      __syncwarp();
      // this group's K rows into registers; then the next group streams in
      // (K rows into the freed buffer, the rest into the other stage)
      uint32_t wd[13];
      load_code_row(kbw, lane, wd);
      __syncwarp();
      if (grp + 4 < g1) issue_nuq(p, s, grp + 4, kbw_s, stw_s + (cur ^ 1) * sb, lane);
      cp_async_commit();
      const unsigned char* stc = stw + cur * sb;
      float z[GQ];
      k_logits_nuq_st<GQ>(p, sm, rope_e, nuq_ptab, wd, stc, grp, lane, w, z, aw);
      softmax_update<GQ>(z, m, lsum, acc, macc, sm.p[w], lane);
      v_accumulate_nuq_st<GQ>(p, sm, stc, nuq_ptab + kPairTableBytes, obuf, lane, w, acc, macc);
      __syncwarp();
      cur ^= 1;
    }
    cp_async_wait<0>();
  }
  if constexpr (KB != 16 && KB != 3) if (quant_split) {
    const int ngroups = Nq / kGroupTokens;
    const int g0 = sp * p.gps;
    const int g1 = min(ngroups, g0 + p.gps);
    for (int grp = g0 + w; grp < g1; grp += 4) {
      float z[GQ];
      if (G.pre_rope) {
        k_logits_rope<KB, GQ>(p, sm, rope_e, s, grp, lane, w, z);
      } else {
        k_logits_uniform<KB, GQ>(p, sm, s, grp, lane, w, z);
      }
      softmax_update<GQ>(z, m, lsum, acc, macc, sm.p[w], lane);
      v_accumulate<VB, GQ>(p, sm, s, grp, lane, w, acc, macc);
    }
  }
  if (!quant_split) {
    int k0, k1;
    if (G.fp16_mode) {
      k0 = sp * p.fp16_tokens_per_split;
      k1 = min(T_s, k0 + p.fp16_tokens_per_split);
    } else {
      k0 = 0;
      k1 = S_eff + Wn;
    }
    for (int c0 = k0 + 32 * w; c0 < k1; c0 += 32 * 4)
      fp16_chunk<GQ>(p, sm.q, sm.p[w], s, c0, k1, S_eff, Nq, lane, m, lsum, acc, macc);
  }

  // ---- combine the 4 warps of this CTA
#pragma unroll
  for (int r = 0; r < GQ; ++r) {
    lsum[r] = warp_sum(lsum[r]);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[r][k] += macc[r];
  }
  __syncthreads();  // all warps are done with sm.work
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < GQ; ++r) {
      sm.ml[w][r][0] = m[r];
      sm.ml[w][r][1] = lsum[r];
    }
  }
  // merge staging: `work`, or the (now idle) NUQ stages of a non-uniform launch
  float (*stage)[GQ][kHeadDim] = reinterpret_cast<float (*)[GQ][kHeadDim]>(
      KB == 3 ? reinterpret_cast<float*>(nuq_stages) : &sm.work[0][0][0]);
  static_assert(sizeof(sm.work) >= 4 * GQ * kHeadDim * sizeof(float), "merge staging");
  static_assert(KB != 3 || 4 * NuqStage::warp_bytes(0) >= 4 * GQ * kHeadDim * (int)sizeof(float), "merge staging");
#pragma unroll
  for (int r = 0; r < GQ; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k) stage[w][r][4 * lane + k] = acc[r][k];
  __syncthreads();
  if (tid < GQ) {
    float M = -INFINITY;
    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, sm.ml[ww][tid][0]);
    float Lc = 0.0f;
    for (int ww = 0; ww < 4; ++ww)
      if (sm.ml[ww][tid][0] != -INFINITY) Lc += exp2f(sm.ml[ww][tid][0] - M) * sm.ml[ww][tid][1];
    sm.comb_ml[tid][0] = M;
    sm.comb_ml[tid][1] = Lc;
  }
  // combined accumulator: thread per (head, channel), written into stage[0]
  float combined[GQ];
#pragma unroll
  for (int r = 0; r < GQ; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, sm.ml[ww][r][0]);
    float a = 0.0f;
#pragma unroll
    for (int ww = 0; ww < 4; ++ww)
      if (sm.ml[ww][r][0] != -INFINITY) a += exp2f(sm.ml[ww][r][0] - M) * stage[ww][r][tid];
    combined[r] = a;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < GQ; ++r) stage[0][r][tid] = combined[r];
  __syncthreads();

  const bool rotate_this = G.hadamard && quant_split;
  if (p.n_split == 1) {
    // single split: finish here
    for (int r = w; r < g; r += 4) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = stage[0][r][4 * lane + k];
      if (rotate_this) warp_fwht(v, p.hadamard_c, lane);
      const float Lc = sm.comb_ml[r][1];
      const size_t o = q_row(G, b, hk, r) * kHeadDim + 4 * lane;
      __half2 h0 = __floats2half2_rn(v[0] / Lc, v[1] / Lc), h1 = __floats2half2_rn(v[2] / Lc, v[3] / Lc);
      uint2 st;
      st.x = *reinterpret_cast<uint32_t*>(&h0);
      st.y = *reinterpret_cast<uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(p.out + o) = st;
      if (p.lse && lane == 0)
        p.lse[q_row(G, b, hk, r)] = (sm.comb_ml[r][0] + log2f(Lc)) * 0.6931471805599453f;
    }
    return;
  }

  // ---- write this split's partial, take a ticket; the last CTA merges
  {
    const size_t base = ((size_t)s * p.n_split + sp) * g;
    for (int r = 0; r < g; ++r) p.part_acc[(base + r) * kHeadDim + tid] = stage[0][r][tid];
    if (tid < g) {
      p.part_ml[(base + tid) * 2] = sm.comb_ml[tid][0];
      p.part_ml[(base + tid) * 2 + 1] = sm.comb_ml[tid][1];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&p.counters[s], 1u);
    sm.is_last = (prev == (unsigned)(p.n_split - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.is_last) return;
  __threadfence();

  for (int r = w; r < g; r += 4) {
    float M = -INFINITY;
    for (int q2 = 0; q2 < p.n_split; ++q2)
      M = fmaxf(M, __ldcg(&p.part_ml[(((size_t)s * p.n_split + q2) * g + r) * 2]));
    float Lc = 0.0f, oq[4] = {0, 0, 0, 0}, ow[4] = {0, 0, 0, 0};
    for (int q2 = 0; q2 < p.n_split; ++q2) {
      const size_t base = ((size_t)s * p.n_split + q2) * g + r;
      const float mq = __ldcg(&p.part_ml[base * 2]);
      if (mq == -INFINITY) continue;
      const float e = exp2f(mq - M);
      Lc += e * __ldcg(&p.part_ml[base * 2 + 1]);
      const float4 a = __ldcg(reinterpret_cast<const float4*>(&p.part_acc[base * kHeadDim + 4 * lane]));
      float* dst = (q2 < p.n_qsplit) ? oq : ow;
      dst[0] += e * a.x;
      dst[1] += e * a.y;
      dst[2] += e * a.z;
      dst[3] += e * a.w;
    }
    if (G.hadamard) warp_fwht(oq, p.hadamard_c, lane);
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = (oq[k] + ow[k]) / Lc;
    const size_t o = q_row(G, b, hk, r) * kHeadDim + 4 * lane;
    __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
    uint2 st;
    st.x = *reinterpret_cast<uint32_t*>(&h0);
    st.y = *reinterpret_cast<uint32_t*>(&h1);
    *reinterpret_cast<uint2*>(p.out + o) = st;
    if (p.lse && lane == 0) p.lse[q_row(G, b, hk, r)] = (M + log2f(Lc)) * 0.6931471805599453f;
  }
  if (tid == 0) p.counters[s] = 0u;
}

template <int KB, int VB, int GQ>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t st, int* occ) {
  const size_t smem = decode_smem_bytes<KB, GQ>(p.geo.pre_rope != 0, p.geo.nout);
  static std::atomic<long long> smem_memo[kMemoDevices], occ_memo[kMemoDevices];
  const cudaError_t e = ensure_smem_limit(decode_kernel<KB, VB, GQ>, smem_memo, (int)smem);
  if (e != cudaSuccess) return e;
  if (occ)  // resident CTAs per SM, for sizing the grid; no launch
    return occupancy_memo(decode_kernel<KB, VB, GQ>, occ_memo, kThreads, (int)smem, occ);
  dim3 grid(p.n_split, p.geo.NS);
  decode_kernel<KB, VB, GQ><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
