// kvq_decode_persist.cuh -- persistent decode: one resident wave of CTAs,
// every warp streaming its own byte-balanced range of work.
//
// The work of a layer is a list of items, stream by stream: the stream's
// quantized 32-token groups, then its fp16 tokens (sinks + recent window,
// or the whole cache in fp16 mode) in items of kF16Tokens tokens.  Items
// are weighted by the bytes they read and the list is cut into as many
// equal ranges as there are resident warps.  Every item -- quantized or
// fp16 -- goes through the warp's asynchronous-copy pipeline (kStages
// shared-memory stages), which runs across the warp's whole range, also
// across stream boundaries: there is no __syncthreads after the prologue.
//
// Accumulators: O (tensor-core D fragments: rows = channels, columns =
// (head, hi/lo), or heads for 5-8 heads -- head_cols), the running maximum
// m_used and the partial sums lsum.  The
// quantized part of a stream accumulates codes weighted by P' = p * scale_v
// (plus V min through macc) in the rotated domain when V is Hadamard-
// rotated.  When the warp reaches the stream's fp16 items (or the end of
// its piece of the stream) that part is folded into a per-warp staging
// buffer -- rotated back there (the rotation is linear, so rotating each
// partial before the sum equals rotating the sum) -- and O is reused for
// the fp16 tokens.  At the end of its piece the warp combines the two,
// stores one partial result (m, l, O per query head) in its slot and takes
// a ticket; the warp that takes the stream's last ticket merges the
// stream's partials by log-sum-exp and writes the output.  Nobody waits for
// anybody.  Slot of (warp i, stream s) = i + s: warp ranges are contiguous
// and ordered, so these are distinct and a stream's slots are consecutive.
#pragma once

#include "kvq_decode_mma.cuh"

namespace kvq {
namespace persist {

using namespace kvq::mma;

template <int KB, int VB, int NT, int GT, bool IQ = false>
struct PersistLayout {
  static constexpr bool kQuant = KB != 16;
  static constexpr int kStages = 2;  // per-warp pipeline depth (items)
  static constexpr int r128(int x) { return (x + 127) / 128 * 128; }
  // the warp's group scratch (InnerQ keys: plus the per-token K scales and the
  // stream's per-head constants)
  static constexpr int kSmem = r128((int)sizeof(MmaWarpSmem<NT>) + (IQ ? (int)sizeof(IqWarpSmem) : 0));
  static constexpr int kQBytes = kQuant ? StageGeom<KB, VB, IQ>::BYTES : 0;
  static constexpr int kStageBytes = kQBytes > F16Geom::BYTES ? kQBytes : F16Geom::BYTES;
  static constexpr int kPerWarpStages = kStages * kStageBytes;
  // this warp's stream's query; once the query is no longer needed (the
  // stream's Q' and fp16 fragments are built) the same bytes hold the
  // staged O[h][c], and the group-bias scratch holds the staged (m, l)
  static constexpr int kPerWarpQ = r128(GT * kHeadDim * 4);
  // a warp's region: scratch, pipeline stages, query
  static constexpr int kPerWarp = kSmem + kPerWarpStages + kPerWarpQ;
  // One CTA per SM holds all of the SM's warps (with several CTAs per SM the
  // warp schedulers favour the earlier CTAs, whose warps then finish their
  // equal shares well before the others).  Warps per SM as measured best:
  // 16 at 128 registers for single-head groups, 12 at 168 for 2-8 heads;
  // fewer when their shared memory would exceed a CTA's 227 KB.
  static constexpr int kWantWarps = GT == 1 ? 16 : 12;
  static constexpr int kMaxCtaSmem = 227 * 1024;
  static constexpr int kWarps = kWantWarps * kPerWarp <= kMaxCtaSmem ? kWantWarps : kMaxCtaSmem / kPerWarp;
  static constexpr int kCtaThreads = 32 * kWarps;
  static constexpr int kBytes = kWarps * kPerWarp;
  static_assert(kWarps >= 1, "one warp's region must fit in a CTA");
};

// Fold the quantized accumulators into the staging buffer: sO[h][c] = the
// (rotated back) sum of codes x P' plus the V-min term, sML[h] = (m, l).
// O, macc and lsum restart from zero; m_used carries on.
template <int VB, int NT, int GT, bool JC>
__device__ __forceinline__ void stage_quant(const DecodeParams& p, float* sO, float* sML, int g, int lane,
                                            float (&O)[8][o_tiles<NT>()][4], float (&macc)[NT][kNVG],
                                            float (&m_used)[NT], float (&lsum)[NT]) {
  constexpr bool HC = head_cols<NT>();
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], o);
#pragma unroll
      for (int j = 0; j < kNVG; ++j) macc[nt][j] += __shfl_xor_sync(0xffffffffu, macc[nt][j], o);
    }
    const int h = slot_head<NT>(nt, tq);
    if constexpr (JC) {
      // D columns of this lane: head tq >> 1, V group tq & 1; macc of that head from its lane
      const int hc = tq >> 1, jj = tq & 1;
      const float m0 = __shfl_sync(0xffffffffu, macc[0][0], (lane & ~3) | hc);
      const float m1 = __shfl_sync(0xffffffffu, macc[0][1], (lane & ~3) | hc);
      const float mj = jj ? m1 : m0;
      if (hc < g) {
#pragma unroll
        for (int mc = 0; mc < 8; ++mc) {
          if (v_group<VB>(mc) != jj) continue;
#pragma unroll
          for (int rh = 0; rh < 2; ++rh)
            sO[hc * kHeadDim + v_chan<VB>(mc, gq, rh)] = O[mc][0][2 * rh] + O[mc][0][2 * rh + 1] + mj;
        }
      }
      if (h < g && gq == 0) {
        sML[2 * h] = m_used[nt];
        sML[2 * h + 1] = lsum[nt];
      }
    } else if (h < g) {
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const float mt = macc[nt][v_group<VB>(mc)];
#pragma unroll
        for (int rh = 0; rh < 2; ++rh)
          sO[h * kHeadDim + v_chan<VB>(mc, gq, rh)] =
              (HC ? O[mc][0][2 * rh + nt] : O[mc][nt][2 * rh] + O[mc][nt][2 * rh + 1]) + mt;
      }
      if (gq == 0) {
        sML[2 * h] = m_used[nt];
        sML[2 * h + 1] = lsum[nt];
      }
    }
  }
  __syncwarp();
  if (p.geo.hadamard) {
#pragma unroll
    for (int r = 0; r < GT; ++r) {
      if (r >= g) break;
      float* row = &sO[r * kHeadDim + 4 * lane];
      const float4 a = *reinterpret_cast<const float4*>(row);
      float v[4] = {a.x, a.y, a.z, a.w};
      if (sML[2 * r] != -INFINITY) warp_fwht(v, p.hadamard_c, lane);
      *reinterpret_cast<float4*>(row) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncwarp();
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    lsum[nt] = 0.0f;
#pragma unroll
    for (int j = 0; j < kNVG; ++j) macc[nt][j] = 0.0f;
  }
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int ot = 0; ot < o_tiles<NT>(); ++ot)
#pragma unroll
      for (int k = 0; k < 4; ++k) O[mc][ot][k] = 0.0f;
}

// End of this warp's piece of stream s: combine the staged quantized part
// (if any) with the fp16 part held in O (plain channel order), store the
// slot, take a ticket, and merge the stream if this was the last piece.
// PAIR: merge two heads at a time (see below)
template <int NT, int GT, bool PAIR>
__device__ __forceinline__ void finalize_stream(const DecodeParams& p, int slot, int s, int wf, int count, float* sO,
                                                float* sML, bool staged, int lane,
                                                const float (&O)[8][o_tiles<NT>()][4],
                                                const float (&m_used)[NT], float (&lsum)[NT]) {
  const Geometry& G = p.geo;
  const int g = G.g;
  const int gq = lane >> 2, tq = lane & 3;
  float mqv[NT], lqv[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], o);
    const int h = slot_head<NT>(nt, tq);
    mqv[nt] = (staged && h < g) ? sML[2 * h] : -INFINITY;
    lqv[nt] = (staged && h < g) ? sML[2 * h + 1] : 0.0f;
  }
  __syncwarp();  // every lane has read the staged (m, l) before they are overwritten
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = slot_head<NT>(nt, tq);
    if (h < g) {
      const float M = fmaxf(mqv[nt], m_used[nt]);
      const float eq = (mqv[nt] == -INFINITY) ? 0.0f : exp2f(mqv[nt] - M);
      const float et = (m_used[nt] == -INFINITY) ? 0.0f : exp2f(m_used[nt] - M);
#pragma unroll
      for (int mc = 0; mc < 8; ++mc)
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          float* d = &sO[h * kHeadDim + 16 * mc + 8 * rh + gq];
          const float t = et * (head_cols<NT>() ? O[mc][0][2 * rh + nt] : O[mc][nt][2 * rh] + O[mc][nt][2 * rh + 1]);
          *d = staged ? fmaf(eq, *d, t) : t;
        }
      if (gq == 0) {
        sML[2 * h] = M;
        sML[2 * h + 1] = eq * lqv[nt] + et * lsum[nt];
      }
    }
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < GT; ++r) {
    if (r >= g) break;
    const float4 a = *reinterpret_cast<const float4*>(&sO[r * kHeadDim + 4 * lane]);
    const size_t base = (size_t)slot * g + r;
    *reinterpret_cast<float4*>(&p.part_acc[base * kHeadDim + 4 * lane]) = a;
    if (lane == 0) {
      p.part_ml[base * 2] = sML[2 * r];
      p.part_ml[base * 2 + 1] = sML[2 * r + 1];
    }
  }
  __syncwarp();
  __threadfence();
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(&p.counters[s], 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != (unsigned)(count - 1)) return;
  __threadfence();
  // last piece of stream s: merge its slots wf + s .. wf + s + count - 1.
  // Lane q reads slot q's (m, l); the first kMB slots' accumulators are read
  // in the same round trip (4 channels per lane), later ones kMB at a time.
  // Single-head streams have ~10 slots and registers to spare at this point
  // (measured: 16 at a time is faster there, 8 for larger groups).  With
  // PAIR, heads are merged two at a time so that their reads share the
  // round trips: one head after the other, the merges of a 4-head stream's
  // ~14 slots were the last ~8 µs of a 32k layer.  Measured per layer kind,
  // pairing is faster for 8-bit keys, InnerQ keys and 8 head slots, and
  // slower (the kernel around it compiles differently) for the 2- and
  // 4-bit per-channel-key layers with 4 head slots.
  constexpr int kMB = GT == 1 ? 16 : 8;
  constexpr int H = PAIR && GT > 1 ? 2 : 1;
  const int b = s / G.Hkv, hk = s % G.Hkv;
  const size_t slot0 = (size_t)(wf + s);
  for (int r0 = 0; r0 < g; r0 += H) {
    bool live[H];
#pragma unroll
    for (int h = 0; h < H; ++h) live[h] = r0 + h < g;  // warp-uniform
    auto acc_at = [&](int h, int q) {
      return __ldcg(reinterpret_cast<const float4*>(&p.part_acc[((slot0 + q) * g + r0 + h) * kHeadDim + 4 * lane]));
    };
    auto ml_at = [&](int h, int q, int i) { return __ldcg(&p.part_ml[((slot0 + q) * g + r0 + h) * 2 + i]); };
    float mq[H], lq[H];
    float4 a[H][kMB];
#pragma unroll
    for (int h = 0; h < H; ++h) {
      mq[h] = -INFINITY;
      lq[h] = 0.0f;
      if (live[h] && lane < count) {
        mq[h] = ml_at(h, lane, 0);
        lq[h] = ml_at(h, lane, 1);
      }
#pragma unroll
      for (int u = 0; u < kMB; ++u) a[h][u] = live[h] && u < count ? acc_at(h, u) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float M[H], L[H], v[H][4];
#pragma unroll
    for (int h = 0; h < H; ++h) {
      M[h] = mq[h];
      if (live[h])
        for (int q0 = lane + 32; q0 < count; q0 += 32) M[h] = fmaxf(M[h], ml_at(h, q0, 0));
      M[h] = warp_max(M[h]);
      L[h] = 0.0f;
      v[h][0] = v[h][1] = v[h][2] = v[h][3] = 0.0f;
    }
    for (int c0 = 0; c0 < count; c0 += 32) {
      // lane q: weight of slot c0 + q
      float e[H];
#pragma unroll
      for (int h = 0; h < H; ++h) {
        if (c0 > 0 && live[h] && c0 + lane < count) {
          mq[h] = ml_at(h, c0 + lane, 0);
          lq[h] = ml_at(h, c0 + lane, 1);
        }
        e[h] = 0.0f;
        if (c0 + lane < count) {
          e[h] = (mq[h] == -INFINITY) ? 0.0f : exp2f(mq[h] - M[h]);
          L[h] += e[h] * lq[h];
        }
      }
      const int n = min(32, count - c0);
      for (int q = 0; q < n; q += kMB) {
        if (c0 + q > 0) {
#pragma unroll
          for (int h = 0; h < H; ++h)
#pragma unroll
            for (int u = 0; u < kMB; ++u)
              a[h][u] = live[h] && q + u < n ? acc_at(h, c0 + q + u) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMB; ++u)
#pragma unroll
          for (int h = 0; h < H; ++h) {
            const float eq = __shfl_sync(0xffffffffu, e[h], (q + u) & 31);  // 0 past the last slot
            v[h][0] = fmaf(eq, a[h][u].x, v[h][0]);
            v[h][1] = fmaf(eq, a[h][u].y, v[h][1]);
            v[h][2] = fmaf(eq, a[h][u].z, v[h][2]);
            v[h][3] = fmaf(eq, a[h][u].w, v[h][3]);
          }
      }
    }
#pragma unroll
    for (int h = 0; h < H; ++h) {
      if (!live[h]) continue;
      const int r = r0 + h;
      const float Lh = warp_sum(L[h]);
      const size_t o = q_row(G, b, hk, r) * kHeadDim + 4 * lane;
      const __half2 h0 = __floats2half2_rn(v[h][0] / Lh, v[h][1] / Lh), h1 = __floats2half2_rn(v[h][2] / Lh, v[h][3] / Lh);
      uint2 stv;
      stv.x = h2_as_u32(h0);
      stv.y = h2_as_u32(h1);
      *reinterpret_cast<uint2*>(p.out + o) = stv;
      if (p.lse && lane == 0) p.lse[q_row(G, b, hk, r)] = (M[h] + log2f(Lh)) * 0.6931471805599453f;
    }
  }
  if (lane == 0) p.counters[s] = 0u;
}

// The counts of the stream a walker (the issue side or the processing side
// of a warp's range) is in: quantized groups, items, fp16 tokens and the
// window counts that address them.  Uniform calls read them from the launch
// parameters (every stream alike); ragged ones keep the current stream's.
template <bool RG>
struct Walk {
  __device__ __forceinline__ void set(const DecodeParams&, int) {}
  __device__ __forceinline__ int ng(const DecodeParams& p) const { return p.ng; }
  __device__ __forceinline__ int n_items(const DecodeParams& p) const { return p.n_items; }
  __device__ __forceinline__ int k1(const DecodeParams& p) const { return p.S_eff + p.W; }
  __device__ __forceinline__ int S_eff(const DecodeParams& p) const { return p.S_eff; }
  __device__ __forceinline__ int Nq(const DecodeParams& p) const { return p.Nq; }
};
template <>
struct Walk<true> {
  int ng_, n_, k1_, se_, nq_;
  __device__ __forceinline__ void set(const DecodeParams& p, int s) {
    const StreamSpan r = stream_span_t<true>(p, s);
    ng_ = r.ng;
    n_ = r.n_items;
    k1_ = r.k1;
    se_ = r.S_eff;
    nq_ = r.Nq;
  }
  __device__ __forceinline__ int ng(const DecodeParams&) const { return ng_; }
  __device__ __forceinline__ int n_items(const DecodeParams&) const { return n_; }
  __device__ __forceinline__ int k1(const DecodeParams&) const { return k1_; }
  __device__ __forceinline__ int S_eff(const DecodeParams&) const { return se_; }
  __device__ __forceinline__ int Nq(const DecodeParams&) const { return nq_; }
};

// RG: a ragged call (every stream at its batch row's length; the row tables
// in the workspace), compiled separately so that the uniform schedule
// carries none of it.
template <int KB, int VB, int NT, int GT, bool IQ = false, bool RG = false>
__global__ void __launch_bounds__(PersistLayout<KB, VB, NT, GT, IQ>::kCtaThreads, 1)
    decode_persist_kernel(const __grid_constant__ DecodeParams p) {
  using LY = PersistLayout<KB, VB, NT, GT, IQ>;
  constexpr int KBq = KB == 16 ? 4 : KB, VBq = VB == 16 ? 4 : VB;  // fp16 mode: quantized helpers unused
  constexpr bool JC = NT == 1 && GT <= 2;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const Geometry& G = p.geo;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = G.g;
  unsigned char* mine = smem_raw + w * LY::kPerWarp;  // this warp's region; no CTA-wide sharing
  MmaWarpSmem<NT>& sm = *reinterpret_cast<MmaWarpSmem<NT>*>(mine);
  IqWarpSmem* iq = IQ ? reinterpret_cast<IqWarpSmem*>(mine + sizeof(MmaWarpSmem<NT>)) : nullptr;
  unsigned char* st0 = mine + LY::kSmem;
  const uint32_t st0_s = smem_u32(st0);
  float (*qw)[kHeadDim] = reinterpret_cast<float (*)[kHeadDim]>(mine + LY::kSmem + LY::kPerWarpStages);
  float* sO = &qw[0][0];     // staging, after the query's last use
  float* sML = &sm.bias[0];  // staging (m, l): 8 * NT >= 2 * GT floats

  const int gw = blockIdx.x * LY::kWarps + w;  // global warp index
  if (gw >= p.nwarps) return;
  long long j0, j1;
  if constexpr (RG) {
    // tables in the workspace were written by the kernel before; inline
    // ones need nothing earlier (the schedule overlaps that kernel)
    if (!p.rows_inline) grid_dep_wait();
    // the rows of this warp's range by a warp-wide search of the row tables
    const long long x0 = warp_x(p, gw), x1 = warp_x(p, gw + 1);
    const int b0 = row_at_warp(rows_x0(p), G.B, x0, lane), b1 = row_at_warp(rows_x0(p), G.B, x1, lane);
    j0 = x0 >= p.wtot ? rows_j0(p)[G.B] : first_item_in_row(p, x0, b0);
    j1 = x1 >= p.wtot ? rows_j0(p)[G.B] : first_item_in_row(p, x1, b1);
  } else {
    j0 = first_item_at_t<false>(p, warp_x(p, gw));
    j1 = first_item_at_t<false>(p, warp_x(p, gw + 1));
  }
  if (j0 >= j1) return;

  float O[8][o_tiles<NT>()][4], macc[NT][kNVG], m_used[NT], lsum[NT];
  auto reset = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_used[nt] = -INFINITY;
      lsum[nt] = 0.0f;
#pragma unroll
      for (int j = 0; j < kNVG; ++j) macc[nt][j] = 0.0f;
    }
#pragma unroll
    for (int mc = 0; mc < 8; ++mc)
#pragma unroll
      for (int ot = 0; ot < o_tiles<NT>(); ++ot)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[mc][ot][k] = 0.0f;
  };
  reset();

  // current item (s, k) and the next item to queue (is, ik, ij); all advance
  // incrementally, each with its stream's counts (sp, isp: quantized groups,
  // items, fp16 tokens), refreshed when it moves to the next stream
  int s, k;
  if constexpr (RG) locate_in_row(p, j0, row_at_warp(rows_j0(p), G.B, j0, lane), &s, &k);
  else locate_item_t<false>(p, j0, &s, &k);
  Walk<RG> sw;
  sw.set(p, s);
  int is = s, ik = k;
  Walk<RG> isw = sw;
  long long ij = j0;
  auto issue_next = [&](int stage) {
    if (ij < j1) {
      const uint32_t dst = st0_s + stage * LY::kStageBytes;
      const int ng = LY::kQuant ? isw.ng(p) : 0;
      if (LY::kQuant && ik < ng) {
        if constexpr (LY::kQuant) issue_group<KBq, VBq, IQ>(p, is, ik, dst, lane);
      } else {
        issue_f16(p, is, kF16Tokens * (ik - ng), isw.k1(p), isw.S_eff(p), isw.Nq(p), dst, lane);
      }
      ++ij;
      if (++ik == isw.n_items(p)) {
        ik = 0;
        ++is;
        if constexpr (RG) {
          if (ij < j1) isw.set(p, is);
        }
      }
    }
    cp_async_commit();
  };
  {
    // this warp's Q' rows start at zero (rows of absent heads stay zero)
    uint4* z = reinterpret_cast<uint4*>(&sm.bq[0][0][0]);
    for (int idx = lane; idx < (int)(sizeof(sm.bq) / 16); idx += 32) z[idx] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
  }
  // everything above used only the parameters and shared memory; the cache,
  // the query and the workspace may still be written by the previous kernel
  grid_dep_wait();
  grid_dep_trigger();
#pragma unroll
  for (int i = 0; i < LY::kStages - 1; ++i) issue_next(i);
  int cur = 0;
  int cur_s = -1;
  bool has_q = false, staged = false, bq_f16 = false;

  auto finish = [&](int sf) {
    if (has_q) stage_quant<VBq, NT, GT, JC>(p, sO, sML, g, lane, O, macc, m_used, lsum);
    staged = staged || has_q;
    const StreamSpan fs = stream_span_t<RG>(p, sf);
    const int wf = owner_of(p, item_pos_in(p, fs, 0));
    const int wl = owner_of(p, item_pos_in(p, fs, fs.n_items - 1));
    finalize_stream<NT, GT, (KB == 8 || IQ || GT == 8)>(p, gw + sf, sf, wf, wl - wf + 1, sO, sML, staged, lane, O,
                                                         m_used, lsum);
    reset();
    has_q = staged = bq_f16 = false;
  };

  for (long long j = j0; j < j1; ++j) {
    {
      const int nxt = cur + LY::kStages - 1;
      issue_next(nxt >= LY::kStages ? nxt - LY::kStages : nxt);
    }
    if (s != cur_s) {
      if (cur_s >= 0) finish(cur_s);
      cur_s = s;
      // this stream's query heads (scaled, fp32) into this warp's buffer, in
      // the Q'-build order (qb_perm_pos): lane L's channels c0, c0 + D, c0 + 1,
      // c0 + D + 1 (two adjacent pairs in global memory)
      const int b = s / G.Hkv, hk = s - b * G.Hkv;
      constexpr int D = qb_pair_dist<KBq>();
      const int c0 = qb_first_channel<KBq>(lane);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < GT; ++r) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < g) {
          const uint16_t* qr = p.q + q_row(G, b, hk, r) * kHeadDim;
          const float2 a = __half22float2(u32_as_h2(__ldg(reinterpret_cast<const uint32_t*>(qr + c0))));
          const float2 c2 = __half22float2(u32_as_h2(__ldg(reinterpret_cast<const uint32_t*>(qr + c0 + D))));
          v = make_float4(a.x * p.q_scale, c2.x * p.q_scale, a.y * p.q_scale, c2.y * p.q_scale);
        }
        *reinterpret_cast<float4*>(&qw[r][4 * lane]) = v;
      }
      __syncwarp();
      // InnerQ keys: the stream's Q' fragments and per-head constants, once
      if constexpr (IQ && LY::kQuant)
        build_bq_iq<KBq, NT>(qw, G.knorm ? p.L.k_norm + (size_t)s * kHeadDim : nullptr, sm, *iq, g, lane);
    }
    cp_async_wait<LY::kStages - 1>();
    __syncwarp();
    const unsigned char* stc = st0 + cur * LY::kStageBytes;
    const int ng = LY::kQuant ? sw.ng(p) : 0;
    if (LY::kQuant && k < ng) {
      if constexpr (LY::kQuant) {
        process_group<KB, VB, NT, JC, GT, IQ>(qw, sm, iq, stc, g, lane, O, macc, m_used, lsum);
        has_q = true;
      }
    } else {
      if (!bq_f16) {
        build_bq_f16<NT, KBq>(qw, sm, g, lane);  // the query's last use: sO may now overwrite it
        bq_f16 = true;
        __syncwarp();
        if (has_q) {
          stage_quant<VBq, NT, GT, JC>(p, sO, sML, g, lane, O, macc, m_used, lsum);
          has_q = false;
          staged = true;
        }
      }
      process_f16<NT>(sm, stc, g, lane, kF16Tokens * (k - ng), sw.k1(p), O, m_used, lsum);
    }
    __syncwarp();
    cur = (cur + 1 == LY::kStages) ? 0 : cur + 1;
    if (++k == sw.n_items(p)) {
      k = 0;
      ++s;
      if constexpr (RG) {
        if (j + 1 < j1) sw.set(p, s);
      }
    }
  }
  cp_async_wait<0>();
  if (cur_s >= 0) finish(cur_s);
}

}  // namespace persist
}  // namespace kvq

namespace kvq {
namespace persist {

template <int KB, int VB, int GT, bool IQ>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t st) {
  constexpr int NT = GT <= 4 ? 1 : 2;
  using LY = PersistLayout<KB, VB, NT, GT, IQ>;
  const int smem = LY::kBytes;
  const int ctas = (p.nwarps + LY::kWarps - 1) / LY::kWarps;
  if (p.ragged) {
    static std::atomic<long long> smem_memo_rg[kMemoDevices];
    cudaError_t e = ensure_smem_limit(decode_persist_kernel<KB, VB, NT, GT, IQ, true>, smem_memo_rg, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_persist_kernel<KB, VB, NT, GT, IQ, true>, dim3(ctas), dim3(LY::kCtaThreads),
                            smem, st, p);
  }
  static std::atomic<long long> smem_memo[kMemoDevices];
  cudaError_t e = ensure_smem_limit(decode_persist_kernel<KB, VB, NT, GT, IQ>, smem_memo, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_persist_kernel<KB, VB, NT, GT, IQ>, dim3(ctas), dim3(LY::kCtaThreads), smem, st,
                          p);
}

// Resident warps per SM of an instantiation (for sizing the persistent grid).
template <int KB, int VB, int GT, bool IQ>
cudaError_t occupancy_t(int* warps_per_sm) {
  constexpr int NT = GT <= 4 ? 1 : 2;
  using LY = PersistLayout<KB, VB, NT, GT, IQ>;
  const int smem = LY::kBytes;
  static std::atomic<long long> smem_memo[kMemoDevices], occ_memo[kMemoDevices];
  cudaError_t e = ensure_smem_limit(decode_persist_kernel<KB, VB, NT, GT, IQ>, smem_memo, smem);
  if (e != cudaSuccess) return e;
  int ctas = 0;
  e = occupancy_memo(decode_persist_kernel<KB, VB, NT, GT, IQ>, occ_memo, LY::kCtaThreads, smem, &ctas);
  *warps_per_sm = ctas * LY::kWarps;
  return e;
}

template <int KB, int VB, bool IQ = false>
cudaError_t dispatch_gt(const DecodeParams& p, cudaStream_t st, int* occ) {
  const int g = p.geo.g;
  if (occ) {
    if (g <= 1) return occupancy_t<KB, VB, 1, IQ>(occ);
    if (g <= 2) return occupancy_t<KB, VB, 2, IQ>(occ);
    if (g <= 4) return occupancy_t<KB, VB, 4, IQ>(occ);
    return occupancy_t<KB, VB, 8, IQ>(occ);
  }
  if (g <= 1) return launch_t<KB, VB, 1, IQ>(p, st);
  if (g <= 2) return launch_t<KB, VB, 2, IQ>(p, st);
  if (g <= 4) return launch_t<KB, VB, 4, IQ>(p, st);
  return launch_t<KB, VB, 8, IQ>(p, st);
}

template <int KB, bool IQ = false>
cudaError_t dispatch_vb(const DecodeParams& p, cudaStream_t st, int* occ) {
  switch (p.geo.vb) {
    case 2: return dispatch_gt<KB, 2, IQ>(p, st, occ);
    case 4: return dispatch_gt<KB, 4, IQ>(p, st, occ);
    case 8: return dispatch_gt<KB, 8, IQ>(p, st, occ);
  }
  return cudaErrorInvalidValue;
}

}  // namespace persist
}  // namespace kvq
