// kvq_decode_persist.cuh -- persistent decode: one resident wave of CTAs,
// every warp streaming its own byte-balanced range of work.
//
// The work of a layer is a list of items, stream by stream: the stream's
// quantized 32-token groups, then its fp16 tokens (sinks + recent window,
// or the whole cache in fp16 mode) in 32-token chunks.  Items are weighted
// by the bytes they read and the list is cut into as many equal ranges as
// there are resident warps.  A warp keeps its cp.async double buffer
// running across its whole range -- also across stream boundaries -- so the
// memory pipeline never drains at a barrier: there is no __syncthreads after
// the prologue.
//
// When a warp leaves a stream it folds what it has into one partial result
// (m, l, O per query head; the quantized part of O already rotated back in
// Hadamard mode -- the rotation is linear, so rotating each partial before
// the sum equals rotating the sum), stores it in its slot, and takes a
// ticket; the warp that takes the stream's last ticket merges the stream's
// partials by log-sum-exp and writes the output.  Nobody waits for anybody.
// Slot of (warp i, stream s) = i + s: warp ranges are contiguous and
// ordered, so these are distinct and a stream's slots are consecutive.
#pragma once

#include "kvq_decode_mma.cuh"

namespace kvq {
namespace persist {

using namespace kvq::mma;

template <int KB, int VB, int NT, int GT>
struct PersistLayout {
  static constexpr bool kQuant = KB != 16;
  static constexpr int kFixed = (int)((sizeof(MmaWarpSmem<NT>) + 127) / 128 * 128);
  static constexpr int kStageBytes = kQuant ? StageGeom<KB, VB>::BYTES : 0;
  static constexpr int kPerWarpStages = 2 * kStageBytes;
  static constexpr int r128(int x) { return (x + 127) / 128 * 128; }
  static constexpr int kPerWarpO = r128(GT * kHeadDim * 4 + GT * 2 * 4);  // staging O[h][c] + (m, l)
  static constexpr int kPerWarpP = r128(kGroupTokens * GT * 4);          // fp16 chunk softmax weights
  static constexpr int kPerWarpQ = r128(GT * kHeadDim * 4);              // this warp's stream's query
  static constexpr int kPerWarp = kPerWarpStages + kPerWarpO + kPerWarpP + kPerWarpQ;
  static constexpr int kBytes = kFixed + 4 * kPerWarp;
};

// Fold this warp's accumulators for stream s into its slot, take a ticket,
// and merge the stream if this was the last piece.
template <int VB, int NT, int GT>
__device__ __forceinline__ void finalize_stream(const DecodeParams& p, int slot, int s, int wf, int count,
                                                float* sO, float* sML, int lane, float (&O)[8][NT][4],
                                                float (&macc)[NT][kNVG], float (&m_used)[NT], float (&lsum)[NT],
                                                float (&m_t)[GT], float (&l_t)[GT], float (&acc_t)[GT][4],
                                                float (&macc_t)[GT]) {
  const Geometry& G = p.geo;
  const int g = G.g;
  const int gq = lane >> 2, tq = lane & 3;
  // quantized part: reduce over the 8 row groups, stage O[h][c] and (m, l)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], o);
#pragma unroll
      for (int j = 0; j < kNVG; ++j) macc[nt][j] += __shfl_xor_sync(0xffffffffu, macc[nt][j], o);
    }
    const int h = 4 * nt + tq;
    if (h < g) {
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const float mt = macc[nt][v_group<VB>(mc)];
#pragma unroll
        for (int rh = 0; rh < 2; ++rh)
          sO[h * kHeadDim + v_chan<VB>(mc, gq, rh)] = O[mc][nt][2 * rh] + O[mc][nt][2 * rh + 1] + mt;
      }
      if (gq == 0) {
        sML[2 * h] = m_used[nt];
        sML[2 * h + 1] = lsum[nt];
      }
    }
  }
  __syncwarp();
  // per head: rotate the quantized part back, add the fp16 part, store the slot
#pragma unroll
  for (int r = 0; r < GT; ++r) {
    if (r >= g) break;
    float vq[4];
    const float4 a = *reinterpret_cast<const float4*>(&sO[r * kHeadDim + 4 * lane]);
    vq[0] = a.x; vq[1] = a.y; vq[2] = a.z; vq[3] = a.w;
    const float mq = sML[2 * r], lq = sML[2 * r + 1];
    if (G.hadamard && mq != -INFINITY) warp_fwht(vq, p.hadamard_c, lane);
    const float lt = warp_sum(l_t[r]);
    const float M = fmaxf(mq, m_t[r]);
    const float eq = (mq == -INFINITY) ? 0.0f : exp2f(mq - M);
    const float et = (m_t[r] == -INFINITY) ? 0.0f : exp2f(m_t[r] - M);
    float4 o;
    o.x = eq * vq[0] + et * (acc_t[r][0] + macc_t[r]);
    o.y = eq * vq[1] + et * (acc_t[r][1] + macc_t[r]);
    o.z = eq * vq[2] + et * (acc_t[r][2] + macc_t[r]);
    o.w = eq * vq[3] + et * (acc_t[r][3] + macc_t[r]);
    const size_t base = (size_t)slot * g + r;
    *reinterpret_cast<float4*>(&p.part_acc[base * kHeadDim + 4 * lane]) = o;
    if (lane == 0) {
      p.part_ml[base * 2] = M;
      p.part_ml[base * 2 + 1] = eq * lq + et * lt;
    }
  }
  __syncwarp();
  __threadfence();
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(&p.counters[s], 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != (unsigned)(count - 1)) return;
  __threadfence();
  // last piece of stream s: merge its slots wf + s .. wf + s + count - 1
  const int b = s / G.Hkv, hk = s % G.Hkv;
  for (int r = 0; r < g; ++r) {
    float M = -INFINITY;
    for (int q2 = 0; q2 < count; ++q2)
      M = fmaxf(M, __ldcg(&p.part_ml[((size_t)(wf + s + q2) * g + r) * 2]));
    float L = 0.0f, v[4] = {0, 0, 0, 0};
    for (int q2 = 0; q2 < count; ++q2) {
      const size_t base = (size_t)(wf + s + q2) * g + r;
      const float mq = __ldcg(&p.part_ml[base * 2]);
      if (mq == -INFINITY) continue;
      const float e = exp2f(mq - M);
      L += e * __ldcg(&p.part_ml[base * 2 + 1]);
      const float4 a = __ldcg(reinterpret_cast<const float4*>(&p.part_acc[base * kHeadDim + 4 * lane]));
      v[0] += e * a.x;
      v[1] += e * a.y;
      v[2] += e * a.z;
      v[3] += e * a.w;
    }
    const size_t o = ((size_t)b * G.Hq + hk * g + r) * kHeadDim + 4 * lane;
    const __half2 h0 = __floats2half2_rn(v[0] / L, v[1] / L), h1 = __floats2half2_rn(v[2] / L, v[3] / L);
    uint2 stv;
    stv.x = h2_as_u32(h0);
    stv.y = h2_as_u32(h1);
    *reinterpret_cast<uint2*>(p.out + o) = stv;
    if (p.lse && lane == 0) p.lse[(size_t)b * G.Hq + hk * g + r] = (M + log2f(L)) * 0.6931471805599453f;
  }
  if (lane == 0) p.counters[s] = 0u;
}

template <int KB, int VB, int NT, int GT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 3 : 2) decode_persist_kernel(const __grid_constant__ DecodeParams p) {
  using LY = PersistLayout<KB, VB, NT, GT>;
  constexpr int GQ = 8 * NT;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  MmaWarpSmem<NT>& sm = *reinterpret_cast<MmaWarpSmem<NT>*>(smem_raw);
  const Geometry& G = p.geo;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = G.g;
  unsigned char* mine = smem_raw + LY::kFixed + w * LY::kPerWarp;
  unsigned char* st0 = mine;
  float* sO = reinterpret_cast<float*>(mine + LY::kPerWarpStages);
  float* sML = sO + GT * kHeadDim;
  float (*pbuf)[GT] = reinterpret_cast<float (*)[GT]>(mine + LY::kPerWarpStages + LY::kPerWarpO);
  float (*qw)[kHeadDim] =
      reinterpret_cast<float (*)[kHeadDim]>(mine + LY::kPerWarpStages + LY::kPerWarpO + LY::kPerWarpP);

  {
    uint32_t* z = reinterpret_cast<uint32_t*>(&sm.bq[0][0][0][0]);
    for (int idx = tid; idx < (int)(sizeof(sm.bq) / 4); idx += kThreads) z[idx] = 0u;
  }
  __syncthreads();

  const int gw = blockIdx.x * 4 + w;  // global warp index
  if (gw >= p.nwarps) return;
  const long long j0 = first_item_at(p, warp_x(p, gw));
  const long long j1 = first_item_at(p, warp_x(p, gw + 1));
  if (j0 >= j1) return;

  int qoff[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int s_, e_;
    k_slot_of<(KB == 16 ? 4 : KB)>(4 * (lane & 7) + k, s_, e_);
    qoff[k] = 4 * s_ + e_;
  }

  float O[8][NT][4], macc[NT][kNVG], m_used[NT], lsum[NT];
  float m_t[GT], l_t[GT], acc_t[GT][4], macc_t[GT];
  auto reset = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_used[nt] = -INFINITY;
      lsum[nt] = 0.0f;
#pragma unroll
      for (int j = 0; j < kNVG; ++j) macc[nt][j] = 0.0f;
#pragma unroll
      for (int mc = 0; mc < 8; ++mc)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[mc][nt][k] = 0.0f;
    }
#pragma unroll
    for (int r = 0; r < GT; ++r) {
      m_t[r] = -INFINITY;
      l_t[r] = 0.0f;
      macc_t[r] = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) acc_t[r][k] = 0.0f;
    }
  };
  reset();

  // next quantized item at or after j (within this warp's range), else j1
  auto next_q = [&](long long j) -> long long {
    if (!LY::kQuant || p.ng == 0) return j1;
    while (j < j1) {
      const long long k = j % p.n_items;
      if (k < p.ng) return j;
      j += p.n_items - k;  // first item of the next stream
    }
    return j1;
  };
  auto issue = [&](long long j, int stage) {
    if constexpr (LY::kQuant) {
      const int s = (int)(j / p.n_items), grp = (int)(j % p.n_items);
      issue_group<(KB == 16 ? 4 : KB), (VB == 16 ? 4 : VB)>(p, s, grp, st0 + stage * LY::kStageBytes, lane);
    }
  };

  long long qa = next_q(j0);
  if (qa < j1) issue(qa, 0);
  cp_async_commit();
  long long qb = (qa < j1) ? next_q(qa + 1) : j1;
  int cur = 0;
  int cur_s = -1;

  auto finish = [&](int s) {
    const long long first = (long long)s * p.n_items;
    const int wf = owner_of(p, item_pos(p, first));
    const int wl = owner_of(p, item_pos(p, first + p.n_items - 1));
    finalize_stream<(VB == 16 ? 4 : VB), NT, GT>(p, gw + s, s, wf, wl - wf + 1, sO, sML, lane, O, macc, m_used,
                                                 lsum, m_t, l_t, acc_t, macc_t);
    reset();
  };

  for (long long j = j0; j < j1; ++j) {
    const int s = (int)(j / p.n_items);
    const int k = (int)(j % p.n_items);
    if (s != cur_s) {
      if (cur_s >= 0) finish(cur_s);
      cur_s = s;
      {
        // this stream's query heads (scaled, fp32) into this warp's buffer
        const int b = s / G.Hkv, hk = s % G.Hkv;
        __syncwarp();
        for (int idx = lane; idx < GT * kHeadDim / 4; idx += 32) {
          const int r = idx / (kHeadDim / 4), c4 = idx % (kHeadDim / 4);
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r < g) {
            const uint2 u =
                __ldg(reinterpret_cast<const uint2*>(p.q + ((size_t)b * G.Hq + hk * g + r) * kHeadDim) + c4);
            const float2 a = __half22float2(u32_as_h2(u.x)), c2 = __half22float2(u32_as_h2(u.y));
            v = make_float4(a.x * p.q_scale, a.y * p.q_scale, c2.x * p.q_scale, c2.y * p.q_scale);
          }
          *reinterpret_cast<float4*>(&qw[r][4 * c4]) = v;
        }
        __syncwarp();
      }
    }
    if (LY::kQuant && k < p.ng) {
      if constexpr (LY::kQuant) {
        if (qb < j1) issue(qb, cur ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        process_group<KB, VB, NT>(p, qw, sm, st0 + cur * LY::kStageBytes, w, lane, qoff, O, macc, m_used, lsum);
        __syncwarp();
        cur ^= 1;
        qa = qb;
        qb = (qb < j1) ? next_q(qb + 1) : j1;
      }
    } else {
      const int c0 = 32 * (k - p.ng);
      const int k1 = p.S_eff + p.W;
      fp16_chunk<GT>(p, qw, pbuf, s, c0, k1, lane, m_t, l_t, acc_t, macc_t);
    }
  }
  cp_async_wait<0>();
  if (cur_s >= 0) finish(cur_s);
}

}  // namespace persist
}  // namespace kvq

namespace kvq {
namespace persist {

template <int KB, int VB, int GT>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t st) {
  constexpr int NT = GT <= 4 ? 1 : 2;
  using LY = PersistLayout<KB, VB, NT, GT>;
  const int smem = LY::kBytes;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_persist_kernel<KB, VB, NT, GT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  const int ctas = (p.nwarps + 3) / 4;
  decode_persist_kernel<KB, VB, NT, GT><<<ctas, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

// Resident CTAs per SM of an instantiation (for sizing the persistent grid).
template <int KB, int VB, int GT>
cudaError_t occupancy_t(int* ctas_per_sm) {
  constexpr int NT = GT <= 4 ? 1 : 2;
  using LY = PersistLayout<KB, VB, NT, GT>;
  const int smem = LY::kBytes;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_persist_kernel<KB, VB, NT, GT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_persist_kernel<KB, VB, NT, GT>,
                                                       kThreads, smem);
}

template <int KB, int VB>
cudaError_t dispatch_gt(const DecodeParams& p, cudaStream_t st, int* occ) {
  const int g = p.geo.g;
  if (occ) {
    if (g <= 1) return occupancy_t<KB, VB, 1>(occ);
    if (g <= 2) return occupancy_t<KB, VB, 2>(occ);
    if (g <= 4) return occupancy_t<KB, VB, 4>(occ);
    return occupancy_t<KB, VB, 8>(occ);
  }
  if (g <= 1) return launch_t<KB, VB, 1>(p, st);
  if (g <= 2) return launch_t<KB, VB, 2>(p, st);
  if (g <= 4) return launch_t<KB, VB, 4>(p, st);
  return launch_t<KB, VB, 8>(p, st);
}

template <int KB>
cudaError_t dispatch_vb(const DecodeParams& p, cudaStream_t st, int* occ) {
  switch (p.geo.vb) {
    case 2: return dispatch_gt<KB, 2>(p, st, occ);
    case 4: return dispatch_gt<KB, 4>(p, st, occ);
    case 8: return dispatch_gt<KB, 8>(p, st, occ);
  }
  return cudaErrorInvalidValue;
}

}  // namespace persist
}  // namespace kvq
