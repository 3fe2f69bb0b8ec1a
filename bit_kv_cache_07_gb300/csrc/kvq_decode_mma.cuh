// kvq_decode_mma.cuh -- tensor-core version of the quantized decode splits
// (uniform K per channel, uniform V per token over 64-channel groups;
// no RoPE).
//
// Why tensor cores: with the whole GQA group per CTA, the CUDA-core loop
// spends several instructions per code (extract, convert, one FMA per
// head) and issues ~4x more instructions than HBM speed allows.  Here the
// dequantized codes feed mma.sync.m16n8k16 (fp16 x fp16 -> fp32):
//   S = Kcodes (16 tokens x 16 channels) . Q'   (Q' = q * scale_k per channel)
//   O += Vcodes^T (16 channels x 16 tokens) . P' (P' = p * scale_v per token)
// Codes become exact fp16 integers with one lop3 (magic exponent 0x6400,
// 1024 + code) and one half-precision subtract per two codes.  The scaled
// operands Q' and P' are split into hi + lo fp16 parts (two mma columns per
// head), which keeps the products at ~2^-22 relative error; a single fp16
// operand would cost ~1e-3 of attention error.  The column layout is
// (head, hi/lo): one n8 tile holds 4 heads, two tiles hold 8.
//
// Tiles are staged per warp in shared memory with cp.async (16-byte
// asynchronous copies, double-buffered: the next 32-token group streams in
// while the current one is computed).  V codes are read back with
// ldmatrix.trans straight from their packed rows: a transposed 8x8 b16 tile
// hands each thread the codes of two consecutive tokens for the same
// channels, which is exactly the k-pair layout of an mma A fragment.
// V rows sit at a 16-byte padded pitch so those ldmatrix reads are free of
// bank conflicts.
//
// Online softmax in base 2 with a lazy rescale: the running maximum is only
// moved (and the accumulators rescaled) when a logit exceeds it by more
// than 2^8, which bounds p by 256 and keeps the fp32 accumulators safe.
#pragma once

#include "kvq_decode.cuh"

namespace kvq {
namespace mma {

constexpr float kLazyRescale = 8.0f;  // log2 units
constexpr int kGV = 64;                // V channel group of this kernel
constexpr int kNVG = kHeadDim / kGV;   // V groups per token

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                              uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

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

__device__ __forceinline__ uint32_t lop3_or_and(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));  // (a & mask) | magic
  return r;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Codes to exact fp16 pairs.  The magic exponent 0x6400 makes the fp16 value
// 1024 + x for an integer x < 1024 placed in the low mantissa bits.
//
// 4-bit: word w holds nibbles 0..7; pair i in 0..3 is (nibble i, nibble i+4).
__device__ __forceinline__ uint32_t ext4(uint32_t w, int i) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
  const __half2 km64 = __halves2half2(__ushort_as_half(0xD400), __ushort_as_half(0xD400));   // -64
  const uint32_t x = (i >= 2) ? (w >> 8) : w;
  if ((i & 1) == 0) return h2_as_u32(__hsub2(u32_as_h2(lop3_or_and(x, 0x000F000Fu, 0x64006400u)), k1024));
  return h2_as_u32(__hfma2(u32_as_h2(lop3_or_and(x, 0x00F000F0u, 0x64006400u)), k16th, km64));
}

// 8-bit: word w holds bytes 0..3; pair i in 0..1 is (byte i, byte i+2).
__device__ __forceinline__ uint32_t ext8(uint32_t w, int i) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const uint32_t sel = (i == 0) ? 0x4240u : 0x4341u;
  return h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, 0x64646464u, sel)), k1024));
}

// 2-bit: word w holds crumbs 0..15; pair i in 0..7 is (crumb i, crumb i+8).
__device__ __forceinline__ uint32_t ext2(uint32_t w, int i) {
  const uint32_t x = (i >= 4) ? (w >> 8) : w;
  const int m = i & 3;
  const uint32_t v = lop3_or_and(x, 0x00030003u << (2 * m), 0x64006400u);  // 1024 + 4^m c
  // (1024 + 4^m c) * 4^-m - 1024 * 4^-m = c, every step exact in fp16
  const uint16_t sc[4] = {0x3C00, 0x3400, 0x2C00, 0x2400};   // 1, 1/4, 1/16, 1/64
  const uint16_t of[4] = {0xE400, 0xDC00, 0xD400, 0xCC00};   // -1024, -256, -64, -16
  const __half2 s = __halves2half2(__ushort_as_half(sc[m]), __ushort_as_half(sc[m]));
  const __half2 o = __halves2half2(__ushort_as_half(of[m]), __ushort_as_half(of[m]));
  return h2_as_u32(__hfma2(u32_as_h2(v), s, o));
}

// ---------------------------------------------------------------- K side
// A fragment of k-step s for one token row, from this thread's 32-channel
// slice of the packed row (words w[]: KB=8: 8 words, KB=4: 4, KB=2: 2).
// Returns (lo, hi): lo holds k-slots (2t, 2t+1), hi holds (2t+8, 2t+9).
template <int KB>
__device__ __forceinline__ void k_frag(const uint32_t* w, int s, uint32_t& lo, uint32_t& hi) {
  if (KB == 8) {
    lo = ext8(w[s], 0);
    hi = ext8(w[s], 1);
  } else if (KB == 4) {
    const int pa = (s & 1) ? 2 : 0;
    lo = ext4(w[s >> 1], pa);
    hi = ext4(w[s >> 1], pa + 1);
  } else {
    const int ia = 2 * (s & 3);
    lo = ext2(w[s >> 2], ia);
    hi = ext2(w[s >> 2], ia + 1);
  }
}

// Where channel offset o (0..31) of a thread's slice lands: k-step s and
// element e (0,1: the lo register's halves; 2,3: the hi register's).
template <int KB>
__device__ __forceinline__ void k_slot_of(int o, int& s, int& e) {
  if (KB == 8) {
    const int n = o & 3;
    s = o >> 2;
    e = 2 * (n & 1) + (n >> 1);
  } else if (KB == 4) {
    const int wi = o >> 3, n = o & 7;
    s = 2 * wi + ((n & 3) >> 1);
    e = 2 * (n & 1) + (n >> 2);
  } else {
    const int wi = o >> 4, n = o & 15, i = n & 7;
    s = 4 * wi + (i >> 1);
    e = 2 * (i & 1) + (n >> 3);
  }
}

// ---------------------------------------------------------------- V side
// D-row channel of V m-tile mc for row half rh (0: row g, 1: row g+8).
template <int VB>
__device__ __forceinline__ int v_chan(int mc, int g, int rh) {
  if (VB == 8) return 16 * mc + 2 * g + rh;
  if (VB == 4) return 32 * (mc >> 1) + 4 * g + (mc & 1) + 2 * rh;
  return 64 * (mc >> 2) + 8 * g + (mc & 3) + 4 * rh;
}

template <int KB, int VB>
struct StageGeom {
  static constexpr int KROW = kHeadDim * KB / 8;
  static constexpr int VROW = kHeadDim * VB / 8;
  static constexpr int KPITCH = KROW + (KB == 8 ? 16 : 0);
  static constexpr int VPITCH = VROW + 16;
  static constexpr int KC = 0;
  static constexpr int KS = KC + kGroupTokens * KPITCH;
  static constexpr int VC = KS + kHeadDim * 4;
  static constexpr int VS = VC + kGroupTokens * VPITCH;
  static constexpr int BYTES = ((VS + kGroupTokens * 4 * 4) + 127) / 128 * 128;  // V scales: up to 4 groups
};

// Per-warp scratch of the group processing (4 warps per CTA).
template <int NT>
struct MmaWarpSmem {
  alignas(16) uint16_t bq[4][NT][32][40];        // each lane's 32 Q' halves per n-tile (+ pad)
  alignas(16) float bias[4][8 * NT];             // q . kmin of the current group, per head
  alignas(16) float vsc[4][kNVG][kGroupTokens];  // V scale of each token of the group (fp32)
  alignas(16) float vmn[4][kNVG][kGroupTokens];  // V min of each token of the group (fp32)
};

template <int KB, int VB>
__device__ __forceinline__ void issue_group(const DecodeParams& p, int s, int grp, unsigned char* dst, int lane) {
  using SG = StageGeom<KB, VB>;
  const Geometry& G = p.geo;
  const size_t row0 = (size_t)s * G.qcap + (size_t)grp * kGroupTokens;
  const uint8_t* kc = p.L.k_codes + row0 * SG::KROW;
  const uint8_t* vc = p.L.v_codes + row0 * SG::VROW;
  const uint32_t* ks = p.L.k_scales + ((size_t)s * G.gcap + grp) * kHeadDim;
  const uint32_t* vs = p.L.v_scales + row0 * kNVG;
  const uint32_t base = smem_u32(dst);
  constexpr int KCH = SG::KROW / 16, VCH = SG::VROW / 16;
  for (int i = lane; i < kGroupTokens * KCH; i += 32) {
    const int r = i / KCH, c = i % KCH;
    cp_async16(base + SG::KC + r * SG::KPITCH + 16 * c, kc + (size_t)r * SG::KROW + 16 * c);
  }
  cp_async16(base + SG::KS + 16 * lane, ks + 4 * lane);  // 512 B = 32 chunks
  for (int i = lane; i < kGroupTokens * VCH; i += 32) {
    const int r = i / VCH, c = i % VCH;
    cp_async16(base + SG::VC + r * SG::VPITCH + 16 * c, vc + (size_t)r * SG::VROW + 16 * c);
  }
  constexpr int vs_chunks = kGroupTokens * kNVG / 4;  // 16-byte chunks of V scales
  for (int i = lane; i < vs_chunks; i += 32) cp_async16(base + SG::VS + 16 * i, vs + 4 * i);
}

// V group (0 .. d/G_V - 1) of m-tile mc: every m-tile lies inside one group.
template <int VB>
__device__ __forceinline__ constexpr int v_group(int mc) {
  return (VB == 8 ? 16 * mc : VB == 4 ? 32 * (mc >> 1) : 64 * (mc >> 2)) / kGV;
}

// One 32-token group for one warp: Q' fragments, S = K Q' (2 m-tiles x NT
// n-tiles), online softmax, O += V^T P' (8 m-tiles x NT).
template <int KB, int VB, int NT>
__device__ __forceinline__ void process_group(const DecodeParams& p, const float (*qw)[kHeadDim],
                                              MmaWarpSmem<NT>& sm, const unsigned char* st,
                                              int w, int lane, const int (&qoff)[4], float (&O)[8][NT][4],
                                              float (&macc)[NT][kNVG], float (&m_used)[NT], float (&lsum)[NT]) {
  using SG = StageGeom<KB, VB>;
  const Geometry& G = p.geo;
  const int g = G.g;
  constexpr int nvg = kNVG;
  const int gq = lane >> 2, tq = lane & 3;

  // (a) Q' = q * scale_k (hi + lo fp16) into this warp's fragment buffer, bias = q . min_k;
  //     V {min, scale} of this lane's token to fp32
  {
    const uint4 sc = *reinterpret_cast<const uint4*>(st + SG::KS + 16 * lane);
    const uint32_t wv[4] = {sc.x, sc.y, sc.z, sc.w};
    float2 ms[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ms[k] = unpack_min_scale(wv[k]);
    const int tsl = lane >> 3;  // the reader thread-in-group owning these channels
#pragma unroll
    for (int r = 0; r < 8 * NT; ++r) {
      if (r >= g) break;
      const int nt = r >> 2, col = 2 * (r & 3);
      uint16_t* dhi = &sm.bq[w][nt][4 * col + tsl][0];
      uint16_t* dlo = &sm.bq[w][nt][4 * (col + 1) + tsl][0];
      const float4 q4 = *reinterpret_cast<const float4*>(&qw[r][4 * lane]);
      const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
      float bp = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float qp = qv[k] * ms[k].y;
        bp = fmaf(qv[k], ms[k].x, bp);
        const __half hi = __float2half_rn(qp);
        const __half lo = __float2half_rn(qp - __half2float(hi));
        dhi[qoff[k]] = __half_as_ushort(hi);
        dlo[qoff[k]] = __half_as_ushort(lo);
      }
      bp = warp_sum(bp);
      if (lane == 0) sm.bias[w][r] = bp;
    }
    const uint32_t* vsw = reinterpret_cast<const uint32_t*>(st + SG::VS);
#pragma unroll
    for (int j = 0; j < kNVG; ++j) {
      const float2 m2 = unpack_min_scale(vsw[lane * kNVG + j]);
      sm.vmn[w][j][lane] = m2.x;
      sm.vsc[w][j][lane] = m2.y;
    }
  }
  __syncwarp();

  // (b) this thread's Q' fragments
  uint32_t bq[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4* src = reinterpret_cast<const uint4*>(&sm.bq[w][nt][lane][0]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 u = src[k];
      bq[nt][4 * k] = u.x; bq[nt][4 * k + 1] = u.y; bq[nt][4 * k + 2] = u.z; bq[nt][4 * k + 3] = u.w;
    }
  }

  // (c) S = K Q'
  float S[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) S[mt][nt][k] = 0.0f;
    constexpr int NW = SG::KROW / 16;  // words in this thread's 32-channel slice
    uint32_t w0[NW], w1[NW];
    const unsigned char* r0 = st + SG::KC + (16 * mt + gq) * SG::KPITCH + 4 * NW * tq;
    const unsigned char* r1 = r0 + 8 * SG::KPITCH;
    if constexpr (NW == 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(r0), b2 = *reinterpret_cast<const uint4*>(r0 + 16);
      const uint4 c = *reinterpret_cast<const uint4*>(r1), d2 = *reinterpret_cast<const uint4*>(r1 + 16);
      w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w; w0[4] = b2.x; w0[5] = b2.y; w0[6] = b2.z; w0[7] = b2.w;
      w1[0] = c.x; w1[1] = c.y; w1[2] = c.z; w1[3] = c.w; w1[4] = d2.x; w1[5] = d2.y; w1[6] = d2.z; w1[7] = d2.w;
    } else if constexpr (NW == 4) {
      const uint4 a = *reinterpret_cast<const uint4*>(r0), c = *reinterpret_cast<const uint4*>(r1);
      w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
      w1[0] = c.x; w1[1] = c.y; w1[2] = c.z; w1[3] = c.w;
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(r0), c = *reinterpret_cast<const uint2*>(r1);
      w0[0] = a.x; w0[1] = a.y;
      w1[0] = c.x; w1[1] = c.y;
    }
    float S2[NT][4];  // odd k-steps accumulate separately: two independent mma chains
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) S2[nt][k] = 0.0f;
#pragma unroll
    for (int s_ = 0; s_ < 8; ++s_) {
      uint32_t lo0, hi0, lo1, hi1;
      k_frag<KB>(w0, s_, lo0, hi0);
      k_frag<KB>(w1, s_, lo1, hi1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (s_ & 1)
          mma16816(S2[nt], lo0, lo1, hi0, hi1, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
        else
          mma16816(S[mt][nt], lo0, lo1, hi0, hi1, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) S[mt][nt][k] += S2[nt][k];
  }

  // (d) online softmax (base 2); this thread's heads are 4*nt + tq
  float P[NT][2][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 4 * nt + tq;
    const float bias = (h < g) ? sm.bias[w][h] : 0.0f;
    float z[2][2];
    float zm = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        z[mt][rh] = (S[mt][nt][2 * rh] + S[mt][nt][2 * rh + 1]) + bias;
        zm = fmaxf(zm, z[mt][rh]);
      }
    zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 4));
    zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 8));
    zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 16));
    if (zm > m_used[nt] + kLazyRescale) {
      const float alpha = (m_used[nt] == -INFINITY) ? 0.0f : exp2f(m_used[nt] - zm);
#pragma unroll
      for (int mc = 0; mc < 8; ++mc)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[mc][nt][k] *= alpha;
#pragma unroll
      for (int j = 0; j < kNVG; ++j) macc[nt][j] *= alpha;
      lsum[nt] *= alpha;
      m_used[nt] = zm;
    }
    float ps = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const float pv = (h < g) ? exp2f(z[mt][rh] - m_used[nt]) : 0.0f;
        P[nt][mt][rh] = pv;
        ps += pv;
        const int tok = 16 * mt + 8 * rh + gq;
#pragma unroll
        for (int j = 0; j < nvg; ++j) macc[nt][j] = fmaf(pv, sm.vmn[w][j][tok], macc[nt][j]);
      }
    lsum[nt] += ps;
  }

  // (e) O += V^T P'
#pragma unroll
  for (int kt = 0; kt < 2; ++kt) {
    // P' fragments per (n-tile, V group): tokens 16kt + {2tq, 2tq+1, 2tq+8, 2tq+9}, column gq
    uint32_t bp[NT][kNVG][2];
    const int src1 = 8 * tq + (gq >> 1), src2 = src1 + 4;
    const int t0 = 16 * kt + 2 * tq;
    const bool lo_col = (gq & 1) != 0;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float v0 = __shfl_sync(0xffffffffu, P[nt][kt][0], src1);
      const float v1 = __shfl_sync(0xffffffffu, P[nt][kt][0], src2);
      const float v2 = __shfl_sync(0xffffffffu, P[nt][kt][1], src1);
      const float v3 = __shfl_sync(0xffffffffu, P[nt][kt][1], src2);
#pragma unroll
      for (int j = 0; j < nvg; ++j) {
        const float2 sa = *reinterpret_cast<const float2*>(&sm.vsc[w][j][t0]);
        const float2 sb = *reinterpret_cast<const float2*>(&sm.vsc[w][j][t0 + 8]);
        float x0 = v0 * sa.x;
        float x1 = v1 * sa.y;
        float x2 = v2 * sb.x;
        float x3 = v3 * sb.y;
        if (lo_col) {
          x0 -= __half2float(__float2half_rn(x0));
          x1 -= __half2float(__float2half_rn(x1));
          x2 -= __half2float(__float2half_rn(x2));
          x3 -= __half2float(__float2half_rn(x3));
        }
        bp[nt][j][0] = h2_as_u32(__floats2half2_rn(x0, x1));
        bp[nt][j][1] = h2_as_u32(__floats2half2_rn(x2, x3));
      }
    }
    // V code fragments via ldmatrix.trans on the packed rows
    const uint32_t vbase = smem_u32(st + SG::VC);
    const int mi = lane >> 3, rr = lane & 7;
    if (VB == 4) {
      uint32_t R[4][2];  // [block][token half]
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int blk = 2 * c + (mi >> 1), th = mi & 1;
        const uint32_t addr = vbase + (16 * kt + 8 * th + rr) * SG::VPITCH + 16 * blk;
        ldsm_x4_trans(R[2 * c][0], R[2 * c][1], R[2 * c + 1][0], R[2 * c + 1][1], addr);
      }
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const int blk = mc >> 1, i = mc & 1;
        const uint32_t a0 = ext4(R[blk][0], i), a1 = ext4(R[blk][0], i + 2);
        const uint32_t a2 = ext4(R[blk][1], i), a3 = ext4(R[blk][1], i + 2);
        const int j = v_group<VB>(mc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(O[mc][nt], a0, a1, a2, a3, bp[nt][j][0], bp[nt][j][1]);
      }
    } else if (VB == 8) {
      uint32_t R[8][2];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int blk = 2 * c + (mi >> 1), th = mi & 1;
        const uint32_t addr = vbase + (16 * kt + 8 * th + rr) * SG::VPITCH + 16 * blk;
        ldsm_x4_trans(R[2 * c][0], R[2 * c][1], R[2 * c + 1][0], R[2 * c + 1][1], addr);
      }
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const uint32_t a0 = ext8(R[mc][0], 0), a1 = ext8(R[mc][0], 1);
        const uint32_t a2 = ext8(R[mc][1], 0), a3 = ext8(R[mc][1], 1);
        const int j = v_group<VB>(mc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(O[mc][nt], a0, a1, a2, a3, bp[nt][j][0], bp[nt][j][1]);
      }
    } else {
      uint32_t R[2][2];
      {
        const int blk = mi >> 1, th = mi & 1;
        const uint32_t addr = vbase + (16 * kt + 8 * th + rr) * SG::VPITCH + 16 * blk;
        ldsm_x4_trans(R[0][0], R[0][1], R[1][0], R[1][1], addr);
      }
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const int blk = mc >> 2, i = mc & 3;
        const uint32_t a0 = ext2(R[blk][0], i), a1 = ext2(R[blk][0], i + 4);
        const uint32_t a2 = ext2(R[blk][1], i), a3 = ext2(R[blk][1], i + 4);
        const int j = v_group<VB>(mc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(O[mc][nt], a0, a1, a2, a3, bp[nt][j][0], bp[nt][j][1]);
      }
    }
  }
}

}  // namespace mma
}  // namespace kvq
