// kvq_append.cu -- cache write path: fp16 window/sink copies and the
// quantize-and-pack kernel that flushes G_K-token groups.
//
// Method (page title, section):
//  * "KVTuner" review, observation 2: K quantized per channel, asymmetric
//    (min/scale), here over groups of G_K = 32 tokens.
//  * InnerQ, Methodology 1-2: V grouped along the hidden dimension (G_V
//    channels) per token, one min and one shared scale per group;
//    Methodology 4: the most recent and the sink tokens stay fp16.
//  * KVQuant, technical approach: non-uniform per-layer levels and
//    per-vector dense-and-sparse outliers (~1 %), pre-RoPE K (K is written
//    as given; RoPE happens in the decode).
//  * Hadamard write-up, "section details": V rotated by a Hadamard matrix
//    before the uniform quantizer.
//
// The fp32 quantizer is evaluated with explicitly rounded intrinsics
// (__fsub_rn, __fdiv_rn, rintf) so that no operation is contracted or
// approximated: codes and scales are bit-reproducible.
#include <cstring>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kRowHalves = kHeadDim;          // 128 fp16 per token row
constexpr int kRowVec = kRowHalves * 2 / 16;  // 16 x 16-byte chunks per row

// Uniform asymmetric quantizer of one value given its group's min and the
// fp32 scale: clamp(rint((x - min) / scale), 0, 2^b - 1); scale 0 -> 0.
// code = clamp(rint(RN((x - mn) / scale)), 0, qmax) without a division per
// element: rs = RN(1 / scale) is shared by the group, and qa = RN(d * rs)
// differs from the quotient by at most 2^-23 relative (< 3.1e-5 for
// quotients below 256) while RN(d / scale) is within half an ulp (< 7.7e-6)
// of it, so both round to the same integer unless qa lies within 1e-4 of a
// half-integer; there the IEEE division decides.
// (0 <= x - mn <= max - mn, so the quotient lies in [0, qmax (1 + 2^-23)]
// and its rounding in [0, qmax]: the clamp of the definition never binds;
// qa - rint(qa) is exact, and its magnitude exceeds 0.4999 exactly when qa
// lies within 1e-4 of a half-integer.)
// rint(d / scale) by the IEEE division, out of line: the rare path of the
// codes below, kept out of their unrolled loops.
__device__ __noinline__ float rint_div(float d, float scale) { return rintf(__fdiv_rn(d, scale)); }
// d / s by the IEEE division, out of line (the non-uniform codes' rare path).
__device__ __noinline__ float div_rn(float d, float s) { return __fdiv_rn(d, s); }

__device__ __forceinline__ uint32_t uniform_code(float x, float mn, float scale, float rs) {
  if (scale == 0.0f) return 0u;
  const float d = __fsub_rn(x, mn);
  const float qa = __fmul_rn(d, rs);
  float r = rintf(qa);
  if (fabsf(__fsub_rn(qa, r)) > 0.4999f) r = rint_div(d, scale);
  return (uint32_t)r;
}

// Parameters of one uniform group from its min, max and exact sum
// (InnerQ, Methodology 2: the group picks a symmetric or an asymmetric grid
// from its own statistics).  Symmetric when `hybrid`, mx > mn and the mean
// lies within half an asymmetric step of zero, |mean| 2^(b+1) <= mx - mn:
// scale = max(|mn|, |mx|) / (2^(b-1) - 1), stored min = -2^(b-1) fp16(scale)
// (falls back to asymmetric if that overflows fp16).  Asymmetric otherwise:
// scale = (mx - mn) / (2^b - 1), stored min = fp16(mn).
// The inputs are fp16 values (units of 2^-24, |x| < 2^16), or fp16 values
// divided by the key normalisation (|x| <= 1, units of 2^-40), so every one
// is an integer in units 2^-sh (sh = 24 or 40) and the sum is computed
// exactly in 64-bit integers (fixed()), in any order; the comparison
// |S| 2^(b+1) <= n (MX - MN), all in those units, is then exact too (the
// same real-number test the oracle makes with its exact fp64 mean).  At most
// 128 values: |S| <= 2^47 and the products stay below 2^57.
// x 2^sh as an integer, from the bits of x (no 64-bit conversion
// instruction): |m| 2^(e - 150 + sh) with m the 24-bit significand and e
// the biased exponent (1 for subnormals); a negative shift only drops zero
// bits, because x 2^sh is an integer.
__device__ __forceinline__ long long fixed(float x, int sh) {
  const uint32_t b = __float_as_uint(x);
  const int e = (int)((b >> 23) & 0xFFu);
  const long long m = (long long)((b & 0x7FFFFFu) | (e ? 0x800000u : 0u));
  const int shift = (e ? e : 1) - 150 + sh;
  const long long a = shift >= 0 ? (m << shift) : (m >> -shift);
  return (b >> 31) ? -a : a;
}
struct GroupQ {
  float mn, scale, rs;  // asymmetric origin, fp32 scale and its reciprocal
  int sym;              // 1: symmetric codes
  uint32_t word;        // stored {min, scale} fp16 pair
};
__device__ __forceinline__ GroupQ group_params(float mn, float mx, long long sum, int sh, int n, int bits,
                                               int hybrid) {
  GroupQ g;
  g.sym = 0;
  long long S = sum < 0 ? -sum : sum;
  if (hybrid && mx > mn && (S << (bits + 1)) <= (long long)n * (fixed(mx, sh) - fixed(mn, sh))) {
    const float a = fmaxf(fabsf(mn), fabsf(mx));
    const float scale = __fdiv_rn(a, (float)((1 << (bits - 1)) - 1));
    const uint16_t sh = float_to_half_bits(scale);
    const uint16_t mh = float_to_half_bits(__fmul_rn(-(float)(1 << (bits - 1)), half_bits_to_float(sh)));
    if (!isinf(half_bits_to_float(mh))) {
      g.sym = 1;
      g.mn = 0.0f;
      g.scale = scale;
      g.rs = __frcp_rn(scale);
      g.word = (uint32_t)mh | ((uint32_t)sh << 16);
      return g;
    }
  }
  g.mn = mn;
  g.scale = __fdiv_rn(__fsub_rn(mx, mn), (float)((1 << bits) - 1));
  g.rs = g.scale == 0.0f ? 0.0f : __frcp_rn(g.scale);
  g.word = (uint32_t)float_to_half_bits(mn) | ((uint32_t)float_to_half_bits(g.scale) << 16);
  return g;
}

// Symmetric code clamp(rint(x / scale), -qs, qs) + 2^(b-1), qs = 2^(b-1) - 1
// (|x| <= qs scale up to rounding: the quotient's magnitude stays below 256,
// so the reciprocal shortcut of uniform_code applies unchanged).
__device__ __forceinline__ uint32_t sym_code(float x, float scale, float rs, int bits) {
  const float qa = __fmul_rn(x, rs);
  float r = rintf(qa);
  if (fabsf(__fsub_rn(qa, r)) > 0.4999f) r = rint_div(x, scale);
  const float qs = (float)((1 << (bits - 1)) - 1);
  r = fminf(fmaxf(r, -qs), qs);
  return (uint32_t)((int)r + (1 << (bits - 1)));
}

__device__ __forceinline__ uint32_t group_code(float x, const GroupQ& g, int bits) {
  return g.sym ? sym_code(x, g.scale, g.rs, bits) : uniform_code(x, g.mn, g.scale, g.rs);
}

// Level midpoints tau_i = (L_i + L_(i+1)) / 2 - L_0 of a LUT, in fp32 as the
// encoder compares them (computed once per CTA).
__device__ __forceinline__ void nuq_midpoints(const float* lut, float (&tau)[7]) {
#pragma unroll
  for (int i = 0; i < 7; ++i) tau[i] = __fsub_rn(__fmul_rn(__fadd_rn(lut[i], lut[i + 1]), 0.5f), lut[0]);
}

// Minimum and maximum of the dense (non-outlier) values of a warp's vector.
__device__ __forceinline__ void dense_min_max(const float (&v)[4], const bool (&is_out)[4], float& mn, float& mx) {
  mn = INFINITY;
  mx = -INFINITY;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (!is_out[q]) { mn = fminf(mn, v[q]); mx = fmaxf(mx, v[q]); }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
}

// The k largest |v| of a token vector held by a warp (lane l: channels
// 4l..4l+3), ties to the lower channel: is_out marks this lane's outliers,
// sel[j] is the channel of the j-th largest (past k: a value that sorts
// last).  The dense min and max of the rest come back in mn, mx.
__device__ __forceinline__ void nuq_outliers(const float (&v)[4], int k, int lane, bool (&is_out)[4],
                                             int (&sel)[kMaxOutliers], float& mn, float& mx) {
#pragma unroll
  for (int q = 0; q < 4; ++q) is_out[q] = false;
#pragma unroll
  for (int j = 0; j < kMaxOutliers; ++j) {
    sel[j] = 1 << 30;  // past k: sorts last, never written
    if (j >= k) continue;
    float bv = -1.0f;
    int bi = 1 << 30;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (!is_out[q]) {
        float a = fabsf(v[q]);
        if (a > bv) { bv = a; bi = 4 * lane + q; }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    sel[j] = bi;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (bi == 4 * lane + q) is_out[q] = true;
  }
  dense_min_max(v, is_out, mn, mx);
}

// The same selection for fp16 values h (v their fp32 widenings), one
// warp-wide integer maximum per outlier: the key (|h| << 16) | (0xFFFF - c)
// orders by magnitude (fp16 magnitude bits order like the magnitudes, for
// finite values) and then by the lower channel c, so its maximum is the
// largest |x| with ties to the lower channel.
__device__ __forceinline__ void nuq_outliers_h(const float (&v)[4], const uint16_t (&h)[4], int k, int lane,
                                               bool (&is_out)[4], int (&sel)[kMaxOutliers], float& mn,
                                               float& mx) {
  uint32_t key[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    is_out[q] = false;
    key[q] = ((uint32_t)(h[q] & 0x7FFFu) << 16) | (0xFFFFu - (uint32_t)(4 * lane + q));
  }
#pragma unroll
  for (int j = 0; j < kMaxOutliers; ++j) {
    sel[j] = 1 << 30;  // past k: sorts last, never written
    if (j >= k) continue;
    uint32_t b = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (!is_out[q]) b = max(b, key[q]);
    b = __reduce_max_sync(0xffffffffu, b);
    const int bi = (int)(0xFFFFu - (b & 0xFFFFu));
    sel[j] = bi;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (bi == 4 * lane + q) is_out[q] = true;
  }
  dense_min_max(v, is_out, mn, mx);
}

// Non-uniform (LUT) encoding of one 128-channel token vector held by a warp
// (lane l owns channels 4l..4l+3).  The k largest |x| (ties to the lower
// channel) become fp16 outliers with code 0; the dense rest is mapped
// affinely onto [L0, L7] and coded by counting the level midpoints below
// u = RN((x - mn) / s).  u comes from RN(d * RN(1 / s)), which is within
// 3 * 2^-24 relative of it; only when that product lies within 2^-21
// relative of a midpoint does the IEEE division decide.
__device__ void nuq_encode_row(const uint16_t* __restrict__ xrow, const float* lut, const float (&tau)[7], int k,
                               uint8_t* __restrict__ code_row, uint32_t* minsc_out,
                               uint8_t* col_out, uint16_t* val_out, int lane) {
  float v[4];
  uint16_t hb[4];
  bool is_out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    hb[q] = xrow[4 * lane + q];
    v[q] = half_bits_to_float(hb[q]);
  }
  int sel[kMaxOutliers];
  float mn, mx;
  nuq_outliers_h(v, hb, k, lane, is_out, sel, mn, mx);
  const float s = __fdiv_rn(__fsub_rn(mx, mn), __fsub_rn(lut[7], lut[0]));
  const float rs = s != 0.0f ? __frcp_rn(s) : 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t c = 0;
    if (!is_out[q] && s != 0.0f) {
      const float d = __fsub_rn(v[q], mn);
      float u = __fmul_rn(d, rs);
      const float band = u * 0x1p-21f;
      bool near = false;
#pragma unroll
      for (int i = 0; i < 7; ++i) near |= fabsf(__fsub_rn(u, tau[i])) <= band;
      if (near) u = div_rn(d, s);
#pragma unroll
      for (int i = 0; i < 7; ++i) c += (u > tau[i]) ? 1u : 0u;
    }
    code_row[4 * lane + q] = (uint8_t)c;
  }
  if (lane == 0) {
    // ascending column order for the CSR row: an odd-even transposition
    // sort, k passes over the first k slots
#pragma unroll
    for (int pass = 0; pass < kMaxOutliers; ++pass) {
      if (pass >= k) break;
#pragma unroll
      for (int a = pass & 1; a + 1 < kMaxOutliers; a += 2)
        if (a + 1 < k && sel[a] > sel[a + 1]) {
          const int t = sel[a];
          sel[a] = sel[a + 1];
          sel[a + 1] = t;
        }
    }
#pragma unroll
    for (int j = 0; j < kMaxOutliers; ++j) {
      if (j >= k) break;
      col_out[j] = (uint8_t)sel[j];
      val_out[j] = xrow[sel[j]];
    }
    *minsc_out = (uint32_t)float_to_half_bits(mn) | ((uint32_t)float_to_half_bits(s) << 16);
  }
}

// In-warp normalised Hadamard rotation of one token vector (lane l owns
// channels 4l..4l+3): fp32 butterflies of width 1, 2, 4, ..., 64, each
// (a, b) -> (a + b, a - b), then times fp32(1/sqrt(d)) and round to fp16.
__device__ __forceinline__ void hadamard_vals(float (&v)[4], float c, int lane) {
  float a0 = __fadd_rn(v[0], v[1]), a1 = __fsub_rn(v[0], v[1]);
  float a2 = __fadd_rn(v[2], v[3]), a3 = __fsub_rn(v[2], v[3]);
  v[0] = __fadd_rn(a0, a2); v[2] = __fsub_rn(a0, a2);
  v[1] = __fadd_rn(a1, a3); v[3] = __fsub_rn(a1, a3);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float o = __shfl_xor_sync(0xffffffffu, v[q], m);
      v[q] = upper ? __fsub_rn(o, v[q]) : __fadd_rn(v[q], o);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = half_bits_to_float(float_to_half_bits(__fmul_rn(v[q], c)));
}

__device__ void hadamard_row_inplace(uint16_t* row, float c, int lane) {
  float v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = half_bits_to_float(row[4 * lane + q]);
  hadamard_vals(v, c, lane);
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) row[4 * lane + q] = float_to_half_bits(v[q]);
  __syncwarp();
}

// Pack rows of 8-bit codes (one byte per channel in shared memory) into the
// little-endian bitstream layout and store them as 32-bit words.  Uniform
// widths gather a word's codes with one shared load and merge the fields
// with shifts and byte permutes; 3-bit words take 12 codes (36 bits cover
// the word's 32 plus its 0-2 bit offset) into a 64-bit accumulator.
__device__ __forceinline__ uint32_t pack4x8(uint32_t x) {  // 4 byte codes < 16 -> 16 bits
  const uint32_t t = x | (x >> 4);                           // byte 0: c0 | c1 << 4, byte 2: c2 | c3 << 4
  return __byte_perm(t, 0u, 0x4420) & 0xFFFFu;
}
__device__ __forceinline__ uint32_t pack2x4(uint32_t x) {  // 4 byte codes < 4 -> 8 bits
  uint32_t t = x | (x >> 6);  // bits 0-3: c0 | c1 << 2; bits 16-19: c2 | c3 << 2
  t |= t >> 12;               // bits 4-7: c2 | c3 << 2
  return t & 0xFFu;
}
template <int bits>
__device__ __forceinline__ void pack_rows(const uint8_t (*codes)[kHeadDim], int rows, uint8_t* dst, int row_bytes,
                                          int tid) {
  const int words = row_bytes / 4;  // 8, 16, 32 (2/4/8 bits) or 12 (3 bits)
  const int lw = __ffs(words) - 1;   // log2 of a power-of-two word count
  for (int idx = tid; idx < rows * words; idx += kThreads) {
    const int r = bits == 3 ? idx / 12 : idx >> lw;
    const int wi = idx - r * words;
    uint32_t word = 0;
    if constexpr (bits == 8) {
      word = *reinterpret_cast<const uint32_t*>(&codes[r][4 * wi]);
    } else if constexpr (bits == 4) {
      const uint2 x = *reinterpret_cast<const uint2*>(&codes[r][8 * wi]);
      word = pack4x8(x.x) | (pack4x8(x.y) << 16);
    } else if constexpr (bits == 2) {
      const uint4 x = *reinterpret_cast<const uint4*>(&codes[r][16 * wi]);
      word = pack2x4(x.x) | (pack2x4(x.y) << 8) | (pack2x4(x.z) << 16) | (pack2x4(x.w) << 24);
    } else if constexpr (bits == 3) {
      const int c0 = (32 * wi) / 3, off = 32 * wi - 3 * c0;
      unsigned long long acc = 0;
#pragma unroll
      for (int m = 0; m < 12; ++m)
        if (c0 + m < kHeadDim) acc |= (unsigned long long)(codes[r][c0 + m] & 7u) << (3 * m);
      word = (uint32_t)(acc >> off);
    } else {
      for (int p = 0; p < 32; ++p) {
        const int gb = wi * 32 + p;
        word |= (uint32_t)((codes[r][gb / bits] >> (gb % bits)) & 1) << p;
      }
    }
    reinterpret_cast<uint32_t*>(dst + (size_t)r * row_bytes)[wi] = word;
  }
}

// One CTA quantizes one G_K-token group of one stream (K and V).  One
// instantiation per key mode and bit widths -- KM = 0: uniform K per channel,
// 1: uniform InnerQ K (per token, 64-channel groups), 2: non-uniform codes
// (KB = VB = 3) -- so that each holds only its own path.
template <int KM, int KB, int VB>
__global__ void __launch_bounds__(kThreads) append_quantize_kernel(const __grid_constant__ AppendParams p) {
  const Geometry& G = p.geo;
  const int s = blockIdx.y;
  const RowAppend ra = row_append(p, s);
  if ((int)blockIdx.x >= (ra.nq_after - ra.nq_before) / kGroupTokens) return;  // (ragged) no such group here
  const int grp = ra.first_group + blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  __shared__ __align__(16) uint16_t sK[kGroupTokens][kRowHalves];
  __shared__ __align__(16) uint16_t sV[kGroupTokens][kRowHalves];
  __shared__ __align__(16) uint8_t sCk[kGroupTokens][kHeadDim];
  __shared__ __align__(16) uint8_t sCv[kGroupTokens][kHeadDim];

  // fp16 sources: tokens written before this call come from the window ring,
  // the others straight from this call's input.  All of a thread's loads are
  // issued before the first shared store.
  {
    constexpr int kPer = kGroupTokens * kRowVec / kThreads;
    static_assert(kPer * kThreads == kGroupTokens * kRowVec, "whole chunks per thread");
    uint4 kx[kPer], vx[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = tid + u * kThreads;
      const int r = idx / kRowVec, ch = idx % kRowVec;
      const int t = G.S + grp * kGroupTokens + r;
      const uint16_t *srck, *srcv;
      if (t >= ra.before) {
        const size_t off = (in_stream(G, s) * p.n_new + (t - ra.before)) * kRowHalves;
        srck = p.k_new + off;
        srcv = p.v_new + off;
      } else {
        const size_t off = ((size_t)s * G.ring + (t - G.S) % G.ring) * kRowHalves;
        srck = p.L.k_ring + off;
        srcv = p.L.v_ring + off;
      }
      kx[u] = reinterpret_cast<const uint4*>(srck)[ch];
      vx[u] = reinterpret_cast<const uint4*>(srcv)[ch];
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = tid + u * kThreads;
      const int r = idx / kRowVec, ch = idx % kRowVec;
      reinterpret_cast<uint4*>(&sK[r][0])[ch] = kx[u];
      reinterpret_cast<uint4*>(&sV[r][0])[ch] = vx[u];
    }
  }
  __syncthreads();

  const int i0 = grp * kGroupTokens;  // quantized index of the group's first token
  const int kmax = G.nout;
  float tau_k[7], tau_v[7];  // NUQ level midpoints
  nuq_midpoints(p.k_lut, tau_k);
  nuq_midpoints(p.v_lut, tau_v);

  // ---- K
  if constexpr (KM == 2) {
    for (int r = w; r < kGroupTokens; r += 4) {
      const int i = i0 + r;
      const size_t csr = (size_t)s * G.qcap * kmax + (size_t)i * kmax;
      nuq_encode_row(sK[r], p.k_lut, tau_k, kmax, sCk[r], &p.L.k_scales[(size_t)s * G.qcap + i],
                     p.L.k_col + csr, p.L.k_val + csr, lane);
      if (lane == 0) {
        int32_t* rp = p.L.k_rowptr + (size_t)s * (G.qcap + 1);
        rp[i + 1] = (i + 1) * kmax;
        if (i == 0) rp[0] = 0;
      }
    }
  } else if constexpr (KM == 1) {
    // InnerQ: per token, groups of 64 channels along the hidden dimension
    // (16 lanes per group), on the keys divided by the channel normalisation
    // the normalisation is a power of two 2^e (|e| <= 24): dividing by it is
    // exactly multiplying by 2^-e, and neither result can be subnormal
    float inv[4] = {1.0f, 1.0f, 1.0f, 1.0f};
    if (G.knorm) {
      const float4 n4 = *reinterpret_cast<const float4*>(&p.L.k_norm[(size_t)s * kHeadDim + 4 * lane]);
      inv[0] = __frcp_rn(n4.x);
      inv[1] = __frcp_rn(n4.y);
      inv[2] = __frcp_rn(n4.z);
      inv[3] = __frcp_rn(n4.w);
    }
    for (int r = w; r < kGroupTokens; r += 4) {
      const int i = i0 + r;
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[q] = half_bits_to_float(sK[r][4 * lane + q]);
        if (G.knorm) v[q] = __fmul_rn(v[q], inv[q]);
      }
      float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
      float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      const int sh = G.knorm ? 40 : 24;
      long long sum = 0;
      if (G.hybrid) sum = (fixed(v[0], sh) + fixed(v[1], sh)) + (fixed(v[2], sh) + fixed(v[3], sh));
      for (int o = 8; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (G.hybrid) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      }
      const GroupQ gq = group_params(mn, mx, sum, sh, 64, KB, G.hybrid);
#pragma unroll
      for (int q = 0; q < 4; ++q) sCk[r][4 * lane + q] = (uint8_t)group_code(v[q], gq, KB);
      if ((lane & 15) == 0) p.L.k_scales[((size_t)s * G.qcap + i) * G.nkg + (lane >> 4)] = gq.word;
    }
  } else {
    const int c = tid;  // one channel per thread, over the group's tokens (held in registers)
    float xk[kGroupTokens];
#pragma unroll
    for (int r = 0; r < kGroupTokens; ++r) xk[r] = half_bits_to_float(sK[r][c]);
    float mn = xk[0], mx = xk[0];
#pragma unroll
    for (int r = 1; r < kGroupTokens; ++r) {
      mn = fminf(mn, xk[r]);
      mx = fmaxf(mx, xk[r]);
    }
    long long sum = 0;
    if (G.hybrid)
      for (int r = 0; r < kGroupTokens; ++r) sum += fixed(xk[r], 24);
    const GroupQ gq = group_params(mn, mx, sum, 24, kGroupTokens, KB, G.hybrid);
#pragma unroll
    for (int r = 0; r < kGroupTokens; ++r) sCk[r][c] = (uint8_t)group_code(xk[r], gq, KB);
    p.L.k_scales[((size_t)s * G.gcap + grp) * kHeadDim + c] = gq.word;
  }

  // ---- V (optionally rotated first)
  for (int r = w; r < kGroupTokens; r += 4) {
    const int i = i0 + r;
    if (G.hadamard) hadamard_row_inplace(sV[r], p.hadamard_c, lane);
    if constexpr (VB == 3) {
      const size_t csr = (size_t)s * G.qcap * kmax + (size_t)i * kmax;
      nuq_encode_row(sV[r], p.v_lut, tau_v, kmax, sCv[r], &p.L.v_scales[(size_t)s * G.qcap + i],
                     p.L.v_col + csr, p.L.v_val + csr, lane);
      if (lane == 0) {
        int32_t* rp = p.L.v_rowptr + (size_t)s * (G.qcap + 1);
        rp[i + 1] = (i + 1) * kmax;
        if (i == 0) rp[0] = 0;
      }
    } else {
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = half_bits_to_float(sV[r][4 * lane + q]);
      float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
      float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      long long sum = 0;
      if (G.hybrid) sum = (fixed(v[0], 24) + fixed(v[1], 24)) + (fixed(v[2], 24) + fixed(v[3], 24));
      const int seg = G.gv / 4;  // lanes per channel group
      for (int o = seg / 2; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (G.hybrid) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      }
      const GroupQ gq = group_params(mn, mx, sum, 24, G.gv, VB, G.hybrid);
#pragma unroll
      for (int q = 0; q < 4; ++q) sCv[r][4 * lane + q] = (uint8_t)group_code(v[q], gq, VB);
      if (lane % seg == 0) p.L.v_scales[((size_t)s * G.qcap + i) * G.nvg + lane / seg] = gq.word;
    }
  }
  __syncthreads();

  pack_rows<KB>(sCk, kGroupTokens, p.L.k_codes + ((size_t)s * G.qcap + i0) * G.krow, G.krow, tid);
  pack_rows<VB>(sCv, kGroupTokens, p.L.v_codes + ((size_t)s * G.qcap + i0) * G.vrow, G.vrow, tid);
}

// InnerQ per-channel key normalisation of an empty cache's first append:
// n_c = the smallest power of two >= max |K_c| over the call's tokens (1 for
// an all-zero channel), per stream.  Two passes: CTAs over (token block,
// stream) fold the block's max |K_c| into the stream's slot with an integer
// atomic max (non-negative floats order like their bit patterns: the max is
// exact in any order), then one thread per (stream, channel) turns the max
// into the power of two, in place.  The slots start at zero.  Only streams
// whose row appends into an empty cache take part (every stream but for a
// ragged append).
__device__ __forceinline__ __half2 u32_as_half2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// In the max pass thread t reads 16-byte pieces (channels 8 (t mod 16) ..
// + 7) of every 8th row from row t / 16 on, keeps the maxima of |x| as fp16
// pairs (exact), and the 8 row slots of a channel meet in shared memory.
constexpr int kNormTokens = 256;  // tokens per CTA of the max pass
__global__ void __launch_bounds__(kHeadDim) key_norm_zero_kernel(const __grid_constant__ AppendParams p) {
  if (row_append(p, blockIdx.x).before == 0) p.L.k_norm[(size_t)blockIdx.x * kHeadDim + threadIdx.x] = 0.0f;
}
__global__ void __launch_bounds__(kHeadDim) key_norm_max_kernel(const __grid_constant__ AppendParams p) {
  __shared__ float part[8][kHeadDim];
  const int s = blockIdx.y, tid = threadIdx.x, piece = tid & 15, row = tid >> 4;
  const RowAppend ra = row_append(p, s);
  if (ra.before != 0) return;
  const int t0 = blockIdx.x * kNormTokens, t1 = min(ra.n, t0 + kNormTokens);
  const uint4* k = reinterpret_cast<const uint4*>(p.k_new + in_stream(p.geo, s) * p.n_new * kRowHalves) + piece;
  __half2 m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __float2half2_rn(0.0f);
#pragma unroll 4
  for (int t = t0 + row; t < t1; t += 8) {
    const uint4 x = k[(size_t)t * (kRowHalves / 8)];
    m[0] = __hmax2(m[0], __habs2(u32_as_half2(x.x)));
    m[1] = __hmax2(m[1], __habs2(u32_as_half2(x.y)));
    m[2] = __hmax2(m[2], __habs2(u32_as_half2(x.z)));
    m[3] = __hmax2(m[3], __habs2(u32_as_half2(x.w)));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(m[i]);
    part[row][8 * piece + 2 * i] = f.x;
    part[row][8 * piece + 2 * i + 1] = f.y;
  }
  __syncthreads();
  float mc = part[0][tid];
#pragma unroll
  for (int r = 1; r < 8; ++r) mc = fmaxf(mc, part[r][tid]);
  atomicMax(reinterpret_cast<unsigned int*>(&p.L.k_norm[(size_t)s * kHeadDim + tid]), __float_as_uint(mc));
}
__global__ void __launch_bounds__(kHeadDim) key_norm_pow2_kernel(const __grid_constant__ AppendParams p) {
  if (row_append(p, blockIdx.x).before != 0) return;
  float* slot = &p.L.k_norm[(size_t)blockIdx.x * kHeadDim + threadIdx.x];
  const float m = *slot;
  float n = 1.0f;
  if (m > 0.0f) {
    int e;
    frexpf(m, &e);  // m = f 2^e, f in [0.5, 1): 2^(e-1) <= m < 2^e
    n = ldexpf(1.0f, e);
    if (ldexpf(1.0f, e - 1) >= m) n = ldexpf(1.0f, e - 1);  // m itself a power of two
  }
  *slot = n;
}

// Copy the fp16 tokens of this call that stay fp16 (sinks and the final
// window) into their slots.  One thread per 16-byte chunk of a K or V row,
// over those tokens only: the call's tokens j < a (sinks; every token of an
// fp16 cache) and j >= b (past the quantized part).
__global__ void __launch_bounds__(256) append_window_kernel(const __grid_constant__ AppendParams p, int ncopy) {
  const Geometry& G = p.geo;
  grid_dep_wait();     // earlier kernels may still read the ring slots written here
  grid_dep_trigger();  // the decode that follows may set up meanwhile
  const size_t total = (size_t)G.NS * ncopy * (2 * kRowVec);
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int ch = (int)(idx % kRowVec);
    const int isv = (int)((idx / kRowVec) % 2);
    const size_t rest = idx / (2 * kRowVec);
    const int jc = (int)(rest % ncopy);
    const int s = (int)(rest / ncopy);
    const RowAppend ra = row_append(p, s);
    int a, b;
    window_split(p, ra, &a, &b);
    if (jc >= a + (ra.n - b)) continue;  // (ragged) this row copies fewer
    const int j = jc < a ? jc : b + (jc - a);
    const int pos = ra.before + j;
    uint16_t* dst;
    if (G.fp16_mode) {
      dst = (isv ? p.L.v_ring : p.L.k_ring) + ((size_t)s * G.ring + pos) * kRowHalves;
    } else if (pos < G.S) {
      dst = (isv ? p.L.v_sink : p.L.k_sink) + ((size_t)s * G.S + pos) * kRowHalves;
    } else {
      dst = (isv ? p.L.v_ring : p.L.k_ring) + ((size_t)s * G.ring + (pos - G.S) % G.ring) * kRowHalves;
    }
    const uint16_t* src = (isv ? p.v_new : p.k_new) + (in_stream(G, s) * p.n_new + j) * kRowHalves;
    reinterpret_cast<uint4*>(dst)[ch] = reinterpret_cast<const uint4*>(src)[ch];
  }
}

// ------------------------------------------------ level-table fitting
// Unweighted per-layer Lloyd fit of the 8 non-uniform levels (KVQuant:
// per-layer datatypes computed offline; the sensitivity weights need a
// model's gradients and are left out).  Every dense value of a calibration
// vector is placed in its vector's dense range exactly as the encoder maps
// it -- outliers removed by the same selection, u = RN((x - mn) / (mx - mn))
// -- on a grid of 2^-16: p = rint(u 2^16), an integer in [0, 2^16].  The
// first kernel counts the positions (a histogram of 2^16 + 1 bins); the
// second takes prefix sums of the counts and of position x count and runs
// Lloyd's iterations on them with the end levels held at 0 and 2^16 (every
// vector's min and max sit there).  All sums are exact integers and every
// level an fp64 quotient of two of them, so the fit does not depend on the
// order in which values are counted.
constexpr int kFitGrid = 1 << 16;
constexpr int kFitWarps = 8;

__global__ void __launch_bounds__(32 * kFitWarps)
    nuq_fit_hist_kernel(const uint16_t* __restrict__ x, long long nvec, int k, int hadamard, float hc,
                        unsigned long long* __restrict__ hist) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kFitWarps;
  unsigned long long n_lo = 0, n_hi = 0;  // positions 0 and 2^16 (each vector's min and max): once per warp
  for (long long v = (long long)blockIdx.x * kFitWarps + (threadIdx.x >> 5); v < nvec; v += warps) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(x + (size_t)v * kHeadDim) + lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    float val[4] = {a.x, a.y, b.x, b.y};
    if (hadamard) hadamard_vals(val, hc, lane);
    bool is_out[4];
    int sel[kMaxOutliers];
    float mn, mx;
    nuq_outliers(val, k, lane, is_out, sel, mn, mx);
    if (!(mx > mn)) continue;  // a constant dense part: no positions (warp-uniform)
    const float span = __fsub_rn(mx, mn);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (is_out[q]) continue;
      const int pos = (int)rintf(__fmul_rn(__fdiv_rn(__fsub_rn(val[q], mn), span), (float)kFitGrid));
      if (pos == 0) ++n_lo;
      else if (pos == kFitGrid) ++n_hi;
      else atomicAdd(&hist[pos], 1ull);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_lo += __shfl_xor_sync(0xffffffffu, n_lo, o);
    n_hi += __shfl_xor_sync(0xffffffffu, n_hi, o);
  }
  if (lane == 0) {
    if (n_lo) atomicAdd(&hist[0], n_lo);
    if (n_hi) atomicAdd(&hist[kFitGrid], n_hi);
  }
}

// One CTA: exclusive prefix sums pc[i] = sum_{b<i} hist[b] and
// ps[i] = sum_{b<i} b hist[b] (i = 0 .. 2^16 + 1), then Lloyd in one thread:
// the positions of level i's cell, (t_{i-1}, t_i] with t the midpoints, are
// the integers floor(t_{i-1}) + 1 .. floor(t_i), so a cell's count and sum
// are two differences of prefix sums.
__global__ void __launch_bounds__(1024)
    nuq_fit_lloyd_kernel(const unsigned long long* __restrict__ hist, unsigned long long* __restrict__ pc,
                         unsigned long long* __restrict__ ps, int max_iters, float* __restrict__ lut_out,
                         int* __restrict__ info_out) {
  constexpr int kBins = kFitGrid + 1;
  constexpr int kPer = (kBins + 1023) / 1024;
  __shared__ unsigned long long wc[32], wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b0 = tid * kPer, b1 = min(kBins, b0 + kPer);
  unsigned long long c = 0, sx = 0;
  for (int b = b0; b < b1; ++b) {
    const unsigned long long h = hist[b];
    c += h;
    sx += (unsigned long long)b * h;
  }
  // block-wide exclusive scan of (c, sx)
  unsigned long long ic = c, is = sx;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long tc = __shfl_up_sync(0xffffffffu, ic, o), ts = __shfl_up_sync(0xffffffffu, is, o);
    if (lane >= o) {
      ic += tc;
      is += ts;
    }
  }
  if (lane == 31) {
    wc[w] = ic;
    wsum[w] = is;
  }
  __syncthreads();
  if (w == 0) {
    unsigned long long vc = wc[lane], vs = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long tc = __shfl_up_sync(0xffffffffu, vc, o), ts = __shfl_up_sync(0xffffffffu, vs, o);
      if (lane >= o) {
        vc += tc;
        vs += ts;
      }
    }
    wc[lane] = vc - wc[lane];  // exclusive over warps
    wsum[lane] = vs - wsum[lane];
  }
  __syncthreads();
  unsigned long long rc = wc[w] + ic - c, rs = wsum[w] + is - sx;
  for (int b = b0; b < b1; ++b) {
    pc[b] = rc;
    ps[b] = rs;
    const unsigned long long h = hist[b];
    rc += h;
    rs += (unsigned long long)b * h;
  }
  if (b1 == kBins && b0 < b1) {
    pc[kBins] = rc;
    ps[kBins] = rs;
  }
  __syncthreads();
  if (tid != 0) return;
  double l[8];
  for (int i = 0; i < 8; ++i) l[i] = (double)i * (double)kFitGrid / 7.0;
  int it = 0;
  while (it < max_iters) {
    double t[7];
    for (int i = 0; i < 7; ++i) t[i] = (l[i] + l[i + 1]) / 2.0;
    ++it;
    bool changed = false;
    for (int i = 1; i < 7; ++i) {
      const long long lo = (long long)floor(t[i - 1]) + 1, hi = (long long)floor(t[i]);
      if (hi < lo) continue;
      const unsigned long long n = pc[hi + 1] - pc[lo];
      if (n == 0) continue;
      const double nl = (double)(ps[hi + 1] - ps[lo]) / (double)n;
      if (nl != l[i]) changed = true;
      l[i] = nl;
    }
    if (!changed) break;
  }
  float lut[8];
  bool ok = true;
  for (int i = 0; i < 8; ++i) {
    lut[i] = __half2float(__float2half_rn((float)(l[i] / (double)kFitGrid)));
    if (i && !(lut[i] > lut[i - 1])) ok = false;
    lut_out[i] = lut[i];
  }
  if (info_out) *info_out = ok ? it : -1;
}

// --------------------------------------------------- distortion per head
// Mean squared error of the cache's uniform quantizers at `bits` on
// calibration tokens (RateQuant, "Methodology" 1 and 3: the distortion-rate
// curve of this quantizer, fitted per head, K and V separately).  One CTA
// per (32-token block, stream): K per channel over the block when it is
// whole (or, InnerQ keys, per token over 64-channel groups of the normalised
// keys), V per token over its channel groups (rotated first with Hadamard
// V); x^ = min + code scale from the stored fp16 pair, errors squared and
// summed in fp64 into sse[layer head][K, V].
__global__ void __launch_bounds__(kThreads)
    distortion_kernel(const __grid_constant__ AppendParams p, int n_tokens, int bits, const float* __restrict__ knorm,
                      double* __restrict__ sse) {
  const Geometry& G = p.geo;
  const int blk = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  __shared__ __align__(16) uint16_t sK[kGroupTokens][kRowHalves];
  __shared__ __align__(16) uint16_t sV[kGroupTokens][kRowHalves];
  __shared__ double red[2][kThreads / 32];
  const int t0 = blk * kGroupTokens, nt = min(kGroupTokens, n_tokens - t0);
  for (int idx = tid; idx < kGroupTokens * kRowVec; idx += kThreads) {
    const int r = idx / kRowVec, ch = idx % kRowVec;
    uint4 kx = make_uint4(0, 0, 0, 0), vx = kx;
    if (r < nt) {
      const size_t off = (in_stream(G, s) * n_tokens + t0 + r) * kRowHalves;
      kx = reinterpret_cast<const uint4*>(p.k_new + off)[ch];
      vx = reinterpret_cast<const uint4*>(p.v_new + off)[ch];
    }
    reinterpret_cast<uint4*>(&sK[r][0])[ch] = kx;
    reinterpret_cast<uint4*>(&sV[r][0])[ch] = vx;
  }
  __syncthreads();
  double ek = 0.0, ev = 0.0;
  if (!G.gkc) {
    if (nt == kGroupTokens) {  // per channel over the whole block
      const int c = tid;
      float x[kGroupTokens];
      float mn = INFINITY, mx = -INFINITY;
      long long sum = 0;
#pragma unroll
      for (int r = 0; r < kGroupTokens; ++r) {
        x[r] = half_bits_to_float(sK[r][c]);
        mn = fminf(mn, x[r]);
        mx = fmaxf(mx, x[r]);
        sum += fixed(x[r], 24);
      }
      const GroupQ gq = group_params(mn, mx, sum, 24, kGroupTokens, bits, G.hybrid);
      const double m = half_bits_to_float((uint16_t)(gq.word & 0xffffu)), sc = half_bits_to_float((uint16_t)(gq.word >> 16));
#pragma unroll
      for (int r = 0; r < kGroupTokens; ++r) {
        const double e = (double)x[r] - (m + (double)group_code(x[r], gq, bits) * sc);
        ek += e * e;
      }
    }
  } else {
    for (int r = w; r < nt; r += 4) {  // InnerQ keys: per token, 64-channel groups
      float v[4], n4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        n4[q] = G.knorm ? knorm[(size_t)s * kHeadDim + 4 * lane + q] : 1.0f;
        v[q] = __fdiv_rn(half_bits_to_float(sK[r][4 * lane + q]), n4[q]);
      }
      float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
      float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      const int sh = G.knorm ? 40 : 24;
      long long sum = (fixed(v[0], sh) + fixed(v[1], sh)) + (fixed(v[2], sh) + fixed(v[3], sh));
      for (int o = 8; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
      }
      const GroupQ gq = group_params(mn, mx, sum, sh, 64, bits, G.hybrid);
      const double m = half_bits_to_float((uint16_t)(gq.word & 0xffffu)), sc = half_bits_to_float((uint16_t)(gq.word >> 16));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const double e = ((double)v[q] - (m + (double)group_code(v[q], gq, bits) * sc)) * (double)n4[q];
        ek += e * e;
      }
    }
  }
  for (int r = w; r < nt; r += 4) {  // V per token over its channel groups
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = half_bits_to_float(sV[r][4 * lane + q]);
    if (G.hadamard) hadamard_vals(v, p.hadamard_c, lane);
    float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
    float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
    long long sum = (fixed(v[0], 24) + fixed(v[1], 24)) + (fixed(v[2], 24) + fixed(v[3], 24));
    const int seg = G.gv / 4;
    for (int o = seg / 2; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    const GroupQ gq = group_params(mn, mx, sum, 24, G.gv, bits, G.hybrid);
    const double m = half_bits_to_float((uint16_t)(gq.word & 0xffffu)), sc = half_bits_to_float((uint16_t)(gq.word >> 16));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const double e = (double)v[q] - (m + (double)group_code(v[q], gq, bits) * sc);
      ev += e * e;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ek += __shfl_xor_sync(0xffffffffu, ek, o);
    ev += __shfl_xor_sync(0xffffffffu, ev, o);
  }
  if (lane == 0) {
    red[0][w] = ek;
    red[1][w] = ev;
  }
  __syncthreads();
  if (tid == 0) {
    double a = 0.0, b = 0.0;
    for (int i = 0; i < kThreads / 32; ++i) {
      a += red[0][i];
      b += red[1][i];
    }
    const int h = layer_head(G, s % G.Hkv);
    atomicAdd(&sse[2 * h], a);
    atomicAdd(&sse[2 * h + 1], b);
  }
}

// The per-stream key normalisation of the calibration tokens (InnerQ keys).
__global__ void __launch_bounds__(kHeadDim) calib_norm_kernel(const __grid_constant__ AppendParams p, int n_tokens,
                                                               float* __restrict__ knorm) {
  const int s = blockIdx.x, c = threadIdx.x;
  const uint16_t* k = p.k_new + in_stream(p.geo, s) * n_tokens * kRowHalves + c;
  float m = 0.0f;
  for (int t = 0; t < n_tokens; ++t) m = fmaxf(m, fabsf(half_bits_to_float(k[(size_t)t * kRowHalves])));
  float n = 1.0f;
  if (m > 0.0f) {
    int e;
    frexpf(m, &e);
    n = ldexpf(1.0f, e);
    if (ldexpf(1.0f, e - 1) >= m) n = ldexpf(1.0f, e - 1);
  }
  knorm[(size_t)s * kHeadDim + c] = n;
}

// sse[h][j] /= count[j]: the mean squared errors.
__global__ void mse_finish_kernel(double* sse, int heads, double nk, double nv) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 2 * heads) sse[i] = (i & 1) ? (nv > 0 ? sse[i] / nv : 0.0) : (nk > 0 ? sse[i] / nk : 0.0);
}

}  // namespace

cudaError_t launch_distortion(const AppendParams& p, int n_tokens, int bits, float* knorm, double* mse,
                              cudaStream_t st) {
  const Geometry& G = p.geo;
  cudaError_t e = cudaMemsetAsync(mse, 0, sizeof(double) * 2 * G.Hkv_tot, st);
  if (e != cudaSuccess) return e;
  if (G.knorm) {
    calib_norm_kernel<<<G.NS, kHeadDim, 0, st>>>(p, n_tokens, knorm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  dim3 grid((n_tokens + kGroupTokens - 1) / kGroupTokens, G.NS);
  distortion_kernel<<<grid, kThreads, 0, st>>>(p, n_tokens, bits, knorm, mse);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // values per layer head: every batch row's keys (whole 32-token blocks per
  // channel, or every token) and values
  const double rows = (double)G.B;
  const double nk = rows * (G.gkc ? (double)n_tokens : (double)(n_tokens / kGroupTokens * kGroupTokens)) * kHeadDim;
  const double nv = rows * (double)n_tokens * kHeadDim;
  mse_finish_kernel<<<(2 * G.Hkv_tot + 127) / 128, 128, 0, st>>>(mse, G.Hkv_tot, nk, nv);
  return cudaGetLastError();
}

cudaError_t launch_nuq_fit(const uint16_t* x, long long nvec, int k, int hadamard, int max_iters, void* ws,
                           float* lut_out, int* info_out, cudaStream_t st) {
  unsigned long long* hist = reinterpret_cast<unsigned long long*>(ws);
  unsigned long long* pc = hist + (kFitGrid + 2);
  unsigned long long* ps = pc + (kFitGrid + 2);
  cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(unsigned long long) * (kFitGrid + 1), st);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  long long blocks = (nvec + kFitWarps - 1) / kFitWarps;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  nuq_fit_hist_kernel<<<(unsigned)blocks, 32 * kFitWarps, 0, st>>>(x, nvec, k, hadamard,
                                                                    (float)(1.0 / std::sqrt((double)kHeadDim)), hist);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  nuq_fit_lloyd_kernel<<<1, 1024, 0, st>>>(hist, pc, ps, max_iters, lut_out, info_out);
  return cudaGetLastError();
}

cudaError_t launch_append_quantize(const AppendParams& p, int n_groups, cudaStream_t st) {
  dim3 grid(n_groups, p.geo.NS);
  const int kb = p.geo.kb, vb = p.geo.vb, km = kb == 3 ? 2 : p.geo.gkc ? 1 : 0;
  bool done = false;
  auto go = [&](auto kernel) {
    kernel<<<grid, kThreads, 0, st>>>(p);
    done = true;
  };
  if (km == 2) go(append_quantize_kernel<2, 3, 3>);
#define KVQ_APPEND(K, V)                                          \
  if (km == 0 && kb == K && vb == V) go(append_quantize_kernel<0, K, V>); \
  if (km == 1 && kb == K && vb == V) go(append_quantize_kernel<1, K, V>);
  KVQ_APPEND(2, 2) KVQ_APPEND(2, 4) KVQ_APPEND(2, 8) KVQ_APPEND(4, 2) KVQ_APPEND(4, 4) KVQ_APPEND(4, 8)
  KVQ_APPEND(8, 2) KVQ_APPEND(8, 4) KVQ_APPEND(8, 8)
#undef KVQ_APPEND
  return done ? cudaGetLastError() : cudaErrorInvalidValue;
}

// A ragged append's per-row counts into the layer buffer's rows region
// (read by the append kernels that follow on the stream).
struct AppendRows {
  int before[kMaxRaggedRows];
  int n[kMaxRaggedRows];
};
__global__ void append_rows_kernel(const __grid_constant__ AppendRows r, int rows, int* dst) {
  const int b = threadIdx.x;
  if (b < rows) {
    dst[b] = r.before[b];
    dst[kMaxRaggedRows + b] = r.n[b];
  }
}
cudaError_t launch_append_rows(const int32_t* before, const int32_t* n, int rows, int* dst, cudaStream_t st) {
  AppendRows r;
  std::memset(&r, 0, sizeof(r));
  for (int b = 0; b < rows; ++b) {
    r.before[b] = before[b];
    r.n[b] = n[b];
  }
  append_rows_kernel<<<1, kMaxRaggedRows, 0, st>>>(r, rows, dst);
  return cudaGetLastError();
}

// A ragged decode's row tables into the workspace (read by the decode that
// follows on the stream, after its dependent-launch wait).
__global__ void ragged_tables_kernel(const __grid_constant__ RaggedTables t, RaggedTables* dst) {
  for (int i = threadIdx.x; i < kMaxRaggedRows + 1; i += blockDim.x) {
    if (i < kMaxRaggedRows) dst->tokens[i] = t.tokens[i];
    dst->j0[i] = t.j0[i];
    dst->x0[i] = t.x0[i];
  }
}
cudaError_t launch_ragged_tables(const RaggedTables& t, RaggedTables* dst, cudaStream_t st) {
  ragged_tables_kernel<<<1, kMaxRaggedRows, 0, st>>>(t, dst);
  return cudaGetLastError();
}

cudaError_t launch_key_norm(const AppendParams& p, cudaStream_t st) {
  key_norm_zero_kernel<<<p.geo.NS, kHeadDim, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  key_norm_max_kernel<<<dim3((p.n_new + kNormTokens - 1) / kNormTokens, p.geo.NS), kHeadDim, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  key_norm_pow2_kernel<<<p.geo.NS, kHeadDim, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append_window(const AppendParams& p, int ncopy, cudaStream_t st) {
  const size_t total = (size_t)p.geo.NS * ncopy * (2 * kRowVec);
  size_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;  // nothing to copy: the launch still keeps the dependent-launch chain
  return launch_dependent(append_window_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p, ncopy);
}

}  // namespace kvq
