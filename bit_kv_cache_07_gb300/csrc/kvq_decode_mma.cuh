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


__device__ __forceinline__ uint32_t lop3_or_and(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));  // (a & mask) | magic
  return r;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// V codes to exact fp16 pairs, centred: the value is code - 2^(b-1), so the
// accumulated sum of codes x P' stays small and the fp32 accumulator loses
// nothing to cancellation against the V-min term (which takes the centre:
// min' = min + 2^(b-1) * scale).  The magic exponent 0x6400 makes the fp16
// value 1024 + x for an integer x < 1024 placed in the low mantissa bits;
// one half-precision subtract or multiply-add removes the offset and the
// centre, every step exact.
//
// 4-bit: word w holds nibbles 0..7; pair i in 0..3 is (nibble i, nibble i+4).
__device__ __forceinline__ uint32_t ext4(uint32_t w, int i) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1024 + 8
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
  const __half2 km72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));   // -(64 + 8)
  const uint32_t x = (i >= 2) ? (w >> 8) : w;
  if ((i & 1) == 0) return h2_as_u32(__hsub2(u32_as_h2(lop3_or_and(x, 0x000F000Fu, 0x64006400u)), k1032));
  return h2_as_u32(__hfma2(u32_as_h2(lop3_or_and(x, 0x00F000F0u, 0x64006400u)), k16th, km72));
}

// 8-bit: word w holds bytes 0..3; pair i in 0..1 is (byte i, byte i+2).
__device__ __forceinline__ uint32_t ext8(uint32_t w, int i) {
  const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1024 + 128
  const uint32_t sel = (i == 0) ? 0x4240u : 0x4341u;
  return h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w, 0x64646464u, sel)), k1152));
}

// 2-bit: word w holds crumbs 0..15; pair i in 0..7 is (crumb i, crumb i+8).
__device__ __forceinline__ uint32_t ext2(uint32_t w, int i) {
  const uint32_t x = (i >= 4) ? (w >> 8) : w;
  const int m = i & 3;
  const uint32_t v = lop3_or_and(x, 0x00030003u << (2 * m), 0x64006400u);  // 1024 + 4^m c
  // (1024 + 4^m c) * 4^-m - (1024 * 4^-m + 2) = c - 2, every step exact in fp16
  const uint16_t sc[4] = {0x3C00, 0x3400, 0x2C00, 0x2400};   // 1, 1/4, 1/16, 1/64
  const uint16_t of[4] = {0xE402, 0xDC08, 0xD420, 0xCC80};   // -1026, -258, -66, -18
  const __half2 s = __halves2half2(__ushort_as_half(sc[m]), __ushort_as_half(sc[m]));
  const __half2 o = __halves2half2(__ushort_as_half(of[m]), __ushort_as_half(of[m]));
  return h2_as_u32(__hfma2(u32_as_h2(v), s, o));
}

// ---------------------------------------------------------------- K side
// A fragment of k-step s for one token row, from this thread's 32-channel
// slice of the packed row (words w[]: KB=8: 8 words, KB=4: 4, KB=2: 2).
// Returns (lo, hi): lo holds k-slots (2t, 2t+1), hi holds (2t+8, 2t+9).
//
// The K codes enter the mma with the magic offset left in: one lop3 (or
// byte permute) per two codes and no fp16 fix-up.  For channel c the
// operand is 1024 + code * u_c, u_c = 1 (8-bit), 16^(c & 1) (4-bit) or
// 4^(c & 3) (2-bit), set by the bit field's place in its 16-bit half.  The
// Q' operand of channel c is scaled by 2^E / u_c (exact powers of two), so
// the mma sums 2^E (code q'_c + 1024 q'_c / u_c); the constant part,
// 1024 * sum_c q'_c / u_c, leaves with the group's bias.
template <int KB>
__device__ __forceinline__ void k_frag(const uint32_t* w, int s, uint32_t& lo, uint32_t& hi) {
  if (KB == 8) {
    lo = __byte_perm(w[s], 0x64646464u, 0x4240u);
    hi = __byte_perm(w[s], 0x64646464u, 0x4341u);
  } else if (KB == 4) {
    const uint32_t x = (s & 1) ? (w[s >> 1] >> 8) : w[s >> 1];
    lo = lop3_or_and(x, 0x000F000Fu, 0x64006400u);  // 1024 + c
    hi = lop3_or_and(x, 0x00F000F0u, 0x64006400u);  // 1024 + 16 c
  } else {
    const int ia = 2 * (s & 3);  // pairs ia, ia + 1 of the word: crumb places ia & 3, (ia + 1) & 3
    const uint32_t x = (ia >= 4) ? (w[s >> 2] >> 8) : w[s >> 2];
    lo = lop3_or_and(x, 0x00030003u << (2 * (ia & 3)), 0x64006400u);        // 1024 + 4^m c
    hi = lop3_or_and(x, 0x00030003u << (2 * ((ia + 1) & 3)), 0x64006400u);
  }
}

// log2 of the common factor 2^E of the K-side B operand (keeps q'_c / u_c
// and its lo part clear of fp16 subnormals).
template <int KB>
__device__ __forceinline__ constexpr int kq_exp() { return KB == 8 ? 0 : KB == 4 ? 4 : 6; }
// Q' multiplier 2^E / u_c for channel c with c & 3 == k.
template <int KB>
__device__ __forceinline__ constexpr float kq_mult(int k) {
  return KB == 8 ? 1.0f : KB == 4 ? ((k & 1) ? 1.0f : 16.0f) : (k == 0 ? 64.0f : k == 1 ? 16.0f : k == 2 ? 4.0f : 1.0f);
}

// Where channel offset o (0..31) of a thread's slice lands: k-step s and
// element e (0,1: the lo register's halves; 2,3: the hi register's).
template <int KB>
__host__ __device__ __forceinline__ void k_slot_of(int o, int& s, int& e) {
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

// ------------------------------------------------------------- stage layout
// One pipeline stage holds one 32-token group: K codes, the group's K
// {min, scale} per channel, V codes, V {min, scale} per (token, channel
// group).  Code rows are stored unpadded; their 16-byte chunks are XOR-
// swizzled by row (chunk ^= bits 7.. of the byte offset, masked), so that
// the fragment reads -- 8 rows x 16 bytes per 8x8 matrix -- touch 32
// distinct banks.
__device__ __forceinline__ uint32_t swz(uint32_t off, uint32_t mask) { return off ^ (((off >> 7) & mask) << 4); }

//
// InnerQ keys (IQ: per-token groups of 64 channels) keep a group's per-token
// K {min, scale} words (2 per token, 256 bytes) where the per-channel words
// would be, and their code rows use a different swizzle (iq_kswz): a thread
// reads the two halves of its key channels from the two 64-channel groups.
template <int KB, int VB, bool IQ = false>
struct StageGeom {
  static constexpr int KROW = kHeadDim * KB / 8;
  static constexpr int VROW = kHeadDim * VB / 8;
  static constexpr uint32_t KSW = KB == 8 ? 7u : 0u;         // 128-byte K rows need it
  static constexpr uint32_t VSW = (uint32_t)(VROW / 16 - 1);  // 32/64/128-byte V rows
  static constexpr int KC = 0;
  static constexpr int KS = KC + kGroupTokens * KROW;
  static constexpr int KSB = IQ ? kGroupTokens * 8 : kHeadDim * 4;  // K scale bytes of a group
  static constexpr int VC = KS + KSB;
  static constexpr int VS = VC + kGroupTokens * VROW;
  static constexpr int BYTES = ((VS + kGroupTokens * kNVG * 4) + 127) / 128 * 128;
};

// Per-warp scratch of the group processing:
//  bq:  each lane's B fragments of Q' (32 halves = one 64-byte row per lane,
//       chunks swizzled like a 64-byte code row)
//  vsc/vmn: V scale / min of the group's tokens in fp32, ordered so that
//       the 4 tokens a lane needs sit in one 16-byte vector:
//       vsc[j][kt][tq][4] holds tokens 16kt + 2tq + {0, 1, 8, 9} (P' build),
//       vmn[j][gq][4]     holds tokens gq + {0, 8, 16, 24}     (softmax rows)
template <int NT>
struct MmaWarpSmem {
  alignas(128) uint16_t bq[NT][32][32];
  alignas(16) float bias[8 * NT];
  alignas(16) float vsc[kNVG][kGroupTokens];
  alignas(16) float vmn[kNVG][kGroupTokens];
};

__device__ __forceinline__ int vsc_index(int t) {  // token -> slot in vsc[j][..]
  const int r = t & 15;
  return (t >> 4) * 16 + ((r & 7) >> 1) * 4 + (r & 1) + 2 * (r >> 3);
}
__device__ __forceinline__ int vmn_index(int t) { return (t & 7) * 4 + (t >> 3); }

__device__ __forceinline__ float ex2(float x) {  // 2^x (hardware approximation; 2^-inf = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// InnerQ key rows: thread tq of a quad reads bytes [NB tq, NB tq + NB) of
// its row (channels 16 tq .. 16 tq + 15 of group 0) and the same bytes of the
// row's second half (group 1), NB = KROW / 8.  Rows r and r + 128 / KROW (the
// same banks) would collide, so rows with bit 7 of their byte offset set swap
// 16-byte chunks by XOR with KROW / 2 (chunk-granular: the 16-byte copies stay
// aligned): the quad's reads of 8 (KB 2), 4 (KB 4) or 2 (KB 8) rows then hit
// distinct banks.
template <int KB>
__host__ __device__ __forceinline__ uint32_t iq_kswz(uint32_t off) {
  constexpr uint32_t half_row = kHeadDim * KB / 16;
  return off ^ (((off >> 7) & 1u) * half_row);
}

// Queue the asynchronous copies of one 32-token group of stream s into the
// stage at shared address dst.  Every lane issues its share.
template <int KB, int VB, bool IQ = false>
__device__ __forceinline__ void issue_group(const DecodeParams& p, int s, int grp, uint32_t dst, int lane) {
  using SG = StageGeom<KB, VB, IQ>;
  // first row of the group in the stream-major regions (< 2^31: checked on the host);
  // the group's K scales are the 128 words at row0 * 4, its V scales the words at row0 * kNVG
  const uint32_t row0 = (uint32_t)s * (uint32_t)p.geo.qcap + (uint32_t)grp * kGroupTokens;
  const uint8_t* kc = p.L.k_codes + (size_t)row0 * SG::KROW + 16 * lane;
  const uint8_t* vc = p.L.v_codes + (size_t)row0 * SG::VROW + 16 * lane;
  // per-channel K: the group's 128 {min, scale} words at row0 * 4; InnerQ K:
  // 2 words per token at row0 * 2
  const uint8_t* ks = reinterpret_cast<const uint8_t*>(p.L.k_scales) + (size_t)row0 * (IQ ? 8 : 16) + 16 * lane;
  const uint8_t* vs = reinterpret_cast<const uint8_t*>(p.L.v_scales) + (size_t)row0 * (4 * kNVG) + 16 * lane;
  constexpr int KCH = kGroupTokens * SG::KROW / 16, VCH = kGroupTokens * SG::VROW / 16;
  static_assert(KCH % 32 == 0 && VCH % 32 == 0, "whole chunks per lane");
#pragma unroll
  for (int n = 0; n < KCH / 32; ++n) {
    const uint32_t off = 16 * (lane + 32 * n);
    cp_async16(dst + SG::KC + (IQ ? iq_kswz<KB>(off) : swz(off, SG::KSW)), kc + 512 * n);
  }
  if (!IQ || lane < SG::KSB / 16) cp_async16(dst + SG::KS + 16 * lane, ks);  // 512 B or 256 B of K scales
#pragma unroll
  for (int n = 0; n < VCH / 32; ++n) cp_async16(dst + SG::VC + swz(16 * (lane + 32 * n), SG::VSW), vc + 512 * n);
  if (lane < kGroupTokens * kNVG / 4) cp_async16(dst + SG::VS + 16 * lane, vs);
}

// V group (0 .. d/G_V - 1) of m-tile mc: every m-tile lies inside one group.
template <int VB>
__device__ __forceinline__ constexpr int v_group(int mc) {
  return (VB == 8 ? 16 * mc : VB == 4 ? 32 * (mc >> 1) : 64 * (mc >> 2)) / kGV;
}

// Warp reduce-scatter of NV per-lane values (NV = 1, 2, 4, 8): afterwards a
// lane holds the warp-wide sum of value head_of_lane<NV>(lane).  Each of the
// first log2(NV) butterfly steps halves the values a lane keeps, the rest
// finish the sum: log2(NV) + 5 - log2(NV) rounds instead of 5 per value.
template <int NV>
__device__ __forceinline__ float reduce_heads(const float (&v)[NV], int lane) {
  float a[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) a[i] = v[i];
#pragma unroll
  for (int n = NV, bit = 16; n > 1; n >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? a[i + n / 2] : a[i];
      const float send = up ? a[i] : a[i + n / 2];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
#pragma unroll
  for (int bit = 16 / NV; bit >= 1; bit >>= 1) a[0] += __shfl_xor_sync(0xffffffffu, a[0], bit);
  return a[0];
}
template <int NV>
__device__ __forceinline__ int head_of_lane(int lane) {
  return NV == 8 ? (lane >> 2) & 7 : NV == 4 ? (lane >> 3) & 3 : NV == 2 ? (lane >> 4) & 1 : 0;
}
// lane bits not used to select the head (lanes that hold the same sum)
template <int NV>
__device__ __forceinline__ constexpr int rest_mask() { return 32 / NV - 1; }

// hi (or lo) fp16 part of x, as a float: lanes with lo = 1 get x - fp16(x).
__device__ __forceinline__ float split_part(float x, float lo) {
  return fmaf(-lo, __half2float(__float2half_rn(x)), x);
}
// The same for two values, packed: fp16x2 of (x0, x1) (lo = 0) or of their
// remainders x - fp16(x) (lo = 1).
__device__ __forceinline__ uint32_t split_pack(float2 x, float lo) {
  const float2 h = __half22float2(__floats2half2_rn(x.x, x.y));
  const float2 y = __ffma2_rn(make_float2(-lo, -lo), h, x);
  return h2_as_u32(__floats2half2_rn(y.x, y.y));
}

// hi and lo fp16 parts of two values, both packed: x = hi + lo to ~2^-22.
__device__ __forceinline__ void split_hilo(float2 x, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x.x, x.y);
  const float2 r = __ffma2_rn(make_float2(-1.0f, -1.0f), __half22float2(h), x);
  hi = h2_as_u32(h);
  lo = h2_as_u32(__floats2half2_rn(r.x, r.y));
}

// Column layouts of the mma B operands (Q' and P') and of the D fragments.
// Up to 4 heads (one n-tile, NT = 1): column = (head, hi/lo), the hi and lo
// products summed over column pairs afterwards.  5-8 heads (NT = 2): the
// head layout -- column = head, and the hi and lo parts go through two mma
// into the same accumulator -- so O needs one n-tile instead of two and the
// logits need no column sums.  A lane's two softmax slots are then heads
// 2 tq + i (its own D columns) instead of 4 i + tq.
template <int NT>
__device__ __forceinline__ constexpr bool head_cols() { return NT == 2; }
template <int NT>
__device__ __forceinline__ constexpr int o_tiles() { return head_cols<NT>() ? 1 : NT; }
template <int NT>
__device__ __forceinline__ int slot_head(int i, int tq) { return head_cols<NT>() ? 2 * tq + i : 4 * i + tq; }

// Channels of this lane in the Q' build: c0, c0 + 1, c0 + D, c0 + D + 1 with
// (c0, c0 + D) and (c0 + 1, c0 + D + 1) the two halves of the B-fragment
// words 2s and 2s + 1 (s = lane & 7) of reader thread lane >> 3, for every
// code width (the k-slot order of k_frag / k_slot_of).
template <int KB>
__device__ __forceinline__ constexpr int qb_pair_dist() { return KB == 8 ? 2 : KB == 4 ? 4 : 8; }
template <int KB>
__device__ __forceinline__ int qb_first_channel(int lane) {
  return KB == 8 ? 4 * lane : KB == 4 ? 8 * (lane >> 1) + 2 * (lane & 1) : 16 * (lane >> 2) + 2 * (lane & 3);
}

// The query of a stream sits in shared memory permuted so that lane L reads
// its four Q'-build channels (c0, c0 + D, c0 + 1, c0 + D + 1) as one float4
// at 4L: position of channel c.
template <int KB>
__device__ __forceinline__ int qb_perm_pos(int c) {
  constexpr int D = qb_pair_dist<KB>();
  int L, c0;
  if (KB == 8) {
    L = c >> 2;
  } else if (KB == 4) {
    L = 2 * (c >> 3) + ((c >> 1) & 1);
  } else {
    L = 4 * (c >> 4) + ((c >> 1) & 3);
  }
  c0 = qb_first_channel<KB>(L);
  const int rel = c - c0;  // 0, 1, D or D + 1
  return 4 * L + (rel >= D ? 1 : 0) + 2 * (rel & 1);
}

// ------------------------------------------------------------- InnerQ keys
// Per-warp scratch of the InnerQ key path: the group's per-token K scale and
// min for its two 64-channel groups (ordered like vmn: the 4 tokens gq + 8i a
// lane needs sit in one 16-byte vector), and per query head of the stream
// the constants {Ohat_0, Ohat_1, Q_0, Q_1} of its two groups (see build_bq_iq).
struct IqWarpSmem {
  alignas(16) float ksc[2][kGroupTokens];
  alignas(16) float kmn[2][kGroupTokens];
  alignas(16) float iqc[kMaxGQA][4];
};

// The inverse of k_slot_of: the channel offset o (0..31) of a thread's slice
// that k-step s, element e takes.
template <int KB>
__host__ __device__ __forceinline__ constexpr int k_offset_of(int s, int e) {
  return KB == 8 ? 4 * s + ((e >> 1) | ((e & 1) << 1))
         : KB == 4 ? 8 * (s >> 1) + (((e & 1) << 2) | ((s & 1) << 1) | (e >> 1))
                   : 16 * (s >> 2) + (((e & 1) << 3) | ((s & 3) << 1) | (e >> 1));
}
// InnerQ: the key channel of slice offset o of thread tq (half from each group)
__host__ __device__ __forceinline__ constexpr int iq_channel(int tq, int o) {
  return o < 16 ? 16 * tq + o : kHeadDim / 2 + 16 * tq + (o - 16);
}

// The Q' fragments of an InnerQ stream, built once per stream: with keys
// grouped per token, K's scales no longer enter q (they multiply each group's
// partial product after the mma), so Q' = q * n_c (the channel's key
// normalisation) * 2^E / u_c, split into hi + lo fp16, is constant over the
// stream.  Each lane writes its own fragment row (the layout process_group's
// step (b) reads).  Per head h and group j it also stores
//   Ohat_j = 2^-E * 1024 * sum_{c in j} (hi + lo)_c   (the magic offset the
//            mma adds: the group's code product is S_j 2^-E - Ohat_j)
//   Q_j    = sum_{c in j} q_c n_c                        (for the K min term)
// in logit units.  qw holds q * softmax scale in the qb_perm_pos<KB> order.
template <int KB, int NT>
__device__ __forceinline__ void build_bq_iq(const float (*qw)[kHeadDim], const float* __restrict__ knorm,
                                            MmaWarpSmem<NT>& sm, IqWarpSmem& iq, int g, int lane) {
  constexpr bool HC = head_cols<NT>();
  constexpr float kE = (float)(1 << kq_exp<KB>());
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = HC ? gq : 4 * nt + (gq >> 1);
    const bool lo = HC ? (nt == 1) : ((gq & 1) != 0);
    uint32_t reg[16];
#pragma unroll
    for (int ri = 0; ri < 16; ++ri) {
      uint32_t hv[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int c = iq_channel(tq, k_offset_of<KB>(ri >> 1, 2 * (ri & 1) + x));
        float v = 0.0f;
        if (h < g) v = qw[h][qb_perm_pos<KB>(c)] * (knorm ? __ldg(knorm + c) : 1.0f) * kq_mult<KB>(c & 3);
        const __half hi = __float2half_rn(v);
        hv[x] = __half_as_ushort(lo ? __float2half_rn(v - __half2float(hi)) : hi);
      }
      reg[ri] = hv[0] | (hv[1] << 16);
    }
    unsigned char* row = reinterpret_cast<unsigned char*>(&sm.bq[nt][lane][0]);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      *reinterpret_cast<uint4*>(row + 16 * (c4 ^ ((lane >> 1) & 3))) =
          make_uint4(reg[4 * c4], reg[4 * c4 + 1], reg[4 * c4 + 2], reg[4 * c4 + 3]);
  }
  // the constants: lane L sums channels 4L..4L+3 (all in group L / 16)
  for (int h = 0; h < g; ++h) {
    float oh = 0.0f, qs = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = 4 * lane + k;
      const float qn = qw[h][qb_perm_pos<KB>(c)] * (knorm ? __ldg(knorm + c) : 1.0f);
      const float v = qn * kq_mult<KB>(c & 3);
      const __half hi = __float2half_rn(v);
      const float lo = __half2float(__float2half_rn(v - __half2float(hi)));
      oh += (__half2float(hi) + lo) * (1024.0f / kE);
      qs += qn;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      oh += __shfl_xor_sync(0xffffffffu, oh, o);
      qs += __shfl_xor_sync(0xffffffffu, qs, o);
    }
    if ((lane & 15) == 0) {
      iq.iqc[h][lane >> 4] = oh;
      iq.iqc[h][2 + (lane >> 4)] = qs;
    }
  }
  __syncwarp();
}

// One 32-token group for one warp: Q' fragments, S = K Q' (2 m-tiles x NT
// n-tiles), online softmax, O += V^T P' (8 m-tiles x o_tiles<NT>()).
//
// JC (one n-tile, at most 2 heads): the PV B operand puts the V group into
// the columns too -- column = (head, V group, hi/lo) -- so a lane builds P'
// for one (head, group) pair instead of one per group; an m-tile's D
// columns of the other group are then unused (see stage_quant).
//
// IQ (InnerQ keys, per-token 64-channel groups): Q' is the stream's (built by
// build_bq_iq), step (a) only stages the group's per-token K {min, scale};
// in (c) k-steps 0-3 cover key group 0 and 4-7 group 1 in separate
// accumulators, and the logit of token t is
//   sum_j scale_tj (S_tj 2^-E - Ohat_j) + min_tj Q_j.
template <int KB, int VB, int NT, bool JC, int GT, bool IQ = false>
__device__ __forceinline__ void process_group(const float (*qw)[kHeadDim], MmaWarpSmem<NT>& sm, IqWarpSmem* iq,
                                              const unsigned char* st, int g, int lane,
                                              float (&O)[8][o_tiles<NT>()][4], float (&macc)[NT][kNVG],
                                              float (&m_used)[NT], float (&lsum)[NT]) {
  using SG = StageGeom<KB, VB, IQ>;
  constexpr bool HC = head_cols<NT>();
  const int gq = lane >> 2, tq = lane & 3;

  // (a) Q' = q * scale_k (hi + lo fp16) into this warp's fragment rows,
  //     bias = q . min_k; V {min, scale} of this lane's token to fp32
  //     (InnerQ keys: this lane's token's K {min, scale} per group instead)
  if constexpr (IQ) {
    const uint2 kw = *reinterpret_cast<const uint2*>(st + SG::KS + 8 * lane);
    const float2 k0 = unpack_min_scale(kw.x), k1 = unpack_min_scale(kw.y);
    const int im = vmn_index(lane);
    iq->kmn[0][im] = k0.x;
    iq->ksc[0][im] = k0.y;
    iq->kmn[1][im] = k1.x;
    iq->ksc[1][im] = k1.y;
  }
  {
    if constexpr (!IQ) {
    constexpr int D = qb_pair_dist<KB>();
    const int c0 = qb_first_channel<KB>(lane);
    const uint2 w01 = *reinterpret_cast<const uint2*>(st + SG::KS + 4 * c0);
    const uint2 w23 = *reinterpret_cast<const uint2*>(st + SG::KS + 4 * (c0 + D));
    const float2 ms[4] = {unpack_min_scale(w01.x), unpack_min_scale(w01.y), unpack_min_scale(w23.x),
                          unpack_min_scale(w23.y)};
    // channels c0, c0 + D share the power-of-two multiplier (same c & 3 class), as do c0 + 1, c0 + D + 1
    const float me = kq_mult<KB>(c0 & 3), mo = kq_mult<KB>((c0 + 1) & 3);
    // pairs A = (c0, c0 + D) -> B-word 2s, B = (c0 + 1, c0 + D + 1) -> B-word 2s + 1
    const float2 skA = make_float2(ms[0].y * me, ms[2].y * me), skB = make_float2(ms[1].y * mo, ms[3].y * mo);
    const float2 mnA = make_float2(ms[0].x, ms[2].x), mnB = make_float2(ms[1].x, ms[3].x);
    const int tsl = lane >> 3;                                        // reader thread-in-group of these channels
    const int wofs = (8 * (lane & 7)) ^ (((tsl >> 1) & 1) << 4);      // words 2s, 2s+1 in the (swizzled) hi row
    float bpart[GT];                                                  // this lane's share of each head's bias
#pragma unroll
    for (int r = 0; r < GT; ++r) {
      bpart[r] = 0.0f;
      if (r >= g) continue;
      // fragment rows (reader lanes) and byte offsets of the hi and lo words
      unsigned char* dhi;
      unsigned char* dlo;
      int whi, wlo;
      if constexpr (HC) {
        const int R = 4 * r + tsl;  // column r in table 0 (hi) and table 1 (lo)
        dhi = reinterpret_cast<unsigned char*>(&sm.bq[0][R][0]);
        dlo = reinterpret_cast<unsigned char*>(&sm.bq[1][R][0]);
        whi = wlo = (8 * (lane & 7)) ^ (((R >> 1) & 3) << 4);
      } else {
        dhi = reinterpret_cast<unsigned char*>(&sm.bq[r >> 2][8 * (r & 3) + tsl][0]);
        dlo = dhi + 4 * 64;
        whi = wofs;
        wlo = wofs ^ 32;
      }
      const float4 q4 = *reinterpret_cast<const float4*>(&qw[r][4 * lane]);  // (c0, c0+D, c0+1, c0+D+1)
      const float2 qA = make_float2(q4.x, q4.y), qB = make_float2(q4.z, q4.w);
      const float2 pA = __fmul2_rn(qA, skA), pB = __fmul2_rn(qB, skB);
      const __half2 hA = __floats2half2_rn(pA.x, pA.y), hB = __floats2half2_rn(pB.x, pB.y);
      const float2 m1 = make_float2(-1.0f, -1.0f);
      const float2 rA = __ffma2_rn(m1, __half22float2(hA), pA), rB = __ffma2_rn(m1, __half22float2(hB), pB);
      const __half2 lA = __floats2half2_rn(rA.x, rA.y), lB = __floats2half2_rn(rB.x, rB.y);
      *reinterpret_cast<uint2*>(dhi + whi) = make_uint2(h2_as_u32(hA), h2_as_u32(hB));
      *reinterpret_cast<uint2*>(dlo + wlo) = make_uint2(h2_as_u32(lA), h2_as_u32(lB));
      const float2 b2 = __ffma2_rn(qA, mnA, __fmul2_rn(qB, mnB));
      const float2 o2 = __fadd2_rn(pA, pB);  // hi + lo = qp to ~2^-22
      // the mma's constant part 1024 * sum_c (hi + lo), in logit units
      bpart[r] = fmaf(-1024.0f * (1.0f / (float)(1 << kq_exp<KB>())), o2.x + o2.y, b2.x + b2.y);
    }
    // all heads' biases with one reduce-scatter over the warp
    const float bsum = reduce_heads<GT>(bpart, lane);
    const int hb = head_of_lane<GT>(lane);
    if ((lane & rest_mask<GT>()) == 0 && hb < g) sm.bias[hb] = bsum;
    }
    const uint32_t* vsw = reinterpret_cast<const uint32_t*>(st + SG::VS);
    const int iv = vsc_index(lane), im = vmn_index(lane);
    constexpr float kVCentre = (float)(1 << (VB - 1));  // the V codes enter the mma centred
#pragma unroll
    for (int j = 0; j < kNVG; ++j) {
      const float2 m2 = unpack_min_scale(vsw[lane * kNVG + j]);
      sm.vmn[j][im] = fmaf(kVCentre, m2.y, m2.x);
      sm.vsc[j][iv] = m2.y;
    }
  }
  __syncwarp();

  // (b) this thread's Q' fragments (row = lane, chunks unswizzled on read)
  uint32_t bq[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const unsigned char* row = reinterpret_cast<const unsigned char*>(&sm.bq[nt][lane][0]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + 16 * (c ^ ((lane >> 1) & 3)));
      bq[nt][4 * c] = u.x; bq[nt][4 * c + 1] = u.y; bq[nt][4 * c + 2] = u.z; bq[nt][4 * c + 3] = u.w;
    }
  }

  // (c) S = K Q'
  float S[2][NT][4];
  float Z[2][NT][2];  // InnerQ keys: the logits (base 2) of this lane's tokens and head slots
  float4 iks0, iks1, ikm0, ikm1;  // InnerQ keys: scale / min of tokens gq + 8i, groups 0 and 1
  if constexpr (IQ) {
    iks0 = *reinterpret_cast<const float4*>(&iq->ksc[0][4 * gq]);
    iks1 = *reinterpret_cast<const float4*>(&iq->ksc[1][4 * gq]);
    ikm0 = *reinterpret_cast<const float4*>(&iq->kmn[0][4 * gq]);
    ikm1 = *reinterpret_cast<const float4*>(&iq->kmn[1][4 * gq]);
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) S[mt][nt][k] = 0.0f;
    constexpr int NW = SG::KROW / 16;  // words in this thread's 32-channel slice
    uint32_t w0[NW], w1[NW];
    const uint32_t o0 = (16 * mt + gq) * SG::KROW + 4 * NW * tq;
    const uint32_t o1 = o0 + 8 * SG::KROW;
    if constexpr (IQ) {
      // half of the slice from each 64-channel group: bytes NB tq .. of both row halves
      constexpr int NB = SG::KROW / 8;
      const uint32_t r0 = (16 * mt + gq) * SG::KROW + NB * tq, r1 = r0 + 8 * SG::KROW;
      const unsigned char* kc = st + SG::KC;
      if constexpr (NW == 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(kc + iq_kswz<KB>(r0));
        const uint4 b2 = *reinterpret_cast<const uint4*>(kc + iq_kswz<KB>(r0 + SG::KROW / 2));
        const uint4 c = *reinterpret_cast<const uint4*>(kc + iq_kswz<KB>(r1));
        const uint4 d2 = *reinterpret_cast<const uint4*>(kc + iq_kswz<KB>(r1 + SG::KROW / 2));
        w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w; w0[4] = b2.x; w0[5] = b2.y; w0[6] = b2.z; w0[7] = b2.w;
        w1[0] = c.x; w1[1] = c.y; w1[2] = c.z; w1[3] = c.w; w1[4] = d2.x; w1[5] = d2.y; w1[6] = d2.z; w1[7] = d2.w;
      } else if constexpr (NW == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(kc + iq_kswz<KB>(r0));
        const uint2 b2 = *reinterpret_cast<const uint2*>(kc + iq_kswz<KB>(r0 + SG::KROW / 2));
        const uint2 c = *reinterpret_cast<const uint2*>(kc + iq_kswz<KB>(r1));
        const uint2 d2 = *reinterpret_cast<const uint2*>(kc + iq_kswz<KB>(r1 + SG::KROW / 2));
        w0[0] = a.x; w0[1] = a.y; w0[2] = b2.x; w0[3] = b2.y;
        w1[0] = c.x; w1[1] = c.y; w1[2] = d2.x; w1[3] = d2.y;
      } else {
        w0[0] = *reinterpret_cast<const uint32_t*>(kc + iq_kswz<KB>(r0));
        w0[1] = *reinterpret_cast<const uint32_t*>(kc + iq_kswz<KB>(r0 + SG::KROW / 2));
        w1[0] = *reinterpret_cast<const uint32_t*>(kc + iq_kswz<KB>(r1));
        w1[1] = *reinterpret_cast<const uint32_t*>(kc + iq_kswz<KB>(r1 + SG::KROW / 2));
      }
    } else if constexpr (NW == 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(st + SG::KC + swz(o0, SG::KSW));
      const uint4 b2 = *reinterpret_cast<const uint4*>(st + SG::KC + swz(o0 + 16, SG::KSW));
      const uint4 c = *reinterpret_cast<const uint4*>(st + SG::KC + swz(o1, SG::KSW));
      const uint4 d2 = *reinterpret_cast<const uint4*>(st + SG::KC + swz(o1 + 16, SG::KSW));
      w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w; w0[4] = b2.x; w0[5] = b2.y; w0[6] = b2.z; w0[7] = b2.w;
      w1[0] = c.x; w1[1] = c.y; w1[2] = c.z; w1[3] = c.w; w1[4] = d2.x; w1[5] = d2.y; w1[6] = d2.z; w1[7] = d2.w;
    } else if constexpr (NW == 4) {
      const uint4 a = *reinterpret_cast<const uint4*>(st + SG::KC + o0);
      const uint4 c = *reinterpret_cast<const uint4*>(st + SG::KC + o1);
      w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
      w1[0] = c.x; w1[1] = c.y; w1[2] = c.z; w1[3] = c.w;
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(st + SG::KC + o0);
      const uint2 c = *reinterpret_cast<const uint2*>(st + SG::KC + o1);
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
      if constexpr (IQ) {
        // key group 0 (k-steps 0-3) into S, group 1 (4-7) into S2; head columns:
        // [0] hi and [1] lo tables
        float (*acc)[4] = s_ < 4 ? S[mt] : S2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma16816(acc[nt], lo0, lo1, hi0, hi1, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
      } else if constexpr (HC) {
        // hi and lo parts: two independent chains, summed below
        mma16816(S[mt][0], lo0, lo1, hi0, hi1, bq[0][2 * s_], bq[0][2 * s_ + 1]);
        mma16816(S[mt][1], lo0, lo1, hi0, hi1, bq[1][2 * s_], bq[1][2 * s_ + 1]);
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (s_ & 1)
            mma16816(S2[nt], lo0, lo1, hi0, hi1, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
          else
            mma16816(S[mt][nt], lo0, lo1, hi0, hi1, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
        }
      }
    }
    if constexpr (IQ) {
      // logit = sum_j scale_tj (S_tj 2^-E - Ohat_j) + min_tj Q_j, tokens gq + 8 (2 mt + rh)
      constexpr float kUn = 1.0f / (float)(1 << kq_exp<KB>());
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = slot_head<NT>(nt, tq);
        const float4 cst = *reinterpret_cast<const float4*>(&iq->iqc[h < g ? h : 0][0]);
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          const int i = 2 * mt + rh;
          const float a = HC ? S[mt][0][2 * rh + nt] + S[mt][1][2 * rh + nt] : S[mt][nt][2 * rh] + S[mt][nt][2 * rh + 1];
          const float b = HC ? S2[0][2 * rh + nt] + S2[1][2 * rh + nt] : S2[nt][2 * rh] + S2[nt][2 * rh + 1];
          const float s0 = i == 0 ? iks0.x : i == 1 ? iks0.y : i == 2 ? iks0.z : iks0.w;
          const float s1 = i == 0 ? iks1.x : i == 1 ? iks1.y : i == 2 ? iks1.z : iks1.w;
          const float m0 = i == 0 ? ikm0.x : i == 1 ? ikm0.y : i == 2 ? ikm0.z : ikm0.w;
          const float m1 = i == 0 ? ikm1.x : i == 1 ? ikm1.y : i == 2 ? ikm1.z : ikm1.w;
          float z = fmaf(s0, fmaf(a, kUn, -cst.x), m0 * cst.z);
          z = fmaf(s1, fmaf(b, kUn, -cst.y), fmaf(m1, cst.w, z));
          Z[mt][nt][rh] = z;
        }
      }
    } else if constexpr (HC) {
#pragma unroll
      for (int k = 0; k < 4; ++k) S[mt][0][k] += S[mt][1][k];
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) S[mt][nt][k] += S2[nt][k];
    }
  }

  // (d) online softmax (base 2); this thread's heads are slot_head(nt), its
  //     tokens gq + {0, 8, 16, 24}
  float P[NT][2][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = slot_head<NT>(nt, tq);
    const bool live = h < g;
    const float bias = (IQ || !live) ? 0.0f : sm.bias[h];
    float zs[2][2];
    float zm = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        // 2^E x (logit - bias); InnerQ keys: the logit
        zs[mt][rh] = IQ ? Z[mt][nt][rh] : HC ? S[mt][0][2 * rh + nt] : S[mt][nt][2 * rh] + S[mt][nt][2 * rh + 1];
        zm = fmaxf(zm, zs[mt][rh]);
      }
    constexpr float kUnscale = IQ ? 1.0f : 1.0f / (float)(1 << kq_exp<KB>());
    // The running maximum moves only when a logit exceeds it by 2^8, which is
    // rare after a stream's first group: test this lane's 4 logits and take
    // the group maximum (shuffles) only when some lane of the warp needs it.
    const bool need = live && fmaf(zm, kUnscale, bias) > m_used[nt] + kLazyRescale;
    if (__any_sync(0xffffffffu, need)) {
      zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 4));
      zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 8));
      zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 16));
      zm = live ? fmaf(zm, kUnscale, bias) : -INFINITY;
      const bool resc = zm > m_used[nt] + kLazyRescale;
      float alpha = 1.0f;
      if (resc) {
        alpha = ex2(m_used[nt] - zm);  // 0 when m_used is -inf
#pragma unroll
        for (int j = 0; j < kNVG; ++j) macc[nt][j] *= alpha;
        lsum[nt] *= alpha;
        m_used[nt] = zm;
      }
      if constexpr (JC) {
        // this lane's O columns belong to head tq >> 1
        const float a_o = __shfl_sync(0xffffffffu, alpha, (lane & ~3) | (tq >> 1));
#pragma unroll
        for (int mc = 0; mc < 8; ++mc)
#pragma unroll
          for (int k = 0; k < 4; ++k) O[mc][nt][k] *= a_o;
      } else if (resc) {
        if constexpr (HC) {
          // this lane's O columns are its own two heads
#pragma unroll
          for (int mc = 0; mc < 8; ++mc) {
            O[mc][0][nt] *= alpha;
            O[mc][0][2 + nt] *= alpha;
          }
        } else {
#pragma unroll
          for (int mc = 0; mc < 8; ++mc)
#pragma unroll
            for (int k = 0; k < 4; ++k) O[mc][nt][k] *= alpha;
        }
      }
    }
    const float bm = live ? bias - m_used[nt] : -INFINITY;
    float ps = 0.0f;
    float pv[4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        pv[2 * mt + rh] = ex2(fmaf(zs[mt][rh], kUnscale, bm));
        P[nt][mt][rh] = pv[2 * mt + rh];
        ps += pv[2 * mt + rh];
      }
#pragma unroll
    for (int j = 0; j < kNVG; ++j) {
      const float4 mn = *reinterpret_cast<const float4*>(&sm.vmn[j][4 * gq]);  // tokens gq + 8i
      macc[nt][j] = fmaf(pv[0], mn.x, fmaf(pv[1], mn.y, fmaf(pv[2], mn.z, fmaf(pv[3], mn.w, macc[nt][j]))));
    }
    lsum[nt] += ps;
  }

  // (e) O += V^T P'
  const float lo_sel = (gq & 1) ? 1.0f : 0.0f;  // this lane's B column is a lo column
#pragma unroll
  for (int kt = 0; kt < 2; ++kt) {
    // V code fragments: ldmatrix.trans on the packed (swizzled) rows, then
    // the A fragment of m-tile mc from blocks of them
    const uint32_t vbase = smem_u32(st + SG::VC);
    const int mi = lane >> 3, rr = lane & 7;
    constexpr int NBLK = VB == 8 ? 8 : VB == 4 ? 4 : 2;  // 16-byte blocks of a V row
    uint32_t R[NBLK][2];  // [block][token half]
#pragma unroll
    for (int c = 0; c < NBLK / 2; ++c) {
      const int blk = 2 * c + (mi >> 1), th = mi & 1;
      const uint32_t addr = vbase + swz((16 * kt + 8 * th + rr) * SG::VROW + 16 * blk, SG::VSW);
      ldsm_x4_trans(R[2 * c][0], R[2 * c][1], R[2 * c + 1][0], R[2 * c + 1][1], addr);
    }
    auto afrag = [&](int mc, uint32_t (&A)[4]) {
      if (VB == 4) {
        const int blk = mc >> 1, i = mc & 1;
        A[0] = ext4(R[blk][0], i); A[1] = ext4(R[blk][0], i + 2);
        A[2] = ext4(R[blk][1], i); A[3] = ext4(R[blk][1], i + 2);
      } else if (VB == 8) {
        A[0] = ext8(R[mc][0], 0); A[1] = ext8(R[mc][0], 1);
        A[2] = ext8(R[mc][1], 0); A[3] = ext8(R[mc][1], 1);
      } else {
        const int blk = mc >> 2, i = mc & 3;
        A[0] = ext2(R[blk][0], i); A[1] = ext2(R[blk][0], i + 4);
        A[2] = ext2(R[blk][1], i); A[3] = ext2(R[blk][1], i + 4);
      }
    };
    if constexpr (HC) {
      // P' of tokens 16kt + 2tq + {0, 1} (+8) for head gq: held by lanes
      // 4 (2tq + e) + (gq >> 1) in softmax slot gq & 1
      float pv[2][2];  // [row half][token parity]
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int src = 4 * (2 * tq + e) + (gq >> 1);
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          const float p0 = __shfl_sync(0xffffffffu, P[0][kt][rh], src);
          const float p1 = __shfl_sync(0xffffffffu, P[1][kt][rh], src);
          pv[rh][e] = (gq & 1) ? p1 : p0;
        }
      }
      uint32_t bh[kNVG][2], bl[kNVG][2];
#pragma unroll
      for (int j = 0; j < kNVG; ++j) {
        const float4 sv = *reinterpret_cast<const float4*>(&sm.vsc[j][16 * kt + 4 * tq]);
        split_hilo(__fmul2_rn(make_float2(pv[0][0], pv[0][1]), make_float2(sv.x, sv.y)), bh[j][0], bl[j][0]);
        split_hilo(__fmul2_rn(make_float2(pv[1][0], pv[1][1]), make_float2(sv.z, sv.w)), bh[j][1], bl[j][1]);
      }
      // hi parts over all m-tiles, then lo parts: no back-to-back accumulator dependence
      uint32_t A[8][4];
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        afrag(mc, A[mc]);
        const int j = v_group<VB>(mc);
        mma16816(O[mc][0], A[mc][0], A[mc][1], A[mc][2], A[mc][3], bh[j][0], bh[j][1]);
      }
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const int j = v_group<VB>(mc);
        mma16816(O[mc][0], A[mc][0], A[mc][1], A[mc][2], A[mc][3], bl[j][0], bl[j][1]);
      }
    } else {
      // P' fragments per (n-tile, V group): tokens 16kt + {2tq, 2tq+1, 2tq+8, 2tq+9}, column gq
      // (JC: one fragment; column gq = head gq >> 2, V group (gq >> 1) & 1)
      uint32_t bp[NT][kNVG][2];
      const int src1 = 8 * tq + (JC ? (gq >> 2) : (gq >> 1)), src2 = src1 + 4;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float v0 = __shfl_sync(0xffffffffu, P[nt][kt][0], src1);
        const float v1 = __shfl_sync(0xffffffffu, P[nt][kt][0], src2);
        const float v2 = __shfl_sync(0xffffffffu, P[nt][kt][1], src1);
        const float v3 = __shfl_sync(0xffffffffu, P[nt][kt][1], src2);
#pragma unroll
        for (int j = 0; j < (JC ? 1 : kNVG); ++j) {
          const int jv = JC ? ((gq >> 1) & 1) : j;
          const float4 sv = *reinterpret_cast<const float4*>(&sm.vsc[jv][16 * kt + 4 * tq]);
          bp[nt][j][0] = split_pack(__fmul2_rn(make_float2(v0, v1), make_float2(sv.x, sv.y)), lo_sel);
          bp[nt][j][1] = split_pack(__fmul2_rn(make_float2(v2, v3), make_float2(sv.z, sv.w)), lo_sel);
        }
      }
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        uint32_t A[4];
        afrag(mc, A);
        const int j = JC ? 0 : v_group<VB>(mc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(O[mc][nt], A[0], A[1], A[2], A[3], bp[nt][j][0], bp[nt][j][1]);
      }
    }
  }
}

// ------------------------------------------------------------ fp16 items
// The fp16 tokens of a stream (sinks, then the recent window; or the whole
// cache in fp16 mode) are processed in items of kF16Tokens tokens that go
// through the same asynchronous-copy pipeline and tensor-core path as the
// quantized groups: K rows are the A operand of S = K Q (rows = tokens), V
// rows (transposed by ldmatrix) the A operand of O += V^T P.  An item's K
// and V rows (256 bytes each) sit in the stage with their 16-byte chunks
// swizzled: K chunk c of row t at c ^ 4(t & 1) (the fragment loads of a
// quarter warp read rows 2i, 2i+1), V chunk c at c ^ (t & 7) (ldmatrix
// reads one chunk of 8 consecutive rows).
constexpr int kF16Tokens = kPersistF16Tokens;

struct F16Geom {
  static constexpr int KC = 0;
  static constexpr int VC = kF16Tokens * kHeadDim * 2;
  static constexpr int BYTES = 2 * kF16Tokens * kHeadDim * 2;
};
__device__ __forceinline__ uint32_t kf16_off(int t, int c) { return t * 256 + 16 * (c ^ (4 * (t & 1))); }
__device__ __forceinline__ uint32_t vf16_off(int t, int c) { return t * 256 + 16 * (c ^ (t & 7)); }

// 16-byte asynchronous copy that writes zeros instead when !valid (the
// source address is not read then, but stays a valid one).
__device__ __forceinline__ void cp_async16_zfill(uint32_t smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem), "l"(gmem), "r"(valid ? 16 : 0));
}

__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// Queue the copies of fp16 item (stream s, first fp16 token kk0; tokens at
// or past k1 are zero-filled).  Lanes 0-15 copy the even tokens' rows,
// lanes 16-31 the odd ones', one 16-byte chunk of K and of V each.
__device__ __forceinline__ void issue_f16(const DecodeParams& p, int s, int kk0, int k1, int S_eff, int Nq,
                                          uint32_t dst, int lane) {
  const int c = lane & 15;
#pragma unroll
  for (int n = 0; n < kF16Tokens / 2; ++n) {
    const int t = 2 * n + (lane >> 4);
    const int kk = kk0 + t;
    const bool valid = kk < k1;
    bool sink;
    int pos;
    const size_t off = fp16_row_at(p, s, valid ? kk : kk0, S_eff, Nq, &sink, &pos);
    const uint16_t* kr = (sink ? p.L.k_sink : p.L.k_ring) + off;
    const uint16_t* vr = (sink ? p.L.v_sink : p.L.v_ring) + off;
    cp_async16_zfill(dst + F16Geom::KC + kf16_off(t, c), kr + 8 * c, valid);
    cp_async16_zfill(dst + F16Geom::VC + vf16_off(t, c), vr + 8 * c, valid);
  }
}

// B fragments of the (unquantized) query for the fp16 items, hi + lo fp16
// per head.  Slot order: thread tq of the k dimension owns the 16-byte K
// chunks tq, tq+4, tq+8, tq+12 (channels 8 * chunk ..); k-step s = 2i + h
// takes channels 8(tq + 4i) + 4h + {0, 1} (lo pair) and + {2, 3} (hi pair).
template <int NT, int KBQ>
__device__ __forceinline__ void build_bq_f16(const float (*qw)[kHeadDim], MmaWarpSmem<NT>& sm, int g,
                                             int lane) {
  const int tqr = (lane >> 1) & 3;                 // reader thread-in-group of channels 4*lane ..
  const int sstep = 2 * (lane >> 3) + (lane & 1);  // their k-step
#pragma unroll
  for (int r = 0; r < 4 * NT; ++r) {
    if (r >= g) break;
    // reader row R of head r's hi (and lo) column, chunk swizzle ((R >> 1) & 3) << 4
    unsigned char* dhi;
    unsigned char* dlo;
    int xr, xl;
    if constexpr (head_cols<NT>()) {
      const int R = 4 * r + tqr;
      dhi = reinterpret_cast<unsigned char*>(&sm.bq[0][R][0]);
      dlo = reinterpret_cast<unsigned char*>(&sm.bq[1][R][0]);
      xr = xl = ((R >> 1) & 3) << 4;
    } else {
      dhi = reinterpret_cast<unsigned char*>(&sm.bq[r >> 2][8 * (r & 3) + tqr][0]);
      dlo = dhi + 4 * 64;
      xr = ((tqr >> 1) & 1) << 4;
      xl = xr ^ 32;
    }
    float qv[4];  // channels 4*lane + k of the permuted query
#pragma unroll
    for (int k = 0; k < 4; ++k) qv[k] = qw[r][qb_perm_pos<KBQ>(4 * lane + k)];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int byte = 2 * (4 * sstep + k);
      const __half hi = __float2half_rn(qv[k]);
      const __half lo = __float2half_rn(qv[k] - __half2float(hi));
      *reinterpret_cast<__half*>(dhi + (byte ^ xr)) = hi;
      *reinterpret_cast<__half*>(dlo + (byte ^ xl)) = lo;
    }
  }
}

// One fp16 item for one warp: S = K Q (token rows 0..7 of the m16 tile),
// online softmax into (m_used, lsum), O += V^T P (m16n8k8: k = the 8 tokens).
// O here is the plain-domain accumulator (standard channel order: row gq of
// m-tile mc is channel 16 mc + gq).
template <int NT>
__device__ __forceinline__ void process_f16(const MmaWarpSmem<NT>& sm, const unsigned char* st, int g, int lane,
                                            int kk0, int k1, float (&O)[8][o_tiles<NT>()][4],
                                            float (&m_used)[NT], float (&lsum)[NT]) {
  constexpr bool HC = head_cols<NT>();
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t bq[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const unsigned char* row = reinterpret_cast<const unsigned char*>(&sm.bq[nt][lane][0]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + 16 * (c ^ ((lane >> 1) & 3)));
      bq[nt][4 * c] = u.x; bq[nt][4 * c + 1] = u.y; bq[nt][4 * c + 2] = u.z; bq[nt][4 * c + 3] = u.w;
    }
  }
  // S = K Q: token row gq; rows 8..15 of the tile are empty.  Head columns:
  // S holds the hi chain, S2 the lo chain; otherwise even / odd k-steps.
  float S[NT][4], S2[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int k = 0; k < 4; ++k) S[nt][k] = S2[nt][k] = 0.0f;
  uint4 kw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) kw[i] = *reinterpret_cast<const uint4*>(st + F16Geom::KC + kf16_off(gq, tq + 4 * i));
#pragma unroll
  for (int s_ = 0; s_ < 8; ++s_) {
    const uint4 u = kw[s_ >> 1];
    const uint32_t lo = (s_ & 1) ? u.z : u.x, hi = (s_ & 1) ? u.w : u.y;
    if constexpr (HC) {
      mma16816(S[0], lo, 0u, hi, 0u, bq[0][2 * s_], bq[0][2 * s_ + 1]);
      mma16816(S2[0], lo, 0u, hi, 0u, bq[1][2 * s_], bq[1][2 * s_ + 1]);
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (s_ & 1)
          mma16816(S2[nt], lo, 0u, hi, 0u, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
        else
          mma16816(S[nt], lo, 0u, hi, 0u, bq[nt][2 * s_], bq[nt][2 * s_ + 1]);
      }
    }
  }
  // online softmax over the item's tokens (this thread: token gq, head slot_head(nt))
  const bool tok_ok = kk0 + gq < k1;
  float P[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool live = slot_head<NT>(nt, tq) < g;
    const float z = HC ? S[0][nt] + S2[0][nt] : (S[nt][0] + S2[nt][0]) + (S[nt][1] + S2[nt][1]);
    float zm = tok_ok ? z : -INFINITY;
    zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 4));
    zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 8));
    zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, 16));
    if (!live) zm = -INFINITY;
    if (zm > m_used[nt] + kLazyRescale) {
      const float alpha = ex2(m_used[nt] - zm);
      if constexpr (HC) {
#pragma unroll
        for (int mc = 0; mc < 8; ++mc) {
          O[mc][0][nt] *= alpha;
          O[mc][0][2 + nt] *= alpha;
        }
      } else {
#pragma unroll
        for (int mc = 0; mc < 8; ++mc)
#pragma unroll
          for (int k = 0; k < 4; ++k) O[mc][nt][k] *= alpha;
      }
      lsum[nt] *= alpha;
      m_used[nt] = zm;
    }
    P[nt] = (live && tok_ok) ? ex2(z - m_used[nt]) : 0.0f;
    lsum[nt] += P[nt];
  }
  const uint32_t vbase = smem_u32(st + F16Geom::VC);
  if constexpr (HC) {
    // O += V^T P: B = P of tokens 2tq, 2tq+1 for column (head) gq, held by
    // lanes 4 (2tq + e) + (gq >> 1) in slot gq & 1; hi and lo as two mma
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int src = 4 * (2 * tq + e) + (gq >> 1);
      const float p0 = __shfl_sync(0xffffffffu, P[0], src);
      const float p1 = __shfl_sync(0xffffffffu, P[1], src);
      v[e] = (gq & 1) ? p1 : p0;
    }
    uint32_t bh, bl;
    split_hilo(make_float2(v[0], v[1]), bh, bl);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t a[4];
      ldsm_x4_trans(a[0], a[1], a[2], a[3], vbase + vf16_off(lane & 7, 4 * b + (lane >> 3)));
      mma1688(O[2 * b][0], a[0], a[1], bh);
      mma1688(O[2 * b + 1][0], a[2], a[3], bh);
      mma1688(O[2 * b][0], a[0], a[1], bl);
      mma1688(O[2 * b + 1][0], a[2], a[3], bl);
    }
  } else {
    // O += V^T P: B = P of tokens 2tq, 2tq+1 for column gq (head gq >> 1, hi / lo)
    const float lo_sel = (gq & 1) ? 1.0f : 0.0f;
    const int src0 = 8 * tq + (gq >> 1);  // lane holding token 2tq, head gq >> 1
    uint32_t bp[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float v0 = __shfl_sync(0xffffffffu, P[nt], src0);
      const float v1 = __shfl_sync(0xffffffffu, P[nt], src0 + 4);
      bp[nt] = split_pack(make_float2(v0, v1), lo_sel);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t a[4];
      ldsm_x4_trans(a[0], a[1], a[2], a[3], vbase + vf16_off(lane & 7, 4 * b + (lane >> 3)));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma1688(O[2 * b][nt], a[0], a[1], bp[nt]);
        mma1688(O[2 * b + 1][nt], a[2], a[3], bp[nt]);
      }
    }
  }
}

}  // namespace mma
}  // namespace kvq
