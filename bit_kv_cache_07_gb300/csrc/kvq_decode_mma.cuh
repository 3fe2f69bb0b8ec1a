// kvq_decode_mma.cuh -- tensor-core version of the quantized decode splits
// (uniform K per channel, uniform V per token; no RoPE).
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

template <int NT>
struct MmaSmem {
  alignas(16) float q[8 * NT][kHeadDim];             // scaled q, heads >= g zero
  alignas(16) uint16_t bq[4][NT][32][40];            // per warp: Q' fragments per lane (32 used + pad)
  alignas(16) float bias[4][8];                      // per warp: q . kmin per head
  alignas(16) float stage_o[4][8 * NT][kHeadDim];    // per warp O for the merge (reused)
  alignas(16) float ml[4][8 * NT][2];
  alignas(16) float comb_ml[8 * NT][2];
  int is_last;
};

}  // namespace mma
}  // namespace kvq
