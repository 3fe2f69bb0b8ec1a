// kvq_internal.cuh -- geometry, parameter blocks and small device helpers
// shared by the host layer (kvq_host.cu) and the kernels (kvq_append.cu,
// kvq_decode*.cu).  Not part of the public ABI (that is include/kvq.h).
#pragma once

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
constexpr int kThreads = 128;      // 4 warps per CTA in every kernel

// Geometry derived once on the host from a kvq_config.
struct Geometry {
  int B, Hq, Hkv, g, NS, d;
  int kb, vb, gk, gv, nvg;
  int S, R, ring, qcap, gcap;
  int krow, vrow;
  int hadamard, pre_rope, nout, fp16_mode;
  float rope_theta;
};

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
};

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
};

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
  int fp16_tokens_per_split;
  float q_scale;          // softmax_scale * log2(e)
  float hadamard_c;       // fp32(1/sqrt(d))
  float k_lut_off[8];     // L_i - L_0 (fp32)
  float v_lut_off[8];
  double theta[kHeadDim / 2];  // RoPE frequencies rope_theta^(-2i/d), fp64
};

// ------------------------------------------------------------ host hooks
cudaError_t launch_append_quantize(const AppendParams& p, int n_groups, cudaStream_t st);
cudaError_t launch_append_window(const AppendParams& p, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st);

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
