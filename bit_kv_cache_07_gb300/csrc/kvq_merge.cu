// kvq_merge.cu -- log-sum-exp merge of attention results over disjoint parts
// of one context (context-parallel decode: one part per GPU shard).
//
// KVQuant summary, abstract and main results: a 10M-token context served on
// an 8-GPU system.  Each shard's decode returns its normalised output o_r and
// lse_r = log sum_{t in shard} exp(logit_t); the attention over the whole
// context is
//   lse = log sum_r exp(lse_r),   o = sum_r exp(lse_r - lse) o_r,
// the same merge the decode kernels apply to their own split partials.
// One warp per output row (lane l owns channels 4l..4l+3); fp32 arithmetic.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kMergeWarps = 8;  // rows per CTA

__global__ void __launch_bounds__(32 * kMergeWarps)
    merge_attn_kernel(int n_parts, long long rows, const uint16_t* __restrict__ outs, const float* __restrict__ lses,
                      uint16_t* __restrict__ out, float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  constexpr float kLog2e = 1.4426950408889634f;
  // the largest part lse (lanes stride over the parts)
  float M = -INFINITY;
  for (int r = lane; r < n_parts; r += 32) M = fmaxf(M, __ldg(&lses[(size_t)r * rows + row]));
  M = warp_max(M);
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, L = 0.0f;
  if (M != -INFINITY) {
    for (int r = 0; r < n_parts; ++r) {
      const float lr = __ldg(&lses[(size_t)r * rows + row]);
      if (lr == -INFINITY) continue;  // an empty part
      const float w = exp2f((lr - M) * kLog2e);
      L += w;
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(outs + ((size_t)r * rows + row) * kHeadDim) + lane);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      acc[0] = fmaf(w, a.x, acc[0]);
      acc[1] = fmaf(w, a.y, acc[1]);
      acc[2] = fmaf(w, b.x, acc[2]);
      acc[3] = fmaf(w, b.y, acc[3]);
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  const __half2 h0 = __floats2half2_rn(acc[0] * inv, acc[1] * inv), h1 = __floats2half2_rn(acc[2] * inv, acc[3] * inv);
  uint2 st;
  st.x = *reinterpret_cast<const uint32_t*>(&h0);
  st.y = *reinterpret_cast<const uint32_t*>(&h1);
  reinterpret_cast<uint2*>(out + (size_t)row * kHeadDim)[lane] = st;
  if (lse_out && lane == 0) lse_out[row] = L > 0.0f ? M + logf(L) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge_attn(int n_parts, long long rows, const uint16_t* outs, const float* lses, uint16_t* out,
                              float* lse_out, cudaStream_t st) {
  const long long blocks = (rows + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  merge_attn_kernel<<<(unsigned)blocks, 32 * kMergeWarps, 0, st>>>(n_parts, rows, outs, lses, out, lse_out);
  return cudaGetLastError();
}

}  // namespace kvq
