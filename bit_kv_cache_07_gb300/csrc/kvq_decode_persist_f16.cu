// kvq_decode_persist_f16.cu -- the persistent decode's host side: which
// configurations it serves, its schedule and workspace, and the dispatch;
// plus its fp16-cache instantiations.
#include "kvq_decode_persist.cuh"

namespace kvq {

cudaError_t persist_k2(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t persist_k4(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t persist_k8(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t persist_iq_k2(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t persist_iq_k4(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t persist_iq_k8(const DecodeParams& p, cudaStream_t st, int* occ);

static cudaError_t persist_f16(const DecodeParams& p, cudaStream_t st, int* occ) {
  return persist::dispatch_gt<16, 16>(p, st, occ);
}

static cudaError_t dispatch(const DecodeParams& p, cudaStream_t st, int* occ) {
  if (p.geo.fp16_mode) return persist_f16(p, st, occ);
  if (p.geo.gkc) {  // InnerQ keys
    switch (p.geo.kb) {
      case 2: return persist_iq_k2(p, st, occ);
      case 4: return persist_iq_k4(p, st, occ);
      case 8: return persist_iq_k8(p, st, occ);
    }
    return cudaErrorInvalidValue;
  }
  switch (p.geo.kb) {
    case 2: return persist_k2(p, st, occ);
    case 4: return persist_k4(p, st, occ);
    case 8: return persist_k8(p, st, occ);
  }
  return cudaErrorInvalidValue;
}

// Uniform K and V (2/4/8 bits) with 64-channel V groups and no RoPE, or a
// plain fp16 cache without RoPE.  Everything else uses the split kernel.
bool persist_eligible(const Geometry& g) {
  if (g.pre_rope || g.g > kMaxGQA) return false;
  if (g.fp16_mode) return true;
  if (g.kb == 3 || g.vb == 3) return false;
  if ((uint64_t)g.NS * (uint64_t)g.qcap >= (1ull << 31)) return false;  // 32-bit row index in the kernel
  return g.gv == 64;
}

cudaError_t plan_persist(DecodeParams& p, uint64_t* ws_need) {
  const Geometry& G = p.geo;
  p.ng = G.fp16_mode ? 0 : p.Nq / kGroupTokens;
  p.nt = (p.S_eff + p.W + mma::kF16Tokens - 1) / mma::kF16Tokens;
  p.n_items = p.ng + p.nt;
  // item weights the warps' ranges are cut by.  fp16 cache: an item's bytes.
  // Quantized cache: every item weighs the bytes of a quantized group (its
  // codes, K scales and V scales), the fp16 items of the sinks and window
  // included: measured per warp, an 8-token fp16 item takes about as long as
  // a 32-token group at any bit width (both bound by per-item work), and with
  // byte weights the warps holding a stream's fp16 items (and its end)
  // finished last: the 32k mixed-pair step took 2.7 % longer
  const long long wgroup = (long long)kGroupTokens * (G.krow + G.vrow) +
                           (G.gkc ? kGroupTokens * G.nkg * 4 : kHeadDim * 4) + kGroupTokens * G.nvg * 4;
  // (with 5-8 query heads per KV head an fp16 item weighs 5/4 of a group:
  // its 8 tokens carry every head's scores and products on the tensor cores
  // at half-filled tiles, and those warps still finished ~4 % late)
  p.wq = G.fp16_mode ? 1 : wgroup;
  p.wt = G.fp16_mode ? (long long)mma::kF16Tokens * kHeadDim * 2 * 2 : (G.g > 4 ? wgroup * 5 / 4 : wgroup);
  p.wstream = (long long)p.ng * p.wq + (long long)p.nt * p.wt;
  p.wtot = (long long)G.NS * p.wstream;
  long long items = (long long)G.NS * p.n_items;
  bool any_groups = p.ng > 0;
  if (p.ragged) plan_rows(p, &items, &any_groups);
  int sms = 0, occ = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  if (G.sm_budget > 0 && G.sm_budget < sms) sms = G.sm_budget;  // a share of the GPU
  e = dispatch(p, nullptr, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  long long nw = (long long)sms * occ;  // occ: resident warps per SM
  if (nw > items) nw = items;
  if (nw > (long long)kMaxQSplits * G.NS) nw = (long long)kMaxQSplits * G.NS;
  // every warp's weight range must hold at least one item start, so that the
  // warps counted for a stream are exactly the ones that work on it
  const long long wmax = any_groups && p.wq > p.wt ? p.wq : p.wt;
  if (nw > p.wtot / wmax) nw = p.wtot / wmax;
  if (nw < 1) nw = 1;
  p.nwarps = (int)nw;
  // the schedule's dividends stay below (wtot + 1) (nwarps + 1)
  if ((unsigned __int128)(p.wtot + 1) * (unsigned __int128)(p.nwarps + 1) >= (unsigned __int128)kFastDivLimit)
    return cudaErrorInvalidValue;
  p.fd_n_items = make_fastdiv(p.n_items);
  p.fd_wq = make_fastdiv(p.wq);
  p.fd_wt = make_fastdiv(p.wt);
  p.fd_wstream = make_fastdiv(p.wstream);
  p.fd_wtot = make_fastdiv(p.wtot);
  p.fd_nwarps = make_fastdiv(p.nwarps);
  const uint64_t slots = (uint64_t)p.nwarps + G.NS;
  const uint64_t cnt = ((uint64_t)G.NS * 4 + 255) / 256 * 256;
  const uint64_t ml = (slots * G.g * 2 * 4 + 255) / 256 * 256;
  *ws_need = cnt + ml + slots * G.g * kHeadDim * 4;
  return cudaSuccess;
}

cudaError_t launch_decode_persist(const DecodeParams& p, cudaStream_t st) { return dispatch(p, st, nullptr); }

}  // namespace kvq
