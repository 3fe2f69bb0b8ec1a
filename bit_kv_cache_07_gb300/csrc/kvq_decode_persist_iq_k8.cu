// kvq_decode_persist_iq_k8.cu -- persistent tensor-core decode instantiations
// for InnerQ keys (per-token 64-channel groups) at 8 bits (V 2, 4 or 8 bits;
// 1, 2, 4 or 8 query heads per KV head).
#include "kvq_decode_persist.cuh"

namespace kvq {
cudaError_t persist_iq_k8(const DecodeParams& p, cudaStream_t st, int* occ) {
  return persist::dispatch_vb<8, true>(p, st, occ);
}
}  // namespace kvq
