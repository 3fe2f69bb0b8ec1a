// kvq_decode_other.cu -- decode kernel instantiations for 3-bit non-uniform
// K and V, and for the plain fp16 cache; plus the dispatch over K bits.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_k2(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t launch_decode_k4(const DecodeParams& p, cudaStream_t st, int* occ);
cudaError_t launch_decode_k8(const DecodeParams& p, cudaStream_t st, int* occ);
template <int KB, int VB>
static cudaError_t by_gq(const DecodeParams& p, cudaStream_t st, int* occ) {
  switch (p.geo.g <= 1 ? 1 : p.geo.g <= 2 ? 2 : p.geo.g <= 4 ? 4 : 8) {
    case 1: return launch_decode_t<KB, VB, 1>(p, st, occ);
    case 2: return launch_decode_t<KB, VB, 2>(p, st, occ);
    case 4: return launch_decode_t<KB, VB, 4>(p, st, occ);
    default: return launch_decode_t<KB, VB, 8>(p, st, occ);
  }
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st, int* occ) {
  if (p.geo.fp16_mode) return by_gq<16, 16>(p, st, occ);
  switch (p.geo.kb) {
    case 2: return launch_decode_k2(p, st, occ);
    case 3: return by_gq<3, 3>(p, st, occ);
    case 4: return launch_decode_k4(p, st, occ);
    case 8: return launch_decode_k8(p, st, occ);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
