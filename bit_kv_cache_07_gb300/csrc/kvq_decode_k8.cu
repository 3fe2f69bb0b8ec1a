// kvq_decode_k8.cu -- decode kernel instantiations for 8-bit uniform K
// (V 2, 4 or 8 bits; 1, 2, 4 or 8 query heads per KV head).
#include "kvq_decode.cuh"

namespace kvq {

template <int VB>
static cudaError_t by_gq(const DecodeParams& p, cudaStream_t st, int* occ) {
  switch (p.geo.g <= 1 ? 1 : p.geo.g <= 2 ? 2 : p.geo.g <= 4 ? 4 : 8) {
    case 1: return launch_decode_t<8, VB, 1>(p, st, occ);
    case 2: return launch_decode_t<8, VB, 2>(p, st, occ);
    case 4: return launch_decode_t<8, VB, 4>(p, st, occ);
    default: return launch_decode_t<8, VB, 8>(p, st, occ);
  }
}

cudaError_t launch_decode_k8(const DecodeParams& p, cudaStream_t st, int* occ) {
  switch (p.geo.vb) {
    case 2: return by_gq<2>(p, st, occ);
    case 4: return by_gq<4>(p, st, occ);
    case 8: return by_gq<8>(p, st, occ);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
