// Multi-query decode (speculative verify) kernels (verify.cuh): contiguous and paged caches,
// head_dim 64 and 128, attention only or the whole step (RoPE + append + attention).
#include "verify.cuh"

namespace rra {

cudaError_t launch_decode_verify(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                                 bool fused, cudaStream_t stream) {
  if (fused) {
    if (a.D == 128)
      return paged ? launch_decode_verify_t<128, true, true>(a, k_map, v_map, stream)
                   : launch_decode_verify_t<128, false, true>(a, k_map, v_map, stream);
    return paged ? launch_decode_verify_t<64, true, true>(a, k_map, v_map, stream)
                 : launch_decode_verify_t<64, false, true>(a, k_map, v_map, stream);
  }
  if (a.D == 128)
    return paged ? launch_decode_verify_t<128, true, false>(a, k_map, v_map, stream)
                 : launch_decode_verify_t<128, false, false>(a, k_map, v_map, stream);
  return paged ? launch_decode_verify_t<64, true, false>(a, k_map, v_map, stream)
               : launch_decode_verify_t<64, false, false>(a, k_map, v_map, stream);
}

}  // namespace rra
