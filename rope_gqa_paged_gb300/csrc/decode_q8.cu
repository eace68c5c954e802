// INT8 KV-cache decode kernels (decode_q8.cuh): contiguous and paged, attention only or the
// whole fused step, head_dim 64 and 128.
#include "decode_q8.cuh"

namespace rra {

cudaError_t launch_decode_q8(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                             const CUtensorMap& kw_map, const CUtensorMap& vw_map, bool paged, bool fused,
                             cudaStream_t stream) {
  if (a.D == 128) {
    if (paged)
      return fused ? launch_decode_q8_t<128, true, true>(a, k_map, v_map, kw_map, vw_map, stream)
                   : launch_decode_q8_t<128, true, false>(a, k_map, v_map, kw_map, vw_map, stream);
    return fused ? launch_decode_q8_t<128, false, true>(a, k_map, v_map, kw_map, vw_map, stream)
                 : launch_decode_q8_t<128, false, false>(a, k_map, v_map, kw_map, vw_map, stream);
  }
  if (paged)
    return fused ? launch_decode_q8_t<64, true, true>(a, k_map, v_map, kw_map, vw_map, stream)
                 : launch_decode_q8_t<64, true, false>(a, k_map, v_map, kw_map, vw_map, stream);
  return fused ? launch_decode_q8_t<64, false, true>(a, k_map, v_map, kw_map, vw_map, stream)
               : launch_decode_q8_t<64, false, false>(a, k_map, v_map, kw_map, vw_map, stream);
}

}  // namespace rra
