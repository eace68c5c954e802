// INT8 / INT4 KV-cache decode kernels (decode_q8.cuh): contiguous and paged, attention only or
// the whole fused step; INT8 for head_dim 64 and 128, INT4 for head_dim 128.
#include "decode_q8.cuh"

namespace rra {

cudaError_t launch_decode_q8(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                             const CUtensorMap& kw_map, const CUtensorMap& vw_map, bool paged, bool fused,
                             cudaStream_t stream) {
  if (a.code_bits == 4) {
    if (paged)
      return fused ? launch_decode_q8_t<128, 4, true, true>(a, k_map, v_map, kw_map, vw_map, stream)
                   : launch_decode_q8_t<128, 4, true, false>(a, k_map, v_map, kw_map, vw_map, stream);
    return fused ? launch_decode_q8_t<128, 4, false, true>(a, k_map, v_map, kw_map, vw_map, stream)
                 : launch_decode_q8_t<128, 4, false, false>(a, k_map, v_map, kw_map, vw_map, stream);
  }
  if (a.D == 128) {
    if (paged)
      return fused ? launch_decode_q8_t<128, 8, true, true>(a, k_map, v_map, kw_map, vw_map, stream)
                   : launch_decode_q8_t<128, 8, true, false>(a, k_map, v_map, kw_map, vw_map, stream);
    return fused ? launch_decode_q8_t<128, 8, false, true>(a, k_map, v_map, kw_map, vw_map, stream)
                 : launch_decode_q8_t<128, 8, false, false>(a, k_map, v_map, kw_map, vw_map, stream);
  }
  if (paged)
    return fused ? launch_decode_q8_t<64, 8, true, true>(a, k_map, v_map, kw_map, vw_map, stream)
                 : launch_decode_q8_t<64, 8, true, false>(a, k_map, v_map, kw_map, vw_map, stream);
  return fused ? launch_decode_q8_t<64, 8, false, true>(a, k_map, v_map, kw_map, vw_map, stream)
               : launch_decode_q8_t<64, 8, false, false>(a, k_map, v_map, kw_map, vw_map, stream);
}

}  // namespace rra
