// Instantiations of the tcgen05 decode kernel (query groups of 16 to 128 heads, head_dim 128).
#include "decode_tc.cuh"

namespace rra {

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                             bool fused, cudaStream_t stream) {
  if (paged)
    return fused ? dtc::launch_t<true, true>(a, k_map, v_map, stream) : dtc::launch_t<true, false>(a, k_map, v_map, stream);
  return fused ? dtc::launch_t<false, true>(a, k_map, v_map, stream) : dtc::launch_t<false, false>(a, k_map, v_map, stream);
}

}  // namespace rra
