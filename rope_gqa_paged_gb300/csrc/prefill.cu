// Prefill attention kernels (prefill.cuh): contiguous and paged caches, head_dim 64 and 128.
#include "prefill.cuh"

namespace rra {

cudaError_t launch_prefill(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                           cudaStream_t stream) {
  if (a.D == 128)
    return paged ? launch_prefill_t<128, true>(a, k_map, v_map, stream)
                 : launch_prefill_t<128, false>(a, k_map, v_map, stream);
  return paged ? launch_prefill_t<64, true>(a, k_map, v_map, stream)
               : launch_prefill_t<64, false>(a, k_map, v_map, stream);
}

}  // namespace rra
