// Prefill attention kernels: the warp-level mma.sync kernel (prefill.cuh; contiguous and paged
// caches, head_dim 64 and 128) and the tcgen05 kernel (prefill_tc.cuh; head_dim 128).
#include "prefill.cuh"
#include "prefill_tc.cuh"

namespace rra {

cudaError_t launch_prefill(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                           cudaStream_t stream) {
  if (a.D == 128)
    return paged ? launch_prefill_t<128, true>(a, k_map, v_map, stream)
                 : launch_prefill_t<128, false>(a, k_map, v_map, stream);
  return paged ? launch_prefill_t<64, true>(a, k_map, v_map, stream)
               : launch_prefill_t<64, false>(a, k_map, v_map, stream);
}

cudaError_t launch_prefill_tc(const DecodeArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                              const CUtensorMap& v_map, bool paged, cudaStream_t stream) {
  return paged ? ptc::launch<true>(a, q_map, k_map, v_map, stream) : ptc::launch<false>(a, q_map, k_map, v_map, stream);
}

}  // namespace rra
