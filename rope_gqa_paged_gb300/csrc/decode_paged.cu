// Instantiations of the decode kernels for the paged (block-table) cache.
#include "decode_kernels.cuh"
#include "decode_mma.cuh"

namespace rra {

cudaError_t launch_decode_paged(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                rra_dtype dt, bool use_mma, cudaStream_t stream) {
  if (use_mma) return launch_decode_mma<true>(a, k_map, v_map, a.hpc, stream);
  return launch_decode_any<true>(a, k_map, v_map, dt, a.hpc, stream);
}

cudaError_t launch_decode_step_paged(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                   cudaStream_t stream) {
  return launch_decode_mma<true, true>(a, k_map, v_map, a.hpc, stream);
}

}  // namespace rra
