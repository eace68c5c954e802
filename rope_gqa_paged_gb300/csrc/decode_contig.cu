// Instantiations of the decode kernels for the contiguous cache, and the split merge.
#include "decode_kernels.cuh"
#include "decode_mma.cuh"

namespace rra {

cudaError_t launch_decode_contig(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                 rra_dtype dt, bool use_mma, cudaStream_t stream) {
  if (use_mma) return launch_decode_mma<false>(a, k_map, v_map, a.hpc, stream);
  return launch_decode_any<false>(a, k_map, v_map, dt, a.hpc, stream);
}

cudaError_t launch_decode_reduce(const DecodeArgs& a, rra_dtype dt, cudaStream_t stream) {
  const int rows = a.B * a.Hq;
  const dim3 grid((rows + kReduceWarps - 1) / kReduceWarps);
  const int threads = kReduceWarps * 32;
  if (dt == RRA_BF16) {
    if (a.D == 128)
      decode_reduce_kernel<__nv_bfloat16, 128><<<grid, threads, 0, stream>>>(a);
    else
      decode_reduce_kernel<__nv_bfloat16, 64><<<grid, threads, 0, stream>>>(a);
  } else {
    if (a.D == 128)
      decode_reduce_kernel<float, 128><<<grid, threads, 0, stream>>>(a);
    else
      decode_reduce_kernel<float, 64><<<grid, threads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace rra
