// rra_decode_attn_paged_noalloc: the paged decode for callers that must not allocate
// device memory. Some callers cannot call cudaMalloc (or any allocator) at the point
// where they run a decode step: code that owns no allocator handle because a host
// framework manages all device memory, loops that forbid allocation after start-up
// (allocation can block, fail, or fragment the pool mid-run), and code paths where the
// caller has promised not to allocate. For them the split-K scratch (per-split partial
// outputs plus running max and sum, and the arrival counters of the split merge) lives in
// one file-scope device array instead of a caller-provided workspace.
//
// Properties of that array:
//   * kStaticScratchBytes (16 MiB) on every GPU that loads this library, held until the
//     process exits. Its first kCounterBytes (1 MiB) hold the arrival counters, at the same
//     place for every call whatever its shape; the rest (15 MiB) holds the partials. A step
//     whose partials or counters need more (for its effective split count) is rejected with
//     RRA_EWORKSPACE before anything is enqueued.
//   * The counters must be zero when the kernel starts. Every call clears the counters it
//     will use with one cudaMemsetAsync on its own stream before its launch (a memset of
//     memory the library already holds, not an allocation), so a call does not depend on
//     what an earlier call of another shape, or one that gave up on a device-side wait,
//     left behind.
//   * Shared by every call on a device: two calls whose kernels overlap on the GPU (two
//     streams, or two host threads) race on it and return wrong results. Issue them in
//     one stream, or serialise them.
//   * Its device address is looked up once per device, on the first call made while
//     that device is current (cudaGetSymbolAddress); make that first call before any
//     stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rra.h"
#include "rra_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr size_t kCounterBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_split_scratch[kStaticScratchBytes];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_split_scratch on the current device (looked up once per device).
int scratch_on_current_device(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    rra::record_cuda_error(e, "cudaGetDevice");
    return RRA_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return RRA_ERANGE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) {
      rra::record_cuda_error(e, "cudaGetSymbolAddress(split scratch)");
      return RRA_ECUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return RRA_OK;
}

}  // namespace

extern "C" {

size_t rra_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }

int rra_decode_attn_paged_noalloc(const void* q_rot, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                                  int block_size, int num_blocks, void* out, int B, int Hq, int Hkv, int D,
                                  float scale, int num_splits, rra_dtype dt, int32_t* err_flag, void* stream) {
  if (block_size < 1 || max_blocks_per_seq < 1) return RRA_EINVAL;
  const int splits = rra_decode_num_splits(B, Hq, Hkv, D, int64_t(max_blocks_per_seq) * block_size, block_size,
                                           num_splits, dt);
  if (splits < 0) return splits;
  const size_t partials = rra::decode_partial_bytes(B, Hq, D, splits);
  const size_t counter_bytes = rra::decode_counter_ints(B, Hq, splits) * sizeof(int);
  if (partials > kStaticScratchBytes - kCounterBytes || counter_bytes > kCounterBytes) return RRA_EWORKSPACE;
  unsigned char* scratch = nullptr;
  int* counters = nullptr;
  if (partials > 0) {
    void* base = nullptr;
    const int st = scratch_on_current_device(&base);
    if (st != RRA_OK) return st;
    scratch = static_cast<unsigned char*>(base);
    counters = reinterpret_cast<int*>(scratch);
    const cudaError_t e = cudaMemsetAsync(counters, 0, counter_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      rra::record_cuda_error(e, "cudaMemsetAsync(split counters)");
      return RRA_ECUDA;
    }
  }
  return rra::decode_attn_paged_ext(q_rot, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, block_size,
                                    num_blocks, out, B, Hq, Hkv, D, scale, num_splits,
                                    scratch != nullptr ? scratch + kCounterBytes : nullptr,
                                    scratch != nullptr ? kStaticScratchBytes - kCounterBytes : 0, counters, dt,
                                    err_flag, stream);
}

}  // extern "C"
