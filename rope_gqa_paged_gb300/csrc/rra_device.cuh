// Device primitives shared by the decode-step kernels (sm_103a):
// mbarrier waits with a time limit, 1-D bulk copies and 4-D tensor (TMA) copies
// from global memory into shared memory, and bf16 / fp32 16-byte unpacking.
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rra.h"

namespace rra {

// Budget of one pipeline wait, in SM clock cycles (about a second at 2 GHz).
constexpr long long kWaitBudgetCycles = 2000000000LL;

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete; false once the budget is spent.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitBudgetCycles) return false;
  }
  return true;
}

// Contiguous global -> shared copy completing on `bar` (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// 4-D tiled tensor copy (box fixed by the tensor map) completing on `bar`.
__device__ __forceinline__ void tma_g2s_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                           uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

// L2 prefetch of one tensor-map box (no shared memory, no barrier). The box is bounds-checked
// by the tensor map like a load; callers still pass coordinates clamped into the tensor.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Programmatic dependent launch. The decode kernels are launched with programmatic stream
// serialisation: each lets the next kernel in the stream be scheduled as soon as it starts,
// and waits for the previous kernel to complete (with its memory visible) before it reads any
// input. Without that launch attribute both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns whether `v` held in every participating thread.
__device__ __forceinline__ bool named_barrier_and(int id, int threads, bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 q, %3, 0;\n\t"
      "bar.red.and.pred p, %1, %2, q;\n\t"
      "selp.s32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(threads), "r"(v ? 1 : 0)
      : "memory");
  return r != 0;
}

// Launches kern<<<grid, block, smem, stream>>>(args...) with programmatic stream serialisation
// (the kernel may start before the previous kernel in the stream ends; it calls pdl_wait()
// before reading anything that kernel may write).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Sets the dynamic shared-memory limit of a kernel once per device.
template <typename Kernel>
inline cudaError_t ensure_smem(Kernel k, int bytes, int* done_per_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done_per_device[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done_per_device[dev] = 1;
  return e;
}

// a*(ch + cl) - b*(sh + sl) to ~1 float32 ulp of the result, where (ch, cl) and (sh, sl)
// are a cosine and a sine split into float32 hi + lo parts. The products a*ch and b*sh
// are kept exactly as p + e with e = fma(x, y, -p) (Dekker's product using the FMA), so
// the difference keeps full relative accuracy when the two products cancel. The explicit
// _rn intrinsics stop the compiler from contracting the products into other operations.
__device__ __forceinline__ float rotate_diff(float a, float b, float ch, float cl, float sh, float sl) {
  const float p = __fmul_rn(a, ch);
  const float ep = __fmaf_rn(a, ch, -p);
  const float q = __fmul_rn(b, sh);
  const float eq = __fmaf_rn(b, sh, -q);
  const float small = __fadd_rn(__fsub_rn(ep, eq), __fsub_rn(__fmul_rn(a, cl), __fmul_rn(b, sl)));
  return __fadd_rn(__fsub_rn(p, q), small);
}

// ---- element types --------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerChunk = 8;  // elements in 16 bytes
  __device__ __forceinline__ static void unpack(const uint4& r, float (&x)[8]) {
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xffff0000u);
    x[4] = __uint_as_float(r.z << 16);
    x[5] = __uint_as_float(r.z & 0xffff0000u);
    x[6] = __uint_as_float(r.w << 16);
    x[7] = __uint_as_float(r.w & 0xffff0000u);
  }
  __device__ __forceinline__ static float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
  // float64 -> bf16 in one rounding (nearest even), no detour through float32.
  __device__ __forceinline__ static void store_f64(__nv_bfloat16* p, double v) { *p = __double2bfloat16(v); }
};

template <>
struct Elem<float> {
  static constexpr int kPerChunk = 4;
  __device__ __forceinline__ static void unpack(const uint4& r, float (&x)[4]) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  }
  __device__ __forceinline__ static float load(const float* p) { return *p; }
  __device__ __forceinline__ static void store(float* p, float v) { *p = v; }
  __device__ __forceinline__ static void store_f64(float* p, double v) { *p = static_cast<float>(v); }
};

// Symmetric INT8 code of x at scale s ("Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践"
// §4.3, per-head calibrated INT8): clamp(round_half_even(x / s), -127, 127), the quotient an
// IEEE float32 division (nearest even). A NaN input gives -127.
__device__ __forceinline__ int8_t quantize_code(float x, float s) {
  const float r = fminf(fmaxf(__fdiv_rn(x, s), -127.f), 127.f);
  return static_cast<int8_t>(__float2int_rn(r));
}

// 4-bit code of x at scale s: clamp(round_half_even(x / s), -7, 7) (float32 quotient).
__device__ __forceinline__ int quantize_code4(float x, float s) {
  const float r = fminf(fmaxf(__fdiv_rn(x, s), -7.f), 7.f);
  return __float2int_rn(r);
}

// Two 4-bit two's complement codes in one byte: `lo` in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint8_t pack_nibbles(int lo, int hi) {
  return static_cast<uint8_t>((lo & 0xf) | ((hi & 0xf) << 4));
}

}  // namespace rra
