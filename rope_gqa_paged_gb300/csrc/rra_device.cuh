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

// ---- RoPE angles in float32 arithmetic ------------------------------------------------------
// ("Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §3: token m rotates pair i by m·θ_i.)
// The angle is carried in turns: φ_i = θ_i / 2π as a 96-bit binary fraction, made on the host
// from the float64 θ_i by exact integer arithmetic, so m·φ_i mod 1 takes three 32-bit integer
// multiplications. The fraction is centred on its nearest quarter turn k/4; the remainder r
// (|r| <= 1/8 turn) becomes u = 2π·r as a float-float pair (hi + lo), and sin u, cos u are their
// Taylor series at 0, the leading terms in float-float arithmetic (error-free products by fma,
// Dekker; error-free sums, Knuth), the small tail in float32. sin and cos of the angle follow
// from k by a swap and signs. Each comes out as float32 hi + lo, |hi + lo - exact| below ~2^-44:
// the whole evaluation is float32 / integer work (the float64 pipe of the part is narrow).

struct FF {  // hi + lo, |lo| <= ulp(hi) / 2
  float hi, lo;
};
__host__ __device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {  // requires |a| >= |b|
  const float s = a + b;
  return {s, b - (s - a)};
}
__host__ __device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__host__ __device__ __forceinline__ FF ff_mul(FF x, FF y) {
  const float p = x.hi * y.hi;
  float e = fmaf(x.hi, y.hi, -p);  // the rounding error of p, exactly
  e = fmaf(x.hi, y.lo, e);
  e = fmaf(x.lo, y.hi, e);
  return ff_fast_two_sum(p, e);
}
__host__ __device__ __forceinline__ FF ff_mul_f(FF x, float y) {
  const float p = x.hi * y;
  float e = fmaf(x.hi, y, -p);
  e = fmaf(x.lo, y, e);
  return ff_fast_two_sum(p, e);
}
__host__ __device__ __forceinline__ FF ff_add(FF x, FF y) {
  const FF s = ff_two_sum(x.hi, y.hi);
  return ff_fast_two_sum(s.hi, s.lo + (x.lo + y.lo));
}
__host__ __device__ constexpr float ff_hi_of(double x) { return static_cast<float>(x); }
__host__ __device__ constexpr float ff_lo_of(double x) {
  return static_cast<float>(x - static_cast<double>(static_cast<float>(x)));
}
// float-float constants, split from float64 values at compile time
constexpr double kRopeTwoPi = 6.283185307179586476925286766559;
constexpr double kInvFact2 = 1.0 / 2.0, kInvFact3 = 1.0 / 6.0, kInvFact4 = 1.0 / 24.0, kInvFact5 = 1.0 / 120.0,
                 kInvFact6 = 1.0 / 720.0, kInvFact7 = 1.0 / 5040.0, kInvFact8 = 1.0 / 40320.0;

// cos and sin of 2π·(pos·φ mod 1), φ = (phi[2]·2^64 + phi[1]·2^32 + phi[0]) / 2^96, pos >= 0:
// cos = ch + cl, sin = sh + sl. Host-callable too (the same float32 operations, for tests).
__host__ __device__ __forceinline__ void rope_cos_sin(int pos, const uint32_t* phi, float& ch, float& cl, float& sh,
                                             float& sl) {
  const uint32_t m = static_cast<uint32_t>(pos);
  const uint64_t t0 = static_cast<uint64_t>(m) * phi[0];
  const uint64_t t1 = static_cast<uint64_t>(m) * phi[1] + (t0 >> 32);
  const uint32_t w2 = m * phi[2] + static_cast<uint32_t>(t1 >> 32);
  const uint64_t f = (static_cast<uint64_t>(w2) << 32) | static_cast<uint32_t>(t1);  // turns, units of 2^-64
  const uint32_t k = static_cast<uint32_t>((f + (1ull << 61)) >> 62);              // nearest quarter (4 -> 0)
  const int64_t r = static_cast<int64_t>(f - (static_cast<uint64_t>(k) << 62));     // |r| <= 2^61
  // r as hi + lo: 2^40 a + 2^16 b + c with a (signed, < 2^21), b (24 bits) and c (16 bits) exact floats
  const float ra = static_cast<float>(static_cast<int32_t>(r >> 40));
  const float rb = static_cast<float>(static_cast<uint32_t>(r >> 16) & 0xffffffu);
  const float rc = static_cast<float>(static_cast<uint32_t>(r) & 0xffffu);
  FF x = ff_two_sum(ra * 0x1p40f, rb * 0x1p16f);
  x = ff_two_sum(x.hi, x.lo + rc);
  x.hi *= 0x1p-64f;
  x.lo *= 0x1p-64f;
  const FF u = ff_mul(x, FF{ff_hi_of(kRopeTwoPi), ff_lo_of(kRopeTwoPi)});  // radians, |u| <= π/4
  const FF v = ff_mul(u, u);
  // sin u = u + u·v·(-1/3! + v/5! - v²/7! + v³·t), t = 1/9! - v/11! + v²/13! - v³/15! in float32
  float t = fmaf(v.hi, -1.f / 1307674368000.f, 1.f / 6227020800.f);
  t = fmaf(v.hi, t, -1.f / 39916800.f);
  t = fmaf(v.hi, t, 1.f / 362880.f);
  FF s = ff_add(FF{-ff_hi_of(kInvFact7), -ff_lo_of(kInvFact7)}, ff_mul_f(v, t));
  s = ff_add(FF{ff_hi_of(kInvFact5), ff_lo_of(kInvFact5)}, ff_mul(v, s));
  s = ff_add(FF{-ff_hi_of(kInvFact3), -ff_lo_of(kInvFact3)}, ff_mul(v, s));
  const FF sn = ff_add(u, ff_mul(ff_mul(u, v), s));
  // cos u = 1 + v·(-1/2! + v/4! - v²/6! + v³/8! + v⁴·t), t = -1/10! + v/12! - v²/14! + v³/16! in float32
  t = fmaf(v.hi, 1.f / 20922789888000.f, -1.f / 87178291200.f);
  t = fmaf(v.hi, t, 1.f / 479001600.f);
  t = fmaf(v.hi, t, -1.f / 3628800.f);
  FF c = ff_add(FF{ff_hi_of(kInvFact8), ff_lo_of(kInvFact8)}, ff_mul_f(v, t));
  c = ff_add(FF{-ff_hi_of(kInvFact6), -ff_lo_of(kInvFact6)}, ff_mul(v, c));
  c = ff_add(FF{ff_hi_of(kInvFact4), ff_lo_of(kInvFact4)}, ff_mul(v, c));
  c = ff_add(FF{-ff_hi_of(kInvFact2), 0.f}, ff_mul(v, c));
  const FF cn = ff_add(FF{1.f, 0.f}, ff_mul(v, c));
  // angle = k·π/2 + u
  const bool odd = k & 1u;
  const FF co = odd ? sn : cn, so = odd ? cn : sn;
  const bool neg_c = k == 1u || k == 2u, neg_s = k >= 2u;
  ch = neg_c ? -co.hi : co.hi;
  cl = neg_c ? -co.lo : co.lo;
  sh = neg_s ? -so.hi : so.hi;
  sl = neg_s ? -so.lo : so.lo;
}

}  // namespace rra
