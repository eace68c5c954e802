// Fused RoPE + KV-cache append for the new token of every sequence.
//
// "Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §3: theta_i = base^(-2(i-1)/d)
// for i = 1..d/2, angle = position * theta_i, q and k rotated pairwise; the cache keeps
// rotated K, so only the new token is rotated. §5.1 b.ii-iii: rotate, then append.
// "4. 自注意力机制推理：单步计算、KV Cache的引入与原理" §4.5: write slot `step` by index.
// "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南" §四: KVCache.update
// (contiguous) and PagedKVCache (block table -> physical block, slot in block).
//
// Grid: (sequence, group of kPairsPerCta frequencies). Each CTA takes the sine and cosine
// of its frequencies once, in float64 (positions reach 131071, where a float32 angle is
// already ~0.004 rad off) and in units of pi (sincospi: exact argument reduction, so no
// slow path for large angles), splits them into float32 hi + lo parts, and rotates that slice
// of every query and key head. The rotation a*c - b*s is computed from error-free
// float32 products (x*y = p + e exactly, with e = fma(x, y, -p): Dekker's product, using
// the FMA) so that it keeps full relative accuracy when the two products cancel; the
// result is then rounded once to the storage type.
#include "rra_device.cuh"
#include "rra_internal.h"

namespace rra {
namespace {

constexpr int kPairsPerCta = 16;
constexpr int kRopeThreads = 128;

// a*(ch + cl) - b*(sh + sl) to ~1 float32 ulp of the result (no contraction: the
// explicit _rn intrinsics keep each product's rounding error where the formula needs it).
__device__ __forceinline__ float rotate_diff(float a, float b, float ch, float cl, float sh, float sl) {
  const float p = __fmul_rn(a, ch);
  const float ep = __fmaf_rn(a, ch, -p);
  const float q = __fmul_rn(b, sh);
  const float eq = __fmaf_rn(b, sh, -q);
  const float small = __fadd_rn(__fsub_rn(ep, eq), __fsub_rn(__fmul_rn(a, cl), __fmul_rn(b, sl)));
  return __fadd_rn(__fsub_rn(p, q), small);
}

template <typename T>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(const RopeArgs a) {
  __shared__ float cs[4][kPairsPerCta];  // cos hi, cos lo, sin hi, sin lo
  const int b = blockIdx.x;
  const int D = a.D, half = a.D / 2;
  const int i0 = blockIdx.y * kPairsPerCta;
  const int np = min(kPairsPerCta, half - i0);
  const int pos = a.positions[b];
  const bool paged = a.block_table != nullptr;
  const long long cap = paged ? (static_cast<long long>(a.max_blocks_per_seq) << a.log2_bs) : a.max_len;
  if (pos < 0 || pos >= cap) {
    if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  if (threadIdx.x < np) {
    double s, c;  // angle / pi = pos * (theta_i / pi): sincospi reduces its argument exactly
    sincospi(static_cast<double>(pos) * a.inv_freq[i0 + threadIdx.x], &s, &c);
    const float ch = static_cast<float>(c), sh = static_cast<float>(s);
    cs[0][threadIdx.x] = ch;
    cs[1][threadIdx.x] = static_cast<float>(c - static_cast<double>(ch));
    cs[2][threadIdx.x] = sh;
    cs[3][threadIdx.x] = static_cast<float>(s - static_cast<double>(sh));
  }

  // Cache row of (sequence b, KV head 0) at the new token's slot; head g adds g * head_stride.
  size_t row0 = 0, head_stride = 0;
  bool append = true;
  if (paged) {
    const int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
    if (phys < 0 || phys >= a.num_blocks) {
      if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(a.err, RRA_ERR_BLOCK_ID);
      append = false;
    } else {
      row0 = ((static_cast<size_t>(phys) << a.log2_bs) + (pos & ((1 << a.log2_bs) - 1))) * a.Hkv;
      head_stride = 1;
    }
  } else {
    row0 = static_cast<size_t>(b) * a.Hkv * a.max_len + pos;
    head_stride = a.max_len;
  }
  __syncthreads();

  const bool inter = a.rope_style == 1;
  const int heads = append ? a.Hq + a.Hkv : a.Hq;
  constexpr int kRows = kRopeThreads / kPairsPerCta;
  const int j = threadIdx.x % kPairsPerCta;
  if (j < np) {
    const int i = i0 + j;
    const int ia = inter ? 2 * i : i;
    const int ib = inter ? 2 * i + 1 : i + half;
    const float ch = cs[0][j], cl = cs[1][j], sh = cs[2][j], sl = cs[3][j];
    for (int hh = threadIdx.x / kPairsPerCta; hh < heads; hh += kRows) {
      const T* src;
      T* dst;
      if (hh < a.Hq) {
        src = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.Hq + hh) * D;
        dst = static_cast<T*>(a.q_out) + (static_cast<size_t>(b) * a.Hq + hh) * D;
      } else {
        const int g = hh - a.Hq;
        src = static_cast<const T*>(a.k_new) + (static_cast<size_t>(b) * a.Hkv + g) * D;
        dst = static_cast<T*>(a.k_cache) + (row0 + g * head_stride) * D;
      }
      const float xa = Elem<T>::load(src + ia), xb = Elem<T>::load(src + ib);
      Elem<T>::store(dst + ia, rotate_diff(xa, xb, ch, cl, sh, sl));   // a cos - b sin
      Elem<T>::store(dst + ib, rotate_diff(xb, -xa, ch, cl, sh, sl));  // b cos + a sin
    }
  }
  if (!append) return;
  // V is stored unrotated: this CTA copies its share of the dims of every KV head.
  const int dims = (D + gridDim.y - 1) / gridDim.y;
  const int d0 = blockIdx.y * dims, d1 = min(D, d0 + dims);
  const T* vn = static_cast<const T*>(a.v_new) + static_cast<size_t>(b) * a.Hkv * D;
  T* vc = static_cast<T*>(a.v_cache);
  for (int idx = threadIdx.x; idx < a.Hkv * (d1 - d0); idx += blockDim.x) {
    const int g = idx / (d1 - d0), d = d0 + idx % (d1 - d0);
    vc[(row0 + g * head_stride) * D + d] = vn[g * D + d];
  }
}

}  // namespace

cudaError_t launch_rope_append(const RopeArgs& a, rra_dtype dt, cudaStream_t stream) {
  const dim3 grid(a.B, (a.D / 2 + kPairsPerCta - 1) / kPairsPerCta);
  if (dt == RRA_BF16)
    rope_append_kernel<__nv_bfloat16><<<grid, kRopeThreads, 0, stream>>>(a);
  else
    rope_append_kernel<float><<<grid, kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rra
