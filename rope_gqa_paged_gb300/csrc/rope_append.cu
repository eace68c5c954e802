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
// of its frequencies once as float32 hi + lo parts (rope_cos_sin: the angle in turns from an
// exact 96-bit fraction theta_i / 2pi, so no precision is lost at large positions, where a
// float32 angle is already ~0.004 rad off at 131071), and rotates that slice of every query
// and key head. The rotation a*c - b*s is computed from error-free
// float32 products (x*y = p + e exactly, with e = fma(x, y, -p): Dekker's product, using
// the FMA) so that it keeps full relative accuracy when the two products cancel; the
// result is then rounded once to the storage type.
//
// Quantised caches (§4.3 of the first page: INT8 or INT4 K/V with per-head calibrated scales,
// recent tokens kept at high precision; rope_append_qx_kernel): the rotated k is rounded to
// bf16 first, then quantised with its KV head's scale into the cache slot; with a window the
// bf16 values also go to slot pos % window of the sequence's ring.
#include <cmath>

#include "rra_device.cuh"
#include "rra_internal.h"

namespace rra {
namespace {

constexpr int kPairsPerCta = 16;
constexpr int kRopeThreads = 128;
constexpr int kRowsKernelMin = 256;  // token rows from which one CTA per row beats splitting each row

template <typename T>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(const RopeArgs a) {
  constexpr int kRows = kRopeThreads / kPairsPerCta;  // head rows handled side by side
  constexpr int kUnroll = 8;                          // head rows per thread loaded before any math
  __shared__ float cs[4][kPairsPerCta];               // cos hi, cos lo, sin hi, sin lo
  __shared__ size_t row_info[2];                      // cache row of KV head 0, stride between heads
  __shared__ int append_ok;
  // One CTA row per new token: token j of sequence b (gamma new tokens per sequence, j = 0 for a
  // decode step) sits at position positions[b] + j; its q / k_new / v_new / q_out row is v.
  const int gam = max(a.gamma, 1);
  const int v = blockIdx.x;
  const int b = v / gam, j_new = v - b * gam;
  const int D = a.D, half = a.D / 2;
  const int i0 = blockIdx.y * kPairsPerCta;
  const int np = min(kPairsPerCta, half - i0);
  const int heads = a.Hq + a.Hkv;
  const bool inter = a.rope_style == 1;
  const int j = threadIdx.x % kPairsPerCta;
  const int ia = inter ? 2 * (i0 + j) : i0 + j;
  const int ib = inter ? 2 * (i0 + j) + 1 : i0 + j + half;

  auto src_row = [&](int hh) -> const T* {
    return hh < a.Hq ? static_cast<const T*>(a.q) + (static_cast<size_t>(v) * a.Hq + hh) * D
                     : static_cast<const T*>(a.k_new) + (static_cast<size_t>(v) * a.Hkv + hh - a.Hq) * D;
  };
  // The first kUnroll rows of q / k_new are loaded before the position is even known.
  float xa[kUnroll], xb[kUnroll];
#pragma unroll
  for (int r = 0; r < kUnroll; ++r) {
    const int hh = threadIdx.x / kPairsPerCta + kRows * r;
    if (hh < heads && j < np) {
      xa[r] = Elem<T>::load(src_row(hh) + ia);
      xb[r] = Elem<T>::load(src_row(hh) + ib);
    }
  }

  const int pos = a.positions[b] + j_new;
  const bool paged = a.block_table != nullptr;
  const long long cap = paged ? (static_cast<long long>(a.max_blocks_per_seq) << a.log2_bs) : a.max_len;
  if (pos < 0 || pos >= cap) {
    if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  if (threadIdx.x < np) {
    rope_cos_sin(pos, a.rope_phi[i0 + threadIdx.x], cs[0][threadIdx.x], cs[1][threadIdx.x], cs[2][threadIdx.x],
                 cs[3][threadIdx.x]);
  }
  if (threadIdx.x == 32) {  // another warp resolves where the new token's K and V go
    int ok = 1;
    size_t row0 = 0, stride = 0;
    if (paged) {
      const int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
      if (phys < 0 || phys >= a.num_blocks) {
        if (blockIdx.y == 0) flag_error(a.err, RRA_ERR_BLOCK_ID);
        ok = 0;
      } else {
        row0 = ((static_cast<size_t>(phys) << a.log2_bs) + (pos & ((1 << a.log2_bs) - 1))) * a.Hkv;
        stride = 1;
      }
    } else {
      row0 = static_cast<size_t>(b) * a.Hkv * a.max_len + pos;
      stride = a.max_len;
    }
    row_info[0] = row0;
    row_info[1] = stride;
    append_ok = ok;
  }
  __syncthreads();
  const size_t row0 = row_info[0], head_stride = row_info[1];
  const bool append = append_ok != 0;

  if (j < np) {
    const float ch = cs[0][j], cl = cs[1][j], sh = cs[2][j], sl = cs[3][j];
    for (int base = 0; base < heads; base += kRows * kUnroll) {
#pragma unroll
      for (int r = 0; r < kUnroll; ++r) {
        const int hh = base + threadIdx.x / kPairsPerCta + kRows * r;
        if (hh >= heads) break;
        if (base > 0) {  // rows past the first kUnroll per thread (more than 64 heads)
          xa[r] = Elem<T>::load(src_row(hh) + ia);
          xb[r] = Elem<T>::load(src_row(hh) + ib);
        }
        const float ra = rotate_diff(xa[r], xb[r], ch, cl, sh, sl);   // a cos - b sin
        const float rb = rotate_diff(xb[r], -xa[r], ch, cl, sh, sl);  // b cos + a sin
        if (hh < a.Hq) {
          T* dst = static_cast<T*>(a.q_out) + (static_cast<size_t>(v) * a.Hq + hh) * D;
          Elem<T>::store(dst + ia, ra);
          Elem<T>::store(dst + ib, rb);
        } else if (append) {
          const int g = hh - a.Hq;
          T* dst = static_cast<T*>(a.k_cache) + (row0 + g * head_stride) * D;
          Elem<T>::store(dst + ia, ra);
          Elem<T>::store(dst + ib, rb);
        }
      }
    }
  }
  if (!append) return;
  // V is stored unrotated: this CTA copies its share of the dims of every KV head.
  const int dims = (D + gridDim.y - 1) / gridDim.y;
  const int d0 = blockIdx.y * dims, d1 = min(D, d0 + dims);
  const T* vn = static_cast<const T*>(a.v_new) + static_cast<size_t>(v) * a.Hkv * D;
  for (int idx = threadIdx.x; idx < a.Hkv * (d1 - d0); idx += blockDim.x) {
    const int g = idx / (d1 - d0), d = d0 + idx % (d1 - d0);
    static_cast<T*>(a.v_cache)[(row0 + g * head_stride) * D + d] = vn[g * D + d];
  }
}

// Many new tokens (prefill, speculative verify), bf16, every row 16-byte aligned: one CTA per
// token row, 16-byte vectors. The rotation and rounding are those of rope_append_kernel (the
// same sine/cosine split and error-free products), so both kernels write the same bits.
__global__ void __launch_bounds__(kRopeThreads) rope_append_rows_kernel(const RopeArgs a) {
  __shared__ float cs[4][kMaxHeadDim / 2];
  __shared__ size_t row_info[2];
  __shared__ int append_ok;
  const int gam = max(a.gamma, 1);
  const int v = blockIdx.x;
  const int b = v / gam, j_new = v - b * gam;
  const int D = a.D, half = a.D / 2;
  const int pos = a.positions[b] + j_new;
  const bool paged = a.block_table != nullptr;
  const long long cap = paged ? (static_cast<long long>(a.max_blocks_per_seq) << a.log2_bs) : a.max_len;
  if (pos < 0 || pos >= cap) {
    if (threadIdx.x == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    rope_cos_sin(pos, a.rope_phi[i], cs[0][i], cs[1][i], cs[2][i], cs[3][i]);
  }
  if (threadIdx.x == kRopeThreads - 1) {  // where the token's K and V go
    int ok = 1;
    size_t row0 = 0, stride = 0;
    if (paged) {
      const int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
      if (phys < 0 || phys >= a.num_blocks) {
        flag_error(a.err, RRA_ERR_BLOCK_ID);
        ok = 0;
      } else {
        row0 = ((static_cast<size_t>(phys) << a.log2_bs) + (pos & ((1 << a.log2_bs) - 1))) * a.Hkv;
        stride = 1;
      }
    } else {
      row0 = static_cast<size_t>(b) * a.Hkv * a.max_len + pos;
      stride = a.max_len;
    }
    row_info[0] = row0;
    row_info[1] = stride;
    append_ok = ok;
  }
  __syncthreads();
  const size_t row0 = row_info[0], head_stride = row_info[1];
  const bool append = append_ok != 0;
  const bool inter = a.rope_style == 1;
  const int heads = a.Hq + a.Hkv;
  // a task is 8 dims: half-split pairs (i, i + D/2) for i in [8t, 8t + 8) (two vectors), or the
  // interleaved pairs (2i, 2i + 1) for i in [4t, 4t + 4) (one vector)
  const int per_head = inter ? D / 8 : half / 8;
  auto pack8 = [](const float (&x)[8]) {
    uint4 r;
    uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t*>(&p);
    }
    return r;
  };
  for (int task = threadIdx.x; task < heads * per_head; task += blockDim.x) {
    const int hh = task / per_head, t = task - hh * per_head;
    const bool is_q = hh < a.Hq;
    if (!is_q && !append) continue;
    const __nv_bfloat16* src =
        is_q ? static_cast<const __nv_bfloat16*>(a.q) + (static_cast<size_t>(v) * a.Hq + hh) * D
             : static_cast<const __nv_bfloat16*>(a.k_new) + (static_cast<size_t>(v) * a.Hkv + hh - a.Hq) * D;
    __nv_bfloat16* dst = is_q ? static_cast<__nv_bfloat16*>(a.q_out) + (static_cast<size_t>(v) * a.Hq + hh) * D
                              : static_cast<__nv_bfloat16*>(a.k_cache) + (row0 + (hh - a.Hq) * head_stride) * D;
    if (!inter) {
      float xa[8], xb[8], oa[8], ob[8];
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(src + 8 * t), xa);
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(src + half + 8 * t), xb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = 8 * t + e;
        oa[e] = rotate_diff(xa[e], xb[e], cs[0][i], cs[1][i], cs[2][i], cs[3][i]);   // a cos - b sin
        ob[e] = rotate_diff(xb[e], -xa[e], cs[0][i], cs[1][i], cs[2][i], cs[3][i]);  // b cos + a sin
      }
      *reinterpret_cast<uint4*>(dst + 8 * t) = pack8(oa);
      *reinterpret_cast<uint4*>(dst + half + 8 * t) = pack8(ob);
    } else {
      float x[8], o[8];
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(src + 8 * t), x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * t + e;
        o[2 * e] = rotate_diff(x[2 * e], x[2 * e + 1], cs[0][i], cs[1][i], cs[2][i], cs[3][i]);
        o[2 * e + 1] = rotate_diff(x[2 * e + 1], -x[2 * e], cs[0][i], cs[1][i], cs[2][i], cs[3][i]);
      }
      *reinterpret_cast<uint4*>(dst + 8 * t) = pack8(o);
    }
  }
  if (!append) return;
  // V is stored unrotated
  const uint4* vn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.v_new) +
                                                   static_cast<size_t>(v) * a.Hkv * D);
  for (int task = threadIdx.x; task < a.Hkv * (D / 8); task += blockDim.x) {
    const int g = task / (D / 8), t = task - g * (D / 8);
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.v_cache) + (row0 + g * head_stride) * D)[t] = vn[task];
  }
}

// Quantised caches (bf16 q / k / v; INT8 codes, or INT4 two per byte at head dim 128): one CTA per
// sequence, one warp per head row. Lane l holds dims E l .. E l + E - 1 (E = D / 32: one vector,
// all of a warp's rows loaded before any arithmetic); a half-split RoPE pair (i, i + D/2) sits in
// lanes l and l ^ 16. INT4: the codes of dims 2j and 2j + 1 go to byte j (the even one in the low
// nibble). Rotation, rounding and codes are those of rope_append_kernel.
constexpr int kQ4Warps = 8;
constexpr int kQ4RowsPerWarp = 6;

template <int D>
struct LaneVec;  // E = D / 32 bf16 per lane
template <>
struct LaneVec<128> {
  using T = uint2;
  __device__ __forceinline__ static void unpack(T w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xffff0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xffff0000u);
  }
  __device__ __forceinline__ static T pack(const __nv_bfloat16 (&o)[4]) {
    return make_uint2(static_cast<uint32_t>(__bfloat16_as_ushort(o[0])) | (static_cast<uint32_t>(__bfloat16_as_ushort(o[1])) << 16),
                      static_cast<uint32_t>(__bfloat16_as_ushort(o[2])) | (static_cast<uint32_t>(__bfloat16_as_ushort(o[3])) << 16));
  }
};
template <>
struct LaneVec<64> {
  using T = uint32_t;
  __device__ __forceinline__ static void unpack(T w, float (&x)[2]) {
    x[0] = __uint_as_float(w << 16);
    x[1] = __uint_as_float(w & 0xffff0000u);
  }
  __device__ __forceinline__ static T pack(const __nv_bfloat16 (&o)[2]) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(o[0])) | (static_cast<uint32_t>(__bfloat16_as_ushort(o[1])) << 16);
  }
};

template <int D, int BITS>
__global__ void __launch_bounds__(kQ4Warps * 32) rope_append_qx_kernel(const RopeArgs a) {
  constexpr int HALF = D / 2, E = D / 32;
  constexpr int RB = D * BITS / 8;  // code bytes per row
  using V = LaneVec<D>;
  using VT = typename V::T;
  __shared__ float cs[4][HALF];
  __shared__ size_t row_info[2];
  __shared__ int append_ok;
  const int b = blockIdx.x;
  const int pos = a.positions[b];
  const bool paged = a.block_table != nullptr;
  const long long cap = paged ? (static_cast<long long>(a.max_blocks_per_seq) << a.log2_bs) : a.max_len;
  if (pos < 0 || pos >= cap) {
    if (threadIdx.x == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  if (threadIdx.x < HALF) {
    rope_cos_sin(pos, a.rope_phi[threadIdx.x], cs[0][threadIdx.x], cs[1][threadIdx.x], cs[2][threadIdx.x],
                 cs[3][threadIdx.x]);
  }
  if (threadIdx.x == kQ4Warps * 32 - 1) {  // where the token's codes go
    int ok = 1;
    size_t row0 = 0, stride = 0;
    if (paged) {
      const int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
      if (phys < 0 || phys >= a.num_blocks) {
        flag_error(a.err, RRA_ERR_BLOCK_ID);
        ok = 0;
      } else {
        row0 = ((static_cast<size_t>(phys) << a.log2_bs) + (pos & ((1 << a.log2_bs) - 1))) * a.Hkv;
        stride = 1;
      }
    } else {
      row0 = static_cast<size_t>(b) * a.Hkv * a.max_len + pos;
      stride = a.max_len;
    }
    row_info[0] = row0;
    row_info[1] = stride;
    append_ok = ok;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = a.Hq + a.Hkv;
  const bool inter = a.rope_style == 1, first = lane < 16;
  const __nv_bfloat16* qin = static_cast<const __nv_bfloat16*>(a.q) + static_cast<size_t>(b) * a.Hq * D;
  __nv_bfloat16* qout = static_cast<__nv_bfloat16*>(a.q_out) + static_cast<size_t>(b) * a.Hq * D;
  const __nv_bfloat16* kin = static_cast<const __nv_bfloat16*>(a.k_new) + static_cast<size_t>(b) * a.Hkv * D;
  const __nv_bfloat16* vin = static_cast<const __nv_bfloat16*>(a.v_new) + static_cast<size_t>(b) * a.Hkv * D;
  for (int base = 0; base < heads; base += kQ4Warps * kQ4RowsPerWarp) {
    VT xr[kQ4RowsPerWarp], vr[kQ4RowsPerWarp];
#pragma unroll
    for (int r = 0; r < kQ4RowsPerWarp; ++r) {
      const int hh = base + warp + kQ4Warps * r;
      if (hh < heads) {
        const bool is_q = hh < a.Hq;
        xr[r] = *reinterpret_cast<const VT*>((is_q ? qin + static_cast<size_t>(hh) * D
                                                   : kin + static_cast<size_t>(hh - a.Hq) * D) + E * lane);
        if (!is_q) vr[r] = *reinterpret_cast<const VT*>(vin + static_cast<size_t>(hh - a.Hq) * D + E * lane);
      }
    }
    __syncthreads();  // the sine / cosine table and the cache row are ready
    const size_t row0 = row_info[0], stride = row_info[1];
    const bool append = append_ok != 0;
#pragma unroll
    for (int r = 0; r < kQ4RowsPerWarp; ++r) {
      const int hh = base + warp + kQ4Warps * r;  // the same for the whole warp
      if (hh >= heads) continue;
      float x[E];
      V::unpack(xr[r], x);
      __nv_bfloat16 o[E];
      if (inter) {  // pairs (2i, 2i + 1) inside the lane
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const int i = (E * lane + e) / 2;
          o[e] = __float2bfloat16_rn(rotate_diff(x[e], x[e + 1], cs[0][i], cs[1][i], cs[2][i], cs[3][i]));
          o[e + 1] = __float2bfloat16_rn(rotate_diff(x[e + 1], -x[e], cs[0][i], cs[1][i], cs[2][i], cs[3][i]));
        }
      } else {  // pairs (i, i + D/2): the partner is 16 lanes away
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
          const int i = E * (lane & 15) + e;
          o[e] = __float2bfloat16_rn(first ? rotate_diff(x[e], partner, cs[0][i], cs[1][i], cs[2][i], cs[3][i])
                                           : rotate_diff(x[e], -partner, cs[0][i], cs[1][i], cs[2][i], cs[3][i]));
        }
      }
      const VT packed = V::pack(o);
      if (hh < a.Hq) {
        *reinterpret_cast<VT*>(qout + static_cast<size_t>(hh) * D + E * lane) = packed;
        continue;
      }
      if (!append) continue;
      const int g = hh - a.Hq;
      const float ks = a.k_scale[g], vs = a.v_scale[g];
      float v[E];
      V::unpack(vr[r], v);
      uint8_t* kd = static_cast<uint8_t*>(a.k_cache) + (row0 + g * stride) * RB + (E * BITS / 8) * lane;
      uint8_t* vd = static_cast<uint8_t*>(a.v_cache) + (row0 + g * stride) * RB + (E * BITS / 8) * lane;
      uint32_t kc = 0, vc = 0;
      if constexpr (BITS == 8) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          kc |= static_cast<uint32_t>(static_cast<uint8_t>(quantize_code(__bfloat162float(o[e]), ks))) << (8 * e);
          vc |= static_cast<uint32_t>(static_cast<uint8_t>(quantize_code(v[e], vs))) << (8 * e);
        }
      } else {
#pragma unroll
        for (int j = 0; j < E / 2; ++j) {
          kc |= static_cast<uint32_t>(pack_nibbles(quantize_code4(__bfloat162float(o[2 * j]), ks),
                                                   quantize_code4(__bfloat162float(o[2 * j + 1]), ks)))
                << (8 * j);
          vc |= static_cast<uint32_t>(pack_nibbles(quantize_code4(v[2 * j], vs), quantize_code4(v[2 * j + 1], vs)))
                << (8 * j);
        }
      }
      if constexpr (E * BITS / 8 == 4) {
        *reinterpret_cast<uint32_t*>(kd) = kc;
        *reinterpret_cast<uint32_t*>(vd) = vc;
      } else {
        *reinterpret_cast<uint16_t*>(kd) = static_cast<uint16_t>(kc);
        *reinterpret_cast<uint16_t*>(vd) = static_cast<uint16_t>(vc);
      }
      if (a.window > 0) {
        const size_t w = ((static_cast<size_t>(b) * a.Hkv + g) * a.window + pos % a.window) * D + E * lane;
        *reinterpret_cast<VT*>(static_cast<__nv_bfloat16*>(a.k_win) + w) = packed;
        *reinterpret_cast<VT*>(static_cast<__nv_bfloat16*>(a.v_win) + w) = vr[r];
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope_append_q4(const RopeArgs& a, cudaStream_t stream) {
  rope_append_qx_kernel<128, 4><<<a.B, kQ4Warps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_append(const RopeArgs& a, rra_dtype dt, cudaStream_t stream) {
  const int rows = a.B * (a.gamma > 1 ? a.gamma : 1);
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (dt == RRA_BF16 && rows >= kRowsKernelMin && a.D % 16 == 0 && al16(a.q) && al16(a.k_new) && al16(a.v_new) && al16(a.q_out) &&
      al16(a.k_cache) && al16(a.v_cache)) {
    rope_append_rows_kernel<<<rows, kRopeThreads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  const dim3 grid(rows, (a.D / 2 + kPairsPerCta - 1) / kPairsPerCta);
  if (dt == RRA_BF16)
    rope_append_kernel<__nv_bfloat16><<<grid, kRopeThreads, 0, stream>>>(a);
  else
    rope_append_kernel<float><<<grid, kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_append_q8(const RopeArgs& a, cudaStream_t stream) {
  if (a.D == 128)
    rope_append_qx_kernel<128, 8><<<a.B, kQ4Warps * 32, 0, stream>>>(a);
  else
    rope_append_qx_kernel<64, 8><<<a.B, kQ4Warps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

// theta_i / 2pi for i < D/2, theta_i = base^(-2i/D) in float64, as a 96-bit binary fraction
// (least significant 32-bit word first), exact up to truncation (< 2^-96): theta = m 2^(e-53) with
// an integer m < 2^53, times floor(2^127 / pi) (2^128 / 2pi, a 128-bit integer), shifted down.
void fill_rope_phi(uint32_t (*phi)[3], int D, double base) {
  // floor(2^127 / pi), computed at 400-bit precision
  constexpr uint64_t kHi = 0x28be60db9391054aULL, kLo = 0x7f09d5f47d4d3770ULL;
  using u128 = unsigned __int128;
  for (int i = 0; i < D / 2; ++i) {
    const double th = std::pow(base, -2.0 * i / D);
    int e = 0;
    const uint64_t m = static_cast<uint64_t>(std::ldexp(std::frexp(th, &e), 53));  // th = m 2^(e-53)
    // m * K as 192 bits p2:p1:p0
    const u128 lo = u128(m) * kLo, hi = u128(m) * kHi;
    const uint64_t p0 = uint64_t(lo);
    const u128 mid = (lo >> 64) + u128(uint64_t(hi));
    const uint64_t p1 = uint64_t(mid);
    const uint64_t p2 = uint64_t(hi >> 64) + uint64_t(mid >> 64);
    // theta / 2pi * 2^96 = m K 2^(e - 53 - 128 + 96) = (m K) >> (85 - e)
    const int sh = 85 - e;
    uint64_t w[3] = {p0, p1, p2}, out[2] = {0, 0};
    for (int j = 0; j < 2; ++j) {  // bits [sh + 64 j, sh + 64 j + 64) of m K
      const int bit = sh + 64 * j, word = bit >> 6, off = bit & 63;
      uint64_t v = 0;
      if (bit >= 0 && word < 3) v = w[word] >> off;
      if (bit >= 0 && off != 0 && word + 1 < 3) v |= w[word + 1] << (64 - off);
      out[j] = v;
    }
    phi[i][0] = static_cast<uint32_t>(out[0]);
    phi[i][1] = static_cast<uint32_t>(out[0] >> 32);
    phi[i][2] = static_cast<uint32_t>(out[1]);
  }
}

namespace {
struct RopePhiTable {
  uint32_t phi[kMaxHeadDim / 2][3];
};
// out[n][4][half]: cos hi, cos lo, sin hi, sin lo of positions[n] * theta_i (NaN for a negative position).
__global__ void rope_cos_sin_kernel(const int32_t* positions, int n, int half, const RopePhiTable t, float* out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  const int p = idx / half, i = idx - p * half;
  const int pos = positions[p];
  float* o = out + static_cast<size_t>(p) * 4 * half;
  if (pos < 0) {
    o[i] = o[half + i] = o[2 * half + i] = o[3 * half + i] = __int_as_float(0x7fc00000);
    return;
  }
  rope_cos_sin(pos, t.phi[i], o[i], o[half + i], o[2 * half + i], o[3 * half + i]);
}
}  // namespace

}  // namespace rra

extern "C" {

RRA_API int rra_rope_phi(int head_dim, double rope_base, uint32_t* phi) {
  if (phi == nullptr || head_dim < 2 || head_dim % 2 != 0 || head_dim > rra::kMaxHeadDim ||
      !(rope_base > 0.0) || !std::isfinite(rope_base))
    return RRA_EINVAL;
  rra::fill_rope_phi(reinterpret_cast<uint32_t(*)[3]>(phi), head_dim, rope_base);
  return RRA_OK;
}

RRA_API int rra_rope_cos_sin_host(int position, const uint32_t* phi, float* out) {
  if (phi == nullptr || out == nullptr || position < 0) return RRA_EINVAL;
  rra::rope_cos_sin(position, phi, out[0], out[1], out[2], out[3]);
  return RRA_OK;
}

RRA_API int rra_rope_cos_sin(const int32_t* positions, int n, int head_dim, double rope_base, float* out,
                             void* stream) {
  if (n < 0 || (n > 0 && (positions == nullptr || out == nullptr)) || head_dim < 2 || head_dim % 2 != 0 ||
      head_dim > rra::kMaxHeadDim || !(rope_base > 0.0) || !std::isfinite(rope_base))
    return RRA_EINVAL;
  const int half = head_dim / 2;
  if (int64_t(n) * half > int64_t(INT32_MAX)) return RRA_ERANGE;
  if (n == 0) return RRA_OK;
  rra::RopePhiTable t{};
  rra::fill_rope_phi(t.phi, head_dim, rope_base);
  const int items = n * half, threads = 128;
  rra::rope_cos_sin_kernel<<<(items + threads - 1) / threads, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      positions, n, half, t, out);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    rra::record_cuda_error(e, "rope_cos_sin kernel launch");
    return RRA_ECUDA;
  }
  return RRA_OK;
}

}  // extern "C"
