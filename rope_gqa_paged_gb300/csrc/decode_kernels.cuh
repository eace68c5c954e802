// Split-K GQA decode attention (flash-decoding) and its log-sum-exp merge.
//
// Math: "Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §2.1 (softmax(QK^T/sqrt(d_k))V,
// one query row in decode), §2.2 (KV head g serves query heads g*n_rep .. g*n_rep+n_rep-1,
// the repeat_interleave mapping), §4.2 (blockwise computation on chip, never writing the
// score matrix to HBM), §5.2 (decode is bound by reading the KV cache from memory).
// "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南" §三 (scale
// 1/sqrt(d_k)), §四 (paged K/V = table-ordered concatenation of blocks).
//
// Structure of decode_split_kernel: one CTA per (split, KV head [x head slice], sequence).
//   * warp 4 (producer): one lane streams the split's K and V rows into a 4-stage ring
//     of 16 KB shared-memory stages with bulk copies (contiguous cache) or 4-D TMA tile
//     copies (paged pool, one copy per block and per K/V), each stage completing on an
//     mbarrier with a byte count. The block ids of the split are copied to shared memory
//     once, when the CTA starts.
//   * warps 0-3 (consumers): 8 lanes per token, 16 tokens in flight per pass. Each lane
//     owns D/8 dims (two 16-byte chunks 128 bytes apart, so the 8 lanes of a token read
//     one full 128-byte bank line) and keeps, for the CTA's HPC query heads, its slice of
//     q (pre-scaled by scale*log2 e), its slice of the output accumulator, and the running
//     max / sum of its own token subsequence (online softmax in base 2, float32).
//     Every K row is read from shared memory once and used by all HPC heads.
//   * end: the 16 token groups merge through shared memory; one split writes the final
//     row, several splits write (unnormalised o, max, sum) for decode_reduce_kernel.
// Every wait has a time limit; a wait that runs out sets RRA_ERR_TIMEOUT and the CTA
// finishes without blocking.
#pragma once

#include "rra_device.cuh"
#include "rra_internal.h"

namespace rra {

template <typename T, int D>
struct DecodeCfg {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kTile = 8192 / kRowBytes;            // tokens per stage (K 8 KB + V 8 KB)
  static constexpr int kStages = 4;
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kGroupLanes = 8;                      // lanes per token
  static constexpr int kGroups = kConsumerWarps * 32 / kGroupLanes;
  static constexpr int kTPG = kTile / kGroups;               // tokens per group per stage
  static constexpr int kEPC = Elem<T>::kPerChunk;            // elements per 16-byte chunk
  static constexpr int kNC = kRowBytes / 16 / kGroupLanes;   // chunks per lane per row
  static constexpr int kDPL = kNC * kEPC;                    // dims per lane
  static constexpr int kStageBytes = 2 * kTile * kRowBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + 2 * kStages * 8 + kMaxTableEntries * 4;
  static_assert(kTPG >= 1 && kNC >= 1, "tile too small for the lane layout");
};

template <typename T, int D, int HPC>
struct ConsumerState {
  using C = DecodeCfg<T, D>;
  float q[HPC][C::kDPL];
  float o[HPC][C::kDPL];
  float m[HPC];
  float l[HPC];
};

// One stage of tokens for one consumer lane. CHECK: the stage holds fewer than kTile
// valid tokens (rows past `valid` may hold stale or NaN data and are never multiplied).
template <typename T, int D, int HPC, bool CHECK>
__device__ __forceinline__ void consume_stage(ConsumerState<T, D, HPC>& st, const T* __restrict__ sK,
                                              const T* __restrict__ sV, int grp, int j, int valid) {
  using C = DecodeCfg<T, D>;
  float sc[C::kTPG][HPC];
#pragma unroll
  for (int p = 0; p < C::kTPG; ++p) {
    const int tt = grp * C::kTPG + p;
    const uint4* row = reinterpret_cast<const uint4*>(sK + tt * D);
    float acc[HPC];
#pragma unroll
    for (int h = 0; h < HPC; ++h) acc[h] = 0.f;
#pragma unroll
    for (int c = 0; c < C::kNC; ++c) {
      float x[C::kEPC];
      Elem<T>::unpack(row[j + C::kGroupLanes * c], x);
#pragma unroll
      for (int h = 0; h < HPC; ++h)
#pragma unroll
        for (int e = 0; e < C::kEPC; ++e) acc[h] = fmaf(st.q[h][c * C::kEPC + e], x[e], acc[h]);
    }
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 4);
      sc[p][h] = (!CHECK || tt < valid) ? acc[h] : -INFINITY;
    }
  }

  // Online softmax: raise the running max once per stage, rescale only when it grew.
  float mnew[HPC];
  bool grow = false;
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    float mx = st.m[h];
#pragma unroll
    for (int p = 0; p < C::kTPG; ++p) mx = fmaxf(mx, sc[p][h]);
    mnew[h] = mx;
    grow |= mx > st.m[h];
  }
  if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      const float alpha = mnew[h] > st.m[h] ? exp2f(st.m[h] - mnew[h]) : 1.f;
      st.l[h] *= alpha;
#pragma unroll
      for (int d = 0; d < C::kDPL; ++d) st.o[h][d] *= alpha;
      st.m[h] = mnew[h];
    }
  }
  float pr[C::kTPG][HPC];
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    const float mref = st.m[h] == -INFINITY ? 0.f : st.m[h];
#pragma unroll
    for (int p = 0; p < C::kTPG; ++p) {
      pr[p][h] = exp2f(sc[p][h] - mref);
      st.l[h] += pr[p][h];
    }
  }

#pragma unroll
  for (int p = 0; p < C::kTPG; ++p) {
    const int tt = grp * C::kTPG + p;
    if (CHECK && tt >= valid) continue;
    const uint4* row = reinterpret_cast<const uint4*>(sV + tt * D);
#pragma unroll
    for (int c = 0; c < C::kNC; ++c) {
      float x[C::kEPC];
      Elem<T>::unpack(row[j + C::kGroupLanes * c], x);
#pragma unroll
      for (int h = 0; h < HPC; ++h)
#pragma unroll
        for (int e = 0; e < C::kEPC; ++e)
          st.o[h][c * C::kEPC + e] = fmaf(pr[p][h], x[e], st.o[h][c * C::kEPC + e]);
    }
  }
}

template <typename T, int D, int HPC, bool PAGED>
__global__ void __launch_bounds__(DecodeCfg<T, D>::kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                        const DecodeArgs a) {
  using C = DecodeCfg<T, D>;
  extern __shared__ __align__(128) uint8_t smem[];

  const int split = blockIdx.x;
  const int n_rep = a.Hq / a.Hkv;
  const int slices = n_rep / HPC;
  const int g = blockIdx.y / slices;
  const int h0 = g * n_rep + (blockIdx.y - g * slices) * HPC;
  const int b = blockIdx.z;

  int L = a.seq_lens[b];
  if (L < 0 || L > a.capacity) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_error(a.err, RRA_ERR_SEQ_LEN);
    L = min(max(L, 0), a.capacity);
  }
  const int start = split * a.chunk;
  if (start >= L) {
    if (L == 0 && a.num_splits == 1) {  // nothing to attend to: a zero row
      T* out = static_cast<T*>(a.out) + (static_cast<size_t>(b) * a.Hq + h0) * D;
      for (int i = threadIdx.x; i < HPC * D; i += blockDim.x) Elem<T>::store(out + i, 0.f);
    }
    return;
  }
  const int end = min(L, start + a.chunk);
  const int n_tiles = (end - start + C::kTile - 1) / C::kTile;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
  uint64_t* empty = full + C::kStages;
  int32_t* tbl = reinterpret_cast<int32_t*>(empty + C::kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    fence_barrier_init();
  }
  int first_blk = 0;
  if constexpr (PAGED) {
    first_blk = start >> a.log2_bs;
    const int n_blk = ((end - 1) >> a.log2_bs) - first_blk + 1;
    const int32_t* row = a.block_table + static_cast<size_t>(b) * a.max_blocks_per_seq + first_blk;
    for (int i = threadIdx.x; i < n_blk; i += blockDim.x) {
      int id = row[i];
      if (id < 0 || id >= a.num_blocks) {
        flag_error(a.err, RRA_ERR_BLOCK_ID);
        id = 0;
      }
      tbl[i] = id;
    }
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer
  if (warp == C::kConsumerWarps) {
    if (lane == 0) {
      if constexpr (PAGED) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
      }
      const size_t head_row = (static_cast<size_t>(b) * a.Hkv + g) * a.max_len;
      const uint8_t* kbase = static_cast<const uint8_t*>(a.k) + head_row * C::kRowBytes;
      const uint8_t* vbase = static_cast<const uint8_t*>(a.v) + head_row * C::kRowBytes;
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1)) {
          flag_error(a.err, RRA_ERR_TIMEOUT);
          break;
        }
        const int t0 = start + it * C::kTile;
        const int rows = min(C::kTile, end - t0);
        uint8_t* dK = smem + s * C::kStageBytes;
        uint8_t* dV = dK + C::kTile * C::kRowBytes;
        if constexpr (PAGED) {
          const int bs = 1 << a.log2_bs;
          if (bs <= C::kTile) {  // whole blocks: one copy per block (box = bs rows)
            const int nblk = (rows + bs - 1) >> a.log2_bs;
            const uint32_t bytes = static_cast<uint32_t>(nblk) * bs * C::kRowBytes;
            mbar_arrive_expect_tx(&full[s], 2 * bytes);
            const int j0 = (t0 >> a.log2_bs) - first_blk;
            for (int jb = 0; jb < nblk; ++jb) {
              const int phys = tbl[j0 + jb];
              tma_g2s_4d(dK + jb * bs * C::kRowBytes, &k_map, 0, g, 0, phys, &full[s]);
              tma_g2s_4d(dV + jb * bs * C::kRowBytes, &v_map, 0, g, 0, phys, &full[s]);
            }
          } else {  // part of one block (box = kTile rows)
            const int phys = tbl[(t0 >> a.log2_bs) - first_blk];
            const int off = t0 & (bs - 1);
            mbar_arrive_expect_tx(&full[s], 2 * C::kTile * C::kRowBytes);
            tma_g2s_4d(dK, &k_map, 0, g, off, phys, &full[s]);
            tma_g2s_4d(dV, &v_map, 0, g, off, phys, &full[s]);
          }
        } else {
          const uint32_t bytes = static_cast<uint32_t>(rows) * C::kRowBytes;
          mbar_arrive_expect_tx(&full[s], 2 * bytes);
          bulk_g2s(dK, kbase + static_cast<size_t>(t0) * C::kRowBytes, bytes, &full[s]);
          bulk_g2s(dV, vbase + static_cast<size_t>(t0) * C::kRowBytes, bytes, &full[s]);
        }
        issued = it + 1;
      }
      // Never leave with copies in flight: wait (bounded) for the last stages to land.
      for (int it = issued > C::kStages ? issued - C::kStages : 0; it < issued; ++it)
        mbar_wait(&full[it % C::kStages], (it / C::kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int grp = warp * (32 / C::kGroupLanes) + lane / C::kGroupLanes;
  const int j = lane % C::kGroupLanes;
  ConsumerState<T, D, HPC> st;
  {
    const T* q = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.Hq + h0) * D;
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      const uint4* qrow = reinterpret_cast<const uint4*>(q + h * D);
#pragma unroll
      for (int c = 0; c < C::kNC; ++c) {
        float x[C::kEPC];
        Elem<T>::unpack(qrow[j + C::kGroupLanes * c], x);
#pragma unroll
        for (int e = 0; e < C::kEPC; ++e) st.q[h][c * C::kEPC + e] = x[e] * a.scale_log2;
      }
#pragma unroll
      for (int d = 0; d < C::kDPL; ++d) st.o[h][d] = 0.f;
      st.m[h] = -INFINITY;
      st.l[h] = 0.f;
    }
  }

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % C::kStages;
    if (!mbar_wait(&full[s], (it / C::kStages) & 1)) {
      flag_error(a.err, RRA_ERR_TIMEOUT);
      break;
    }
    const T* sK = reinterpret_cast<const T*>(smem + s * C::kStageBytes);
    const T* sV = sK + C::kTile * D;
    const int valid = min(C::kTile, end - (start + it * C::kTile));
    if (valid == C::kTile)
      consume_stage<T, D, HPC, false>(st, sK, sV, grp, j, valid);
    else
      consume_stage<T, D, HPC, true>(st, sK, sV, grp, j, valid);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ------------------------------------------------------------------ merge the 16 groups
  constexpr int kConsumers = C::kConsumerWarps * 32;
  named_barrier_sync(1, kConsumers);  // every consumer is done with the ring
  float* red_o = reinterpret_cast<float*>(smem);           // [groups][HPC][D]
  float* red_m = red_o + C::kGroups * HPC * D;             // [groups][HPC]
  float* red_l = red_m + C::kGroups * HPC;
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
#pragma unroll
    for (int c = 0; c < C::kNC; ++c)
#pragma unroll
      for (int e = 0; e < C::kEPC; ++e)
        red_o[(grp * HPC + h) * D + (j + C::kGroupLanes * c) * C::kEPC + e] = st.o[h][c * C::kEPC + e];
    if (j == 0) {
      red_m[grp * HPC + h] = st.m[h];
      red_l[grp * HPC + h] = st.l[h];
    }
  }
  named_barrier_sync(1, kConsumers);
  for (int idx = threadIdx.x; idx < HPC * D; idx += kConsumers) {
    const int h = idx / D, d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < C::kGroups; ++q) M = fmaxf(M, red_m[q * HPC + h]);
    float lsum = 0.f, osum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int q = 0; q < C::kGroups; ++q) {
        const float w = exp2f(red_m[q * HPC + h] - M);
        lsum = fmaf(w, red_l[q * HPC + h], lsum);
        osum = fmaf(w, red_o[(q * HPC + h) * D + d], osum);
      }
    }
    const size_t bh = static_cast<size_t>(b) * a.Hq + h0 + h;
    if (a.num_splits == 1) {
      Elem<T>::store(static_cast<T*>(a.out) + bh * D + d, lsum > 0.f ? osum / lsum : 0.f);
    } else {
      const size_t ps = bh * a.num_splits + split;
      a.ws_o[ps * D + d] = osum;
      if (d == 0) {
        a.ws_ml[2 * ps] = M;
        a.ws_ml[2 * ps + 1] = lsum;
      }
    }
  }
}

// Merge the splits of one (sequence, query head): M = max_s m_s, w_s = 2^(m_s - M),
// out = sum_s w_s o_s / sum_s w_s l_s. One warp per (sequence, head), each lane owning
// D/32 consecutive dims; only the splits that held tokens are read.
constexpr int kReduceWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_kernel(const DecodeArgs a) {
  constexpr int kDL = D / 32;  // dims per lane
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kReduceWarps + (threadIdx.x >> 5);  // b * Hq + hq
  if (row >= a.B * a.Hq) return;
  const int b = row / a.Hq;
  const int L = min(max(a.seq_lens[b], 0), a.capacity);
  const int n = (L + a.chunk - 1) / a.chunk;
  const float* ml = a.ws_ml + static_cast<size_t>(row) * a.num_splits * 2;
  const float* o = a.ws_o + static_cast<size_t>(row) * a.num_splits * D + lane * kDL;

  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));

  float lsum = 0.f, acc[kDL];
#pragma unroll
  for (int e = 0; e < kDL; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < n; s0 += 32) {
    const int s = s0 + lane;
    const float w = s < n ? exp2f(ml[2 * s] - M) : 0.f;
    lsum = fmaf(w, s < n ? ml[2 * s + 1] : 0.f, lsum);
    const int cnt = min(32, n - s0);
    for (int k = 0; k < cnt; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      const float* os = o + static_cast<size_t>(s0 + k) * D;
      if constexpr (kDL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(os);
        acc[0] = fmaf(wk, v.x, acc[0]);
        acc[1] = fmaf(wk, v.y, acc[1]);
        acc[2] = fmaf(wk, v.z, acc[2]);
        acc[3] = fmaf(wk, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(os);
        acc[0] = fmaf(wk, v.x, acc[0]);
        acc[1] = fmaf(wk, v.y, acc[1]);
      }
    }
  }
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, x);
  const float inv = (n > 0 && lsum > 0.f) ? 1.f / lsum : 0.f;
  T* out = static_cast<T*>(a.out) + static_cast<size_t>(row) * D + lane * kDL;
#pragma unroll
  for (int e = 0; e < kDL; ++e) Elem<T>::store(out + e, acc[e] * inv);
}

template <typename T, int D, int HPC, bool PAGED>
cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t st) {
  using C = DecodeCfg<T, D>;
  static int done[64] = {0};
  auto kern = decode_split_kernel<T, D, HPC, PAGED>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_splits, a.Hkv * (a.Hq / a.Hkv / HPC), a.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(km, vm, a);
  return cudaGetLastError();
}

template <typename T, int D, bool PAGED>
cudaError_t launch_decode_hpc(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, int hpc,
                              cudaStream_t st) {
  switch (hpc) {
    case 4: return launch_decode_t<T, D, 4, PAGED>(a, km, vm, st);
    case 2: return launch_decode_t<T, D, 2, PAGED>(a, km, vm, st);
    default: return launch_decode_t<T, D, 1, PAGED>(a, km, vm, st);
  }
}

template <bool PAGED>
cudaError_t launch_decode_any(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, rra_dtype dt,
                              int hpc, cudaStream_t st) {
  if (dt == RRA_BF16) {
    if (a.D == 128) return launch_decode_hpc<__nv_bfloat16, 128, PAGED>(a, km, vm, hpc, st);
    return launch_decode_hpc<__nv_bfloat16, 64, PAGED>(a, km, vm, hpc, st);
  }
  if (a.D == 128) return launch_decode_hpc<float, 128, PAGED>(a, km, vm, hpc, st);
  return launch_decode_hpc<float, 64, PAGED>(a, km, vm, hpc, st);
}

}  // namespace rra
