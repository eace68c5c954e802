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
//   * end: the 16 token groups merge through shared memory; a sequence with one split
//     writes its final row, otherwise each split publishes (unnormalised o, max, sum) and
//     the last split to finish merges them (finish_split).
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

// ---- split-K completion ----------------------------------------------------------
// A partial (for one query head) is an unnormalised output o[D] with its running max m
// (log2 units) and running sum l. Merging partials i: M = max m_i, w_i = 2^(m_i - M),
// o = sum w_i o_i, l = sum w_i l_i; the final row is o / l.

__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// The block ids of a split's chunk, loaded before the sequence length is known so that the two
// global loads overlap: entries first_blk .. of sequence b's table row that the chunk can reach
// whatever the length (clamped to the row), N per thread. Only the first n_blk, those the length
// reaches, are checked and kept (store): the others may be unused (-1) entries.
template <int N>
struct ChunkBlockIds {
  int id[N];
  __device__ __forceinline__ void load(const DecodeArgs& a, int b, int first_blk, int tid, int nthreads) {
    const int32_t* row = a.block_table + static_cast<size_t>(b) * a.max_blocks_per_seq + first_blk;
    const int reach = min(((a.chunk + (1 << a.log2_bs) - 1) >> a.log2_bs) + 1, a.max_blocks_per_seq - first_blk);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int i = tid + k * nthreads;
      id[k] = i < reach ? row[i] : 0;
    }
  }
  __device__ __forceinline__ void store(const DecodeArgs& a, int32_t* tbl, int n_blk, int tid, int nthreads) const {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int i = tid + k * nthreads;
      if (i < n_blk) {
        int v = id[k];
        if (v < 0 || v >= a.num_blocks) {
          flag_error(a.err, RRA_ERR_BLOCK_ID);
          v = 0;
        }
        tbl[i] = v;
      }
    }
  }
};

// Counts this CTA's arrival at `cnt` (all `nthreads` consumer threads call it after their
// last write). True in the CTA whose arrival brings the count to `target`; that CTA also puts
// the counter back to zero, ready for the next call. No CTA ever waits for another.
// Ordering: the barrier orders every thread's partial writes before thread 0's arrival, whose
// release makes them visible device-wide; its acquire (in the last CTA) and the second barrier
// order the other CTAs' partials before this CTA's merge reads (which bypass L1).
__device__ __forceinline__ bool arrive_last(int* cnt, int target, int* s_flag, int32_t* err, int tid,
                                            int nthreads) {
  named_barrier_sync(1, nthreads);
  if (tid == 0) {
    const int arrived = atomic_add_acq_rel_gpu(cnt, 1) + 1;
    int last = 0;
    if (arrived == target) {
      last = 1;
      atomicExch(cnt, 0);
    } else if (arrived > target) {  // the workspace did not start zeroed: results are invalid
      flag_error(err, RRA_ERR_WORKSPACE);
      atomicExch(cnt, 0);
    }
    *s_flag = last;
  }
  named_barrier_sync(1, nthreads);
  return *s_flag != 0;
}

// Partial row r is output row r (decode: rows b * Hq + h).
struct SameRow {
  __device__ size_t operator()(size_t r) const { return r; }
};

// Merges partials first .. first+count-1 of rows row0 .. row0+hpc-1 of a [rows][stride]
// partial array into the final output rows out_row(row0 + h) (dst_o == nullptr) or into one
// partial at index dst_idx of a [rows][dst_stride] partial array.
// EARLY: the partial outputs are fetched 16 at a time per thread, the first batch before the
// weights are known (one output item per thread, as the decode kernels have); otherwise 8 at a
// time after them (the verify kernel, with several items per thread, measured faster so).
template <typename T, int D, typename OutRow = SameRow, bool EARLY = true>
__device__ void merge_partials(const DecodeArgs& a, const float* src_o, const float* src_ml, int stride, int first,
                               int count, int hpc, size_t row0, float* dst_o, float* dst_ml, int dst_stride,
                               int dst_idx, float* scratch, int tid, int nthreads, OutRow out_row = OutRow()) {
  float* sm_w = scratch;                  // [hpc][count]: m_i, then the weights
  float* sm_l = scratch + hpc * count;    // [hpc][count]
  float* sm_ml = sm_l + hpc * count;      // [hpc][2]: merged (M, l)
  constexpr int kQ = D / 4;
  constexpr int kBatch = 16;              // o rows of partials one thread fetches at once
  const int n_items = hpc * kQ;           // (head, 4 dims) output items
  // The first batch of this thread's first item is fetched before the weights are known (it
  // does not depend on them), so its L2 round trip overlaps the (m, l) one.
  float4 pre[kBatch];
  if (EARLY && tid < n_items) {
    const int h = tid / kQ, d = (tid - h * kQ) * 4;
    const float4* o = reinterpret_cast<const float4*>(src_o + ((row0 + h) * stride + first) * D + d);
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      pre[k] = k < count ? __ldcg(o + static_cast<size_t>(k) * kQ) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i = tid; i < hpc * count; i += nthreads) {
    const int h = i / count, k = i - h * count;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(src_ml) + (row0 + h) * stride + first + k);
    sm_w[i] = ml.x;
    sm_l[i] = ml.y;
  }
  named_barrier_sync(1, nthreads);
  const bool final_row = dst_o == nullptr;
  const int warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < hpc; h += nthreads >> 5) {
    float M = -INFINITY;
    for (int k = lane; k < count; k += 32) M = fmaxf(M, sm_w[h * count + k]);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
    float ls = 0.f;
    if (M != -INFINITY)
      for (int k = lane; k < count; k += 32) ls = fmaf(exp2f(sm_w[h * count + k] - M), sm_l[h * count + k], ls);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, x);
    const float scale = final_row ? (ls > 0.f ? 1.f / ls : 0.f) : 1.f;
    __syncwarp();
    for (int k = lane; k < count; k += 32)
      sm_w[h * count + k] = M != -INFINITY ? exp2f(sm_w[h * count + k] - M) * scale : 0.f;
    if (lane == 0) {
      sm_ml[2 * h] = M;
      sm_ml[2 * h + 1] = ls;
    }
  }
  named_barrier_sync(1, nthreads);
  for (int i = tid; i < n_items; i += nthreads) {
    const int h = i / kQ, d = (i - h * kQ) * 4;
    const float4* o = reinterpret_cast<const float4*>(src_o + ((row0 + h) * stride + first) * D + d);
    const float* wts = sm_w + h * count;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float wv, const float4& v) {
      acc.x = fmaf(wv, v.x, acc.x);
      acc.y = fmaf(wv, v.y, acc.y);
      acc.z = fmaf(wv, v.z, acc.z);
      acc.w = fmaf(wv, v.w, acc.w);
    };
    if constexpr (!EARLY) {
#pragma unroll 8
      for (int k = 0; k < count; ++k) add(wts[k], __ldcg(o + static_cast<size_t>(k) * kQ));
    }
    int k0 = EARLY ? 0 : count;
    if (EARLY && i == tid) {  // the batch fetched ahead
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (k < count) add(wts[k], pre[k]);
      k0 = kBatch;
    }
    for (; k0 < count; k0 += kBatch) {  // all loads of a batch are issued before its FMAs
      float4 v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        v[k] = k0 + k < count ? __ldcg(o + static_cast<size_t>(k0 + k) * kQ) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (k0 + k < count) add(wts[k0 + k], v[k]);
    }
    if (final_row) {
      T* out = static_cast<T*>(a.out) + out_row(row0 + h) * D + d;
      Elem<T>::store(out, acc.x);
      Elem<T>::store(out + 1, acc.y);
      Elem<T>::store(out + 2, acc.z);
      Elem<T>::store(out + 3, acc.w);
    } else {
      const size_t pd = (row0 + h) * dst_stride + dst_idx;
      *reinterpret_cast<float4*>(dst_o + pd * D + d) = acc;
      if (d == 0) *reinterpret_cast<float2*>(dst_ml + 2 * pd) = make_float2(sm_ml[2 * h], sm_ml[2 * h + 1]);
    }
  }
}

// merge_partials with the partial o rows brought into shared memory by bulk copies: the `count`
// rows of one head are contiguous in the [rows][stride][D] array, so one copy per head moves
// them, all copies of a chunk of heads in flight at once instead of one L2 round trip per output
// item and batch. `scratch_bytes` of shared memory at `scratch` (16-byte aligned, free of pending
// copies) hold a barrier, the weights and as many heads' rows as fit, chunk after chunk of
// heads; returns false, having done nothing, when not even one head fits. (One CTA's bulk copies
// move a few tens of GB/s, so the gain is largest where the register path is weakest: many heads,
// many partials or few threads, as in the two-consumer-warp CTAs of a 128-split step.)
template <typename T, int D, typename OutRow = SameRow>
__device__ bool merge_partials_bulk(const DecodeArgs& a, const float* src_o, const float* src_ml, int stride, int first,
                                    int count, int hpc, size_t row0, float* dst_o, float* dst_ml, int dst_stride,
                                    int dst_idx, float* scratch, int scratch_bytes, int tid, int nthreads,
                                    OutRow out_row = OutRow()) {
  constexpr int kQ = D / 4;
  const int head_bytes = count * D * 4;
  const int w_floats = ((2 * hpc * count + 2 * hpc) + 3) & ~3;  // weights, sums, merged (M, l)
  const int o_off = 16 + w_floats * 4;                            // bytes: barrier, weights, rows
  const int chunk = (scratch_bytes - o_off) / head_bytes;         // heads per chunk
  if (chunk < 1) return false;
  uint64_t* bar = reinterpret_cast<uint64_t*>(scratch);
  float* sm_w = scratch + 4;                 // [hpc][count]: m_i, then the weights
  float* sm_l = sm_w + hpc * count;          // [hpc][count]
  float* sm_ml = sm_l + hpc * count;         // [hpc][2]
  float* obuf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(scratch) + o_off);
  const int warp = tid >> 5, lane = tid & 31;
  // the first chunk's copies go out before the (m, l) loads so that the round trips overlap
  auto issue = [&](int hA, int hB) {
    if (warp != 0) return;
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>((hB - hA) * head_bytes));
    __syncwarp();
    for (int h = hA + lane; h < hB; h += 32)
      bulk_g2s(obuf + static_cast<size_t>(h - hA) * count * D, src_o + ((row0 + h) * stride + first) * D,
               static_cast<uint32_t>(head_bytes), bar);
  };
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    // the partials were written through the generic proxy and acquired by the arrival counter
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  named_barrier_sync(1, nthreads);
  issue(0, min(chunk, hpc));
  for (int i = tid; i < hpc * count; i += nthreads) {
    const int h = i / count, k = i - h * count;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(src_ml) + (row0 + h) * stride + first + k);
    sm_w[i] = ml.x;
    sm_l[i] = ml.y;
  }
  named_barrier_sync(1, nthreads);
  const bool final_row = dst_o == nullptr;
  for (int h = warp; h < hpc; h += nthreads >> 5) {
    float M = -INFINITY;
    for (int k = lane; k < count; k += 32) M = fmaxf(M, sm_w[h * count + k]);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
    float ls = 0.f;
    if (M != -INFINITY)
      for (int k = lane; k < count; k += 32) ls = fmaf(exp2f(sm_w[h * count + k] - M), sm_l[h * count + k], ls);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, x);
    const float scale = final_row ? (ls > 0.f ? 1.f / ls : 0.f) : 1.f;
    __syncwarp();
    for (int k = lane; k < count; k += 32)
      sm_w[h * count + k] = M != -INFINITY ? exp2f(sm_w[h * count + k] - M) * scale : 0.f;
    if (lane == 0) {
      sm_ml[2 * h] = M;
      sm_ml[2 * h + 1] = ls;
    }
  }
  named_barrier_sync(1, nthreads);
  bool ok = true;
  uint32_t parity = 0;
  for (int hA = 0; hA < hpc; hA += chunk, parity ^= 1u) {
    const int hB = min(hpc, hA + chunk);
    if (hA > 0) issue(hA, hB);
    // every thread waits for the chunk; the vote keeps the threads on one path if a wait ran out
    ok = named_barrier_and(1, nthreads, mbar_wait(bar, parity));
    if (!ok) break;
    {
      for (int i = tid; i < (hB - hA) * kQ; i += nthreads) {
        const int hl = i / kQ, q = i - hl * kQ, h = hA + hl;
        const float4* o = reinterpret_cast<const float4*>(obuf + static_cast<size_t>(hl) * count * D) + q;
        const float* wts = sm_w + h * count;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < count; ++k) {
          const float4 v = o[k * kQ];
          const float wv = wts[k];
          acc.x = fmaf(wv, v.x, acc.x);
          acc.y = fmaf(wv, v.y, acc.y);
          acc.z = fmaf(wv, v.z, acc.z);
          acc.w = fmaf(wv, v.w, acc.w);
        }
        const int d = 4 * q;
        if (final_row) {
          T* out = static_cast<T*>(a.out) + out_row(row0 + h) * D + d;
          Elem<T>::store(out, acc.x);
          Elem<T>::store(out + 1, acc.y);
          Elem<T>::store(out + 2, acc.z);
          Elem<T>::store(out + 3, acc.w);
        } else {
          const size_t pd = (row0 + h) * dst_stride + dst_idx;
          *reinterpret_cast<float4*>(dst_o + pd * D + d) = acc;
          if (d == 0) *reinterpret_cast<float2*>(dst_ml + 2 * pd) = make_float2(sm_ml[2 * h], sm_ml[2 * h + 1]);
        }
      }
    }
    named_barrier_sync(1, nthreads);  // the chunk's rows are read before the next copies land
  }
  if (!ok && tid == 0) flag_error(a.err, RRA_ERR_TIMEOUT);
  if (tid == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
  return true;
}

// Run by all consumer threads of a CTA after each has written its share of this split's
// partial (index `split` of the [rows][num_splits] partial arrays). With n <= F splits
// (F = merge_fanin(num_splits)), the last split to arrive merges them all into the output. With
// more, splits form groups of F: the last arrival of each group merges the group into a level-2
// partial, and the last group to finish merges the level-2 partials into the output, so no
// single CTA has to read every split at the end of the kernel.
template <typename T, int D, typename OutRow = SameRow, bool EARLY = true>
__device__ __forceinline__ void finish_split_rows(const DecodeArgs& a, size_t row0, int hpc, int split, int n,
                                                  float* scratch, int* s_flag, int tid, int nthreads,
                                                  OutRow out_row = OutRow(), int scratch_bytes = 0) {
  const int S = a.num_splits, G = a.num_groups, F = merge_fanin(S);
  // scratch_bytes > 0: the partials come in by bulk copies when they fit (see merge_partials_bulk)
  auto merge = [&](const float* so, const float* sml, int stride, int first, int count, float* dst_o, float* dst_ml,
                   int dst_stride, int dst_idx, auto orow) {
    if (scratch_bytes > 0 && merge_partials_bulk<T, D>(a, so, sml, stride, first, count, hpc, row0, dst_o, dst_ml,
                                                       dst_stride, dst_idx, scratch, scratch_bytes, tid, nthreads, orow))
      return;
    merge_partials<T, D, decltype(orow), EARLY>(a, so, sml, stride, first, count, hpc, row0, dst_o, dst_ml, dst_stride,
                                                dst_idx, scratch, tid, nthreads, orow);
  };
  if (n <= F) {
    if (arrive_last(a.counters + row0, n, s_flag, a.err, tid, nthreads))
      merge(a.ws_o, a.ws_ml, S, 0, n, nullptr, nullptr, 0, 0, out_row);
    return;
  }
  const int grp = split / F, first = grp * F;
  const int gsize = min(F, n - first);
  if (!arrive_last(a.group_counters + row0 * G + grp, gsize, s_flag, a.err, tid, nthreads)) return;
  merge(a.ws_o, a.ws_ml, S, first, gsize, a.ws2_o, a.ws2_ml, G, grp, SameRow());
  const int groups = (n + F - 1) / F;
  if (arrive_last(a.counters + row0, groups, s_flag, a.err, tid, nthreads))
    merge(a.ws2_o, a.ws2_ml, G, 0, groups, nullptr, nullptr, 0, 0, out_row);
}

template <typename T, int D>
__device__ __forceinline__ void finish_split(const DecodeArgs& a, int b, int h0, int hpc, int split, int n,
                                             float* scratch, int* s_flag, int tid, int nthreads, int scratch_bytes = 0) {
  finish_split_rows<T, D>(a, static_cast<size_t>(b) * a.Hq + h0, hpc, split, n, scratch, s_flag, tid, nthreads,
                          SameRow(), scratch_bytes);
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

  int L = a.positions != nullptr ? a.positions[b] + 1 : a.seq_lens[b];
  if (L < 0 || L > a.capacity) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0)
      flag_error(a.err, a.positions != nullptr ? RRA_ERR_POSITION : RRA_ERR_SEQ_LEN);
    L = min(max(L, 0), a.capacity);
  }
  const int start = split * a.chunk;
  const int n_work = (L + a.chunk - 1) / a.chunk;  // splits of this sequence that hold tokens
  if (start >= L) {
    if (L == 0 && split == 0) {  // nothing to attend to: a zero row
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
    if (n_work == 1) {
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
  if (n_work > 1) {
    __shared__ int s_last;
    finish_split<T, D>(a, b, h0, HPC, split, n_work, reinterpret_cast<float*>(smem), &s_last, threadIdx.x,
                       kConsumers);
  }
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
