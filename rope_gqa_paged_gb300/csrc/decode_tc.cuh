// Split-K decode attention for query groups of 16 to 128 heads (MQA-like GQA) on the
// fifth-generation tensor cores: one CTA serves every query head of one KV head, so each K/V
// tile is read from L2 or HBM once for the whole group.
//
// "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南" §六 (GQA: n_rep query heads
// share one KV head; n_kv = 1 is MQA), "Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践"
// §2.1, §2.2, §4.2 (softmax(q K^T / sqrt(d)) V, blockwise with a running max and sum).
//
// The 128 rows of the M dimension hold 128 / R copies of the group's query heads (R = 32, 64 or
// 128: the group size rounded up; rows past the group are zero). Copy c owns tokens
// [c R, c R + R) of every key tile; key tiles of 128 tokens stream through a ring of K and V tiles
// (TMA, 128-byte swizzle, 64-dim halves; paged blocks gathered per block). For key tile j:
//   S_(j%2) = Q K_j^T    8 MMAs (M 128, N 128, K 16) into TMEM columns [128 (j%2), + 128), Q
//                        (bf16 pairs) the A operand from TMEM columns [384, 448)
//   softmax              warps 0-3, one row per thread: the R S columns of the row's copy from
//                        TMEM, running max (moved only when it grows by more than 2^8), P as bf16
//                        pairs over the first 64 columns of S_(j%2) (zeros in the columns of the
//                        other copies)
//   O += P V_j           8 MMAs, P the A operand from TMEM, V an MN-major operand in shared
//                        memory, into TMEM columns [256, 384)
// so the O rows of copy c accumulate that copy's share of every tile, and a group of 32 heads
// spreads its softmax over the four warps (32 columns per thread) instead of running whole
// 128-column rows in one. The copies' running max, sum and O rows merge in shared memory when
// the split ends.
// One lane of warp 5 issues the MMAs in the order S_0, S_1, PV_0, S_2, PV_1, ..., so the tensor
// core computes the next tile's scores while the softmax of this one runs (S_(j+2) overwrites
// P_j after PV_j, which reads it, in issue order); warp 4 is the TMA
// producer. The split's partial (o unnormalised, running max and sum per head) goes to the
// workspace and the splits merge as in the other decode kernels (finish_split); a sequence with
// one split writes its rows directly.
//
// Fused step (FUSED): the softmax threads rotate their own query row at the new token's
// position (sin / cos of pos * theta_i in float64 once per CTA, error-free float32 rotation)
// before writing it into the Q tile, split 0 publishes q_rot, and the CTA whose chunk holds the
// new token appends it (one warp) before its producer loads the tile that holds it.
//
// Every wait is bounded (a timeout sets RRA_ERR_TIMEOUT and the roles drain); the MMA lane waits
// for its last commit and the producer for its last copies before Tensor Memory is released.
#pragma once

#include "decode_kernels.cuh"
#include "decode_mma.cuh"
#include "tcgen05.cuh"

// K / V tile slots of 32 KB. Q and P live in Tensor Memory, so six slots (three key tiles, 192 KB
// in flight per SM) fit next to the barriers and the block table.
#ifndef RRA_TC_RING
#define RRA_TC_RING 6
#endif

namespace rra {
namespace dtc {

constexpr int kRows = 128;                    // M of every MMA: the query heads of the group
constexpr int kTile = 128;                    // tokens per key tile
constexpr int kD = 128;                       // head dim
constexpr int kHalfBytes = 128 * 128;         // one 64-element half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalfBytes;    // a 128 x 128 bf16 tile
constexpr int kRing = RRA_TC_RING;            // K / V tile slots (K_0, V_0, K_1, V_1, ...)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;               // O: columns [256, 384)
constexpr uint32_t kColQ = 384;               // Q as bf16 pairs: columns [384, 448)
constexpr float kRescaleLog2 = 8.f;           // move the running max only when it grows by more

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, false);   // Q (K-major) . K^T (K-major)
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, 128, true);   // P (K-major) . V (MN-major)

constexpr int kOffRing = 0;
constexpr int kOffBar = kOffRing + kRing * kTileBytes;
// q_ready, ring_full[kRing], ring_empty[kRing], s_full[2], p_full, o_done, mma_done, appended
constexpr int kNumBars = 1 + 2 * kRing + 2 + 3 + 1;
constexpr int kOffTable = kOffBar + kNumBars * 8;
constexpr int kOffCs = kOffTable + kMmaTableEntries * 4;
constexpr int kOffTmemSlot = kOffCs + 4 * (kD / 2) * 4;
constexpr int kSmemBytes = 1024 + kOffTmemSlot + 16;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kThreads = kSoftmaxThreads + 64;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert((kRows * kD + 2 * kRows) * 4 <= kRing * kTileBytes, "the copy merge's scratch fits the ring");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ float ex2(float x) {  // 2^x on the special-function unit (2^-inf = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// N columns of this thread's S row from column address taddr (N / 32 loads, one wait).
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&s)[N]) {
  uint32_t v[N / 32][32];
#pragma unroll
  for (int c = 0; c < N / 32; ++c) tc::tmem_ld32(taddr + 32 * c, v[c]);
  tc::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < N / 32; ++c)
#pragma unroll
    for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(v[c][i]);
}

// N columns of this thread's row from registers (N = 16, 32 or 64).
template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 16) {
    tc::tmem_st16(taddr, v);
  } else {
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
      uint32_t t[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) t[i] = v[32 * h + i];
      tc::tmem_st32(taddr + 32 * h, t);
    }
  }
}

template <bool PAGED, bool FUSED, int R>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                     const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  static_assert(R == 32 || R == 64 || R == 128, "rows per copy of the query group");
  constexpr int kCopies = kRows / R;
  const int n_rep = a.Hq / a.Hkv;   // heads of the group (<= R)
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int h0 = g * n_rep;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_launch_dependents();
  pdl_wait();

  int L;
  if constexpr (FUSED) {
    const int pos = a.positions[b];
    if (pos < 0 || pos >= a.capacity) {
      if (threadIdx.x == 0 && split == 0 && g == 0) flag_error(a.err, RRA_ERR_POSITION);
      return;
    }
    L = pos + 1;
  } else {
    L = a.seq_lens[b];
    if (L < 0 || L > a.capacity) {
      if (threadIdx.x == 0 && split == 0 && g == 0) flag_error(a.err, RRA_ERR_SEQ_LEN);
      L = min(max(L, 0), a.capacity);
    }
  }
  const int start = split * a.chunk;
  const int n_work = (L + a.chunk - 1) / a.chunk;  // splits of this sequence that hold tokens
  if (start >= L) {
    if (L == 0 && split == 0) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(b) * a.Hq + h0) * kD;
      for (int i = threadIdx.x; i < n_rep * kD; i += blockDim.x) out[i] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int end = min(L, start + a.chunk);
  const int n_tiles = (end - start + kTile - 1) / kTile;
  const int last_valid = end - start - (n_tiles - 1) * kTile;  // tokens of the last tile
  const bool appender = FUSED && end == L;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_ready = bars;
  uint64_t* ring_full = bars + 1;
  uint64_t* ring_empty = ring_full + kRing;
  uint64_t* s_full = ring_empty + kRing;   // [2]
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* mma_done = o_done + 1;
  uint64_t* appended = mma_done + 1;
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + kOffTable);
  float* cs = reinterpret_cast<float*>(smem + kOffCs);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  if (threadIdx.x == 0) {
    mbar_init(q_ready, kSoftmaxThreads);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, kSoftmaxThreads);
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    mbar_init(appended, 1);
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
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
    tc::fence_before_sync();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // ring position r: K of tile r / 2 (r even) or its V (r odd), in slot r % kRing
  auto slot_of = [](int r) { return r % kRing; };
  auto phase_of = [](int r) { return static_cast<uint32_t>((r / kRing) & 1); };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
    const int bs = PAGED ? (1 << a.log2_bs) : 0;
    const int box = PAGED ? min(bs, kTile) : kTile;  // rows per TMA box, as the tensor maps were encoded
    int issued = 0;
    for (int r = 0; r < 2 * n_tiles; ++r) {
      const int s = slot_of(r);
      const int tile0 = start + (r >> 1) * kTile;
      const int nbox = (min(kTile, end - tile0) + box - 1) / box;
      int ok = 1;
      if (lane == 0) {
        if (r >= kRing && !mbar_wait(&ring_empty[s], phase_of(r) ^ 1u)) {
          ok = 0;
        } else if (appender && (r >> 1) == n_tiles - 1 && !mbar_wait(appended, 0)) {  // the new token's tile
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&ring_full[s], static_cast<uint32_t>(nbox * box * 128 * 2));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const CUtensorMap* map = (r & 1) ? &v_map : &k_map;
      uint8_t* dst = smem + kOffRing + s * kTileBytes;
      for (int c = lane; c < 2 * nbox; c += 32) {  // (box, half) copies, from all lanes at once
        const int bx = c >> 1, hf = c & 1;
        const int t = tile0 + bx * box;
        uint8_t* d = dst + hf * kHalfBytes + bx * box * 128;
        if constexpr (PAGED)
          tma_g2s_4d(d, map, 64 * hf, g, t & (bs - 1), tbl[(t >> a.log2_bs) - first_blk], &ring_full[s]);
        else
          tma_g2s_3d(d, map, 64 * hf, t, b * a.Hkv + g, &ring_full[s]);
      }
      __syncwarp();
      issued = r + 1;
    }
    if (lane == 0) {
      if (issued < 2 * n_tiles) flag_error(a.err, RRA_ERR_TIMEOUT);
      // no copy may still be landing when the CTA exits
      for (int r = max(issued - kRing, 0); r < issued; ++r) mbar_wait(&ring_full[slot_of(r)], phase_of(r));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue (one lane)
    if (lane == 0) {
      const uint32_t ring_base = smem_addr(smem + kOffRing);
      bool ok = mbar_wait(q_ready, 0);
      tc::fence_after_sync();
      auto issue_s = [&](int j) -> bool {
        const int r = 2 * j;
        if (!mbar_wait(&ring_full[slot_of(r)], phase_of(r))) return false;
        tc::fence_after_sync();
        const uint32_t k_base = ring_base + slot_of(r) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          tc::mma_bf16_ts(tmem + kTile * (j & 1), tmem + kColQ + 8 * kk, tc::sw128_desc(k_base + off, 1024, 1024),
                          kIdescS, kk > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[j & 1]);
        tc::commit(&ring_empty[slot_of(r)]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n_tiles > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int rv = 2 * j + 1;
        if (!mbar_wait(&ring_full[slot_of(rv)], phase_of(rv)) || !mbar_wait(p_full, j & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t v_base = ring_base + slot_of(rv) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)  // P_j: bf16 pairs over S_(j%2)
          tc::mma_bf16_ts(tmem + kColO, tmem + kTile * (j & 1) + 8 * kk,
                          tc::sw128_desc(v_base + kk * 2048, kHalfBytes, 1024), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        tc::commit(o_done);
        tc::commit(&ring_empty[slot_of(rv)]);
        // the softmax of tile j has read S_(j%2): tile j + 2 may overwrite it
        if (j + 2 < n_tiles && !issue_s(j + 2)) ok = false;
      }
      if (!ok) flag_error(a.err, RRA_ERR_TIMEOUT);
      tc::commit(mma_done);  // every MMA issued above has completed once this arrives
      mbar_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------------ softmax: thread = query head
    const int r = threadIdx.x;                     // row = TMEM lane
    const int copy = kCopies == 1 ? 0 : r / R;    // copy of the group
    const int hr = r - copy * R;                   // head h0 + hr
    const int col0 = copy * R;                     // first token (S column) of the copy
    const bool real = hr < n_rep;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t o_col = tmem + lane_base + kColO;
    // the query row into the Q tile (K-major, swizzled): rotated here in the fused step
    {
      uint4 qv[kD / 8];
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                        (static_cast<size_t>(b) * a.Hq + h0 + (real ? hr : 0)) * kD);
#pragma unroll
      for (int c = 0; c < kD / 8; ++c) qv[c] = real ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (FUSED) {
        const int pos = L - 1;
        // the appending warp fetches the new token's k and v and its block id while sin / cos run
        const bool app_warp = appender && warp == 1;
        uint32_t kraw[kD / 64], vraw[kD / 64];
        int phys = 0;
        if (app_warp) {
          const size_t off = (static_cast<size_t>(b) * a.Hkv + g) * kD + lane * (kD / 32);
          const uint32_t* kn = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.k_new) + off);
          const uint32_t* vn = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.v_new) + off);
#pragma unroll
          for (int w = 0; w < kD / 64; ++w) {
            kraw[w] = kn[w];
            vraw[w] = vn[w];
          }
          if constexpr (PAGED) phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
        }
        if (r < kD / 2) {
          rope_cos_sin(pos, a.rope_phi[r], cs[r], cs[kD / 2 + r], cs[kD + r], cs[3 * (kD / 2) + r]);
        }
        named_barrier_sync(1, kSoftmaxThreads);
        // rotate the row (16-byte chunks c of 8 dims; half-split pairs (i, i + D/2) are chunks c and c + 8)
        auto w2f = [](uint32_t w, float& lo, float& hi) {
          lo = __uint_as_float(w << 16);
          hi = __uint_as_float(w & 0xffff0000u);
        };
        auto rot = [&](float x, float y, int i) {  // x cos_i - y sin_i
          return rotate_diff(x, y, cs[i], cs[kD / 2 + i], cs[kD + i], cs[3 * (kD / 2) + i]);
        };
        if (a.rope_style == 1) {  // interleaved pairs (2i, 2i + 1): the two halves of each 32-bit word
#pragma unroll
          for (int c = 0; c < kD / 8; ++c) {
            uint32_t* w = reinterpret_cast<uint32_t*>(&qv[c]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x0, x1;
              w2f(w[e], x0, x1);
              const int i = 4 * c + e;
              w[e] = pack_bf16x2(rot(x0, x1, i), rot(x1, -x0, i));
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < kD / 16; ++c) {
            uint32_t* wa = reinterpret_cast<uint32_t*>(&qv[c]);
            uint32_t* wb = reinterpret_cast<uint32_t*>(&qv[c + kD / 16]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float a0, a1, b0, b1;
              w2f(wa[e], a0, a1);
              w2f(wb[e], b0, b1);
              const int i = 8 * c + 2 * e;
              wa[e] = pack_bf16x2(rot(a0, b0, i), rot(a1, b1, i + 1));
              wb[e] = pack_bf16x2(rot(b0, -a0, i), rot(b1, -a1, i + 1));
            }
          }
        }
        if (real && copy == 0 && split == 0) {  // publish q_rot (rounded to bf16, as used here)
          uint4* qo = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.q_out) +
                                               (static_cast<size_t>(b) * a.Hq + h0 + hr) * kD);
#pragma unroll
          for (int c = 0; c < kD / 8; ++c) qo[c] = qv[c];
        }
        if (app_warp) append_token_bf16<kD, PAGED>(a, cs, kraw, vraw, phys, b, g, pos, lane, appended);
      }
      {  // the row into Tensor Memory: dims (2c, 2c + 1) in column kColQ + c
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(qv);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t t[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = qw[32 * h + i];
          tc::tmem_st32(tmem + lane_base + kColQ + 32 * h, t);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
      }
      mbar_arrive(q_ready);
    }
    const float sl = a.scale_log2;
    float m_use = -INFINITY, l = 0.f;  // running max (log2 units) and sum
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(&s_full[j & 1], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const int nvalid = j == n_tiles - 1 ? last_valid : kTile;
      float sv[R];
      ld_cols<R>(tmem + lane_base + kTile * (j & 1) + col0, sv);
      if (nvalid < col0 + R) {
#pragma unroll
        for (int i = 0; i < R; ++i) sv[i] = col0 + i < nvalid ? sv[i] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = sv[i];
#pragma unroll
      for (int i = 8; i < R; ++i) mx[i & 7] = fmaxf(mx[i & 7], sv[i]);
      const float rmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m_use, rmax * sl);
      const bool rescale = m_new > m_use + kRescaleLog2;  // also the first finite max
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m_use - m_new);
        m_use = m_new;
      }
      const float mref = m_use == -INFINITY ? 0.f : m_use;
      // the previous P.V has read the P tile and O is stable
      if (j > 0) {
        if (!warp_wait(o_done, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
      }
      if (j == n_tiles - 1 && nvalid < kTile) {
        // tokens past the chunk's end: their V rows (stale, poisoned or another split's) become
        // zeros so that 0 * V stays 0 in the tensor core
        const int rv = 2 * j + 1;
        if (!warp_wait(&ring_full[slot_of(rv)], phase_of(rv))) {
          ok = false;
          break;
        }
        if (r >= nvalid) {
          uint8_t* vrow = smem + kOffRing + slot_of(rv) * kTileBytes + r * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            *reinterpret_cast<uint4*>(vrow + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(vrow + kHalfBytes + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pw[R / 2];  // P of the copy's tokens as bf16 pairs
#pragma unroll
      for (int q = 0; q < R / 8; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 8 * q + 2 * e;
          const float e0 = ex2(fmaf(sv[i], sl, -mref)), e1 = ex2(fmaf(sv[i + 1], sl, -mref));
          ls[e] += e0 + e1;
          pw[4 * q + e] = pack_bf16x2(e0, e1);
        }
      }
      {  // P_j over the first 64 columns of S_(j%2): this copy's pairs, zeros in the others'
        const uint32_t pcol = tmem + lane_base + kTile * (j & 1);
#pragma unroll
        for (int c = 0; c < kCopies; ++c) {
          uint32_t t[R / 2];
#pragma unroll
          for (int i = 0; i < R / 2; ++i) t[i] = c == copy ? pw[i] : 0u;
          st_cols<R / 2>(pcol + c * (R / 2), t);
        }
      }
      l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {  // O rows whose max moved (alpha = 1 elsewhere)
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t v[32];
          tc::tmem_ld32(o_col + 32 * c, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tc::tmem_st32(o_col + 32 * c, v);
        }
        tc::tmem_wait_st();
      }
      tc::tmem_wait_st();
      tc::fence_smem_to_async();  // the zeroed V rows of a partial last tile, for the MMA's reads
      tc::fence_before_sync();
      mbar_arrive(p_full);
    }
    // ------------------------------------------------------------------ epilogue: this split's rows
    const bool done = ok && warp_wait(o_done, (n_tiles - 1) & 1);  // warp-uniform
    if (!done) flag_error(a.err, RRA_ERR_TIMEOUT);
    if constexpr (kCopies == 1) {
      if (done) {
        tc::fence_after_sync();
        const size_t bh = static_cast<size_t>(b) * a.Hq + h0 + r;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t v[32];
          tc::tmem_ld32(o_col + 32 * c, v);
          tc::tmem_wait_ld();
          if (!real) continue;
          if (n_work == 1) {
            uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + bh * kD) + 4 * c;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              out[i] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                                  pack_bf16x2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                                  pack_bf16x2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                                  pack_bf16x2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
          } else {
            float4* po = reinterpret_cast<float4*>(a.ws_o + (bh * a.num_splits + split) * kD) + 8 * c;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              po[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                  __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        }
        if (real && n_work > 1)
          *reinterpret_cast<float2*>(a.ws_ml + 2 * (bh * a.num_splits + split)) = make_float2(m_use, l);
      }
    } else {
      // merge the copies of each head: O rows scaled to the common max go through shared memory
      // (the ring: every copy has landed and every MMA has read it by now), float4 column group
      // q of row x at slot (q + x) % 32 so that eight consecutive rows hit distinct banks
      float* xo = reinterpret_cast<float*>(smem + kOffRing);  // [128 rows][kD]
      float* xm = xo + kRows * kD;                             // [128] running max
      float* xl = xm + kRows;                                  // [128] running sum
      xm[r] = done ? m_use : -INFINITY;
      xl[r] = done ? l : 0.f;
      named_barrier_sync(1, kSoftmaxThreads);
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kCopies; ++c) M = fmaxf(M, xm[c * R + hr]);
      const float wself = (done && m_use != -INFINITY) ? ex2(m_use - M) : 0.f;
      if (done) tc::fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t v[32];
        if (done) {
          tc::tmem_ld32(o_col + 32 * c, v);
          tc::tmem_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = done ? make_float4(__uint_as_float(v[4 * i]) * wself, __uint_as_float(v[4 * i + 1]) * wself,
                                              __uint_as_float(v[4 * i + 2]) * wself, __uint_as_float(v[4 * i + 3]) * wself)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(xo + r * kD + 4 * ((8 * c + i + r) & 31)) = x;
        }
      }
      named_barrier_sync(1, kSoftmaxThreads);
      if (copy == 0 && real) {  // one thread per head sums the copies
        float L = 0.f;
#pragma unroll
        for (int c = 0; c < kCopies; ++c) {
          const float mc = xm[c * R + hr];
          if (mc != -INFINITY) L = fmaf(ex2(mc - M), xl[c * R + hr], L);
        }
        const size_t bh = static_cast<size_t>(b) * a.Hq + h0 + hr;
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
        for (int q = 0; q < kD / 4; ++q) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kCopies; ++c) {
            const int x = c * R + hr;
            const float4 y = *reinterpret_cast<const float4*>(xo + x * kD + 4 * ((q + x) & 31));
            acc.x += y.x;
            acc.y += y.y;
            acc.z += y.z;
            acc.w += y.w;
          }
          if (n_work == 1) {
            uint2* out = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + bh * kD) + q;
            *out = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
          } else {
            reinterpret_cast<float4*>(a.ws_o + (bh * a.num_splits + split) * kD)[q] = acc;
          }
        }
        if (n_work > 1) *reinterpret_cast<float2*>(a.ws_ml + 2 * (bh * a.num_splits + split)) = make_float2(M, L);
      }
    }
    tc::fence_before_sync();
    if (n_work > 1) {  // the last split of this (sequence, KV head) merges the partials
      __shared__ int s_last;
      // scratch: the ring (every copy has landed and every MMA has read it by now)
      finish_split<__nv_bfloat16, kD>(a, b, h0, n_rep, split, n_work, reinterpret_cast<float*>(smem + kOffRing),
                                      &s_last, threadIdx.x, kSoftmaxThreads, kRing * kTileBytes);
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool PAGED, bool FUSED, int R>
cudaError_t launch_r(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t st) {
  static int done[64] = {0};
  auto kern = decode_tc_kernel<PAGED, FUSED, R>;
  cudaError_t e = ensure_smem(kern, kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_splits, a.Hkv, a.B);
  return launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, st, km, vm, a);
}

// Rows per copy of the query group: the group size rounded up to 32, 64 or 128.
template <bool PAGED, bool FUSED>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t st) {
  const int n_rep = a.Hq / a.Hkv;
  if (n_rep <= 32) return launch_r<PAGED, FUSED, 32>(a, km, vm, st);
  if (n_rep <= 64) return launch_r<PAGED, FUSED, 64>(a, km, vm, st);
  return launch_r<PAGED, FUSED, 128>(a, km, vm, st);
}

}  // namespace dtc
}  // namespace rra
