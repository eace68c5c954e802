// Prefill (causal attention of a prompt, or of a chunk of one after a cached prefix) on the
// fifth-generation tensor cores: tcgen05.mma with Q, K, V and P in shared memory and the score
// and output accumulators in Tensor Memory.
//
// "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南" §三: FlashAttention computes
// softmax(Q K^T / sqrt(d)) V block by block with a running max and sum, never forming the T x T
// score matrix. Token t of sequence b sits at position p_b + t, is already rotated and in the
// cache (the append kernel with gamma = T), and attends keys [0, p_b + t].
//
// One CTA owns NQ query tiles of 128 rows: the same 128 prompt tokens for NQ query heads of one
// KV group (NQ = 2 when the group has an even number of heads), so every K/V tile brought into
// shared memory serves NQ x 128 rows. Key tiles of 128 tokens stream through a three-slot ring
// (K_0, V_0, K_1, V_1, ... by TMA with the 128-byte swizzle). For query tile k and key tile j:
//   S_k = Q_k K_j^T   8 MMAs (M 128, N 128, K 16) into TMEM columns [128k, 128k + 128)
//   softmax           warpgroup k, one row per thread: the S row from TMEM into registers (one
//                     wait), causal mask on diagonal tiles, running max, P in bf16 to shared
//                     memory in the K-major 128-byte-swizzled layout
//   O_k += P_k V_j    8 MMAs (M 128, N 128, K 16; V as an MN-major operand: its two 64-dim
//                     halves are the N atoms) into TMEM columns [256 + 128k, 384 + 128k)
// One lane of the last warp issues every MMA in the order PV_0, S_0 (next tile), PV_1, S_1 (next
// tile), so the tensor cores work on one query tile while the other tile's softmax runs; the warp
// before it is the TMA producer. The running max only moves (and O and the sum are rescaled in
// TMEM) when it grows by more than 2^8, so P stays below 2^8. Rows that see fewer than 256 keys
// at the start of the block take P as a bf16 part plus the bf16 rounding of its remainder (two
// P.V passes), as the warp-level kernels do, keeping short rows' P to about 2^-17.
//
// Every wait is bounded (a timeout sets RRA_ERR_TIMEOUT and the roles drain); the MMA lane waits
// for all its MMAs and the producer for all its copies before the CTA releases Tensor Memory.
#pragma once

#include "decode_mma.cuh"
#include "tcgen05.cuh"

namespace rra {
namespace ptc {

constexpr int kRows = 128;                    // query rows per tile: M of every MMA
constexpr int kKeys = 128;                    // keys per tile
constexpr int kD = 128;                       // head dim
constexpr int kHalfBytes = 128 * 128;         // one 64-element half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalfBytes;    // a 128 x 128 bf16 tile
constexpr int kRing = 3;                      // K / V tile slots
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;           // move the running max only when it grows by more
constexpr int kPreciseKeys = 256;             // blocks whose first row sees fewer keys split P

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, false);   // Q (K-major) . K^T (K-major)
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, 128, true);   // P (K-major) . V (MN-major)

template <int NQ>
struct Cfg {
  static constexpr int kOffQ = 0;                            // NQ query tiles
  static constexpr int kOffRing = kOffQ + NQ * kTileBytes;   // kRing K / V slots
  static constexpr int kOffP = kOffRing + kRing * kTileBytes;  // NQ P tiles
  static constexpr int kOffBar = kOffP + NQ * kTileBytes;
  // q_full, ring_full[3], ring_empty[3], s_full[NQ], p_full[NQ], o_done[NQ], mma_done
  static constexpr int kNumBars = 1 + 2 * kRing + 3 * NQ + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = 1024 + kOffTmemSlot + 16;
  static constexpr int kSoftmaxThreads = 128 * NQ;
  static constexpr int kThreads = kSoftmaxThreads + 64;      // + producer warp + MMA warp
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// A bounded wait whose outcome every lane of the warp shares (the tcgen05 loads and stores that
// follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// Byte offset of 16-byte chunk `chunk16` (0..15: bf16 columns 8 chunk16 .. + 7) of row r of a
// 128 x 128 tile stored as two 64-column halves of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_chunk_offset(int r, int chunk16) {
  return (chunk16 >> 3) * kHalfBytes + r * 128 + (((chunk16 & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ float ex2(float x) {  // 2^x on the special-function unit (2^-inf = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The whole S row of this thread (128 columns: four 32-column loads, one wait).
__device__ __forceinline__ void ld_row(uint32_t taddr, float (&s)[kKeys]) {
  uint32_t v[kKeys / 32][32];
#pragma unroll
  for (int c = 0; c < kKeys / 32; ++c) tc::tmem_ld32(taddr + 32 * c, v[c]);
  tc::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < kKeys / 32; ++c)
#pragma unroll
    for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(v[c][i]);
}

__device__ __forceinline__ float row_max(const float (&s)[kKeys]) {
  float mx[8];  // independent chains
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
  for (int i = 8; i < kKeys; ++i) mx[i & 7] = fmaxf(mx[i & 7], s[i]);
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// 2^(S * scale_log2 - mref) of the row into its P row (K-major, swizzled), as bf16 (LO false;
// returns the row's sum) or as the bf16 rounding of what that leaves (LO true). Masked columns
// hold -inf and give 0.
template <bool LO>
__device__ __forceinline__ float row_probs(const float (&s)[kKeys], uint8_t* p_smem, int r, float sl, float mref) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains
#pragma unroll
  for (int q = 0; q < kKeys / 8; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 8 * q + 2 * e;
      const float e0 = ex2(fmaf(s[i], sl, -mref)), e1 = ex2(fmaf(s[i + 1], sl, -mref));
      const uint32_t hi = pack_bf16x2(e0, e1);
      if constexpr (LO) {
        w[e] = pack_bf16x2(e0 - __uint_as_float(hi << 16), e1 - __uint_as_float(hi & 0xffff0000u));
      } else {
        ls[e] += e0 + e1;
        w[e] = hi;
      }
    }
    *reinterpret_cast<uint4*>(p_smem + tile_chunk_offset(r, q)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

template <int NQ, bool PAGED>
__global__ void __launch_bounds__(Cfg<NQ>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  using C = Cfg<NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int T = a.gamma;
  const int n_qb = (T + kRows - 1) / kRows;
  // One CTA per (query block, head group). The GPU starts CTAs in index order: within a band of
  // KV groups whose K and V fit in L2 together, the longest causal blocks of all its head groups
  // come first (the short ones make the tail), then the next band.
  const int hg_band = (a.kv_band > 0 ? a.kv_band : a.Hkv) * ((a.Hq / a.Hkv) / NQ);  // head groups per band
  const int band_ctas = n_qb * hg_band;
  const int band = static_cast<int>(blockIdx.x) / band_ctas;
  const int j = static_cast<int>(blockIdx.x) - band * band_ctas;
  const int qb = n_qb - 1 - j / hg_band;
  const int h0 = (band * hg_band + j % hg_band) * NQ;  // query heads h0 .. h0 + NQ - 1, one KV group
  const int g = h0 / (a.Hq / a.Hkv);
  const int b = blockIdx.z;
  const int q0 = qb * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int producer_warp = 4 * NQ, mma_warp = 4 * NQ + 1;

  pdl_launch_dependents();
  pdl_wait();  // the append kernel before this one wrote the prompt's K, V and q_rot

  const int p0 = a.positions[b];
  if (p0 < 0 || p0 + T > a.capacity) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  const int q_end = min(T, q0 + kRows);
  const int end = p0 + q_end;                          // keys [0, end)
  const int n_tiles = (end + kKeys - 1) / kKeys;
  const int last_valid = end - (n_tiles - 1) * kKeys;  // keys of the last tile
  const int passes = p0 + q0 < kPreciseKeys ? 2 : 1;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* ring_full = bars + 1;
  uint64_t* ring_empty = ring_full + kRing;
  uint64_t* s_full = ring_empty + kRing;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_done = p_full + NQ;
  uint64_t* mma_done = o_done + NQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int k = 0; k < NQ; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], 128);
      mbar_init(&o_done[k], 1);
    }
    mbar_init(mma_done, 1);
    fence_barrier_init();
  }
  if (warp == mma_warp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
    tc::fence_before_sync();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // ring position r: K of tile r / 2 (r even) or its V (r odd), in slot r % 3
  auto slot_of = [](int r) { return r % kRing; };
  auto phase_of = [](int r) { return static_cast<uint32_t>((r / kRing) & 1); };

  if (warp == producer_warp) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      mbar_arrive_expect_tx(q_full, NQ * kTileBytes);
      for (int k = 0; k < NQ; ++k)
        for (int hf = 0; hf < 2; ++hf)
          tma_g2s_3d(smem + C::kOffQ + k * kTileBytes + hf * kHalfBytes, &q_map, 64 * hf, h0 + k, b * T + q0, q_full);
      const int bs = PAGED ? (1 << a.log2_bs) : 0;
      const int box = PAGED ? min(bs, 64) : 64;    // rows per TMA box, as the tensor maps were encoded
      const int32_t* row = PAGED ? a.block_table + static_cast<size_t>(b) * a.max_blocks_per_seq : nullptr;
      int issued = 0;
      for (int r = 0; r < 2 * n_tiles; ++r) {
        const int s = slot_of(r);
        if (r >= kRing && !mbar_wait(&ring_empty[s], phase_of(r) ^ 1u)) break;
        const CUtensorMap* map = (r & 1) ? &v_map : &k_map;
        uint8_t* dst = smem + C::kOffRing + s * kTileBytes;
        const int tile0 = (r >> 1) * kKeys;
        const int nbox = (min(kKeys, end - tile0) + box - 1) / box;
        mbar_arrive_expect_tx(&ring_full[s], static_cast<uint32_t>(nbox * box * 128 * 2));
        for (int bx = 0; bx < nbox; ++bx) {
          const int t = tile0 + bx * box;
          int phys = 0;
          if constexpr (PAGED) {
            phys = row[t >> a.log2_bs];
            if (phys < 0 || phys >= a.num_blocks) {
              flag_error(a.err, RRA_ERR_BLOCK_ID);
              phys = 0;
            }
          }
          for (int hf = 0; hf < 2; ++hf) {
            uint8_t* d = dst + hf * kHalfBytes + bx * box * 128;
            if constexpr (PAGED)
              tma_g2s_4d(d, map, 64 * hf, g, t & (bs - 1), phys, &ring_full[s]);
            else
              tma_g2s_3d(d, map, 64 * hf, t, b * a.Hkv + g, &ring_full[s]);
          }
        }
        issued = r + 1;
      }
      if (issued < 2 * n_tiles) flag_error(a.err, RRA_ERR_TIMEOUT);
      // no copy may still be landing when the CTA exits (the last kRing loads use distinct slots)
      mbar_wait(q_full, 0);
      for (int r = max(issued - kRing, 0); r < issued; ++r) mbar_wait(&ring_full[slot_of(r)], phase_of(r));
    }
  } else if (warp == mma_warp) {
    // ------------------------------------------------------------------ MMA issue (one lane)
    if (lane == 0) {
      const uint32_t q_base = smem_addr(smem + C::kOffQ), p_base = smem_addr(smem + C::kOffP);
      const uint32_t ring_base = smem_addr(smem + C::kOffRing);
      bool ok = mbar_wait(q_full, 0);
      // S_k of tile j; query tile 0 waits for K_j to land, the last one releases its slot
      auto issue_s = [&](int k, int j) -> bool {
        const int r = 2 * j;
        if (k == 0) {
          if (!mbar_wait(&ring_full[slot_of(r)], phase_of(r))) return false;
          tc::fence_after_sync();
        }
        const uint32_t k_base = ring_base + slot_of(r) * kTileBytes;
        const uint32_t qk = q_base + k * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          tc::mma_bf16_ss(tmem + k * kKeys, tc::sw128_desc(qk + off, 1024, 1024),
                          tc::sw128_desc(k_base + off, 1024, 1024), kIdescS, kk > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[k]);
        if (k == NQ - 1) tc::commit(&ring_empty[slot_of(r)]);
        return true;
      };
      for (int k = 0; ok && k < NQ; ++k) ok = issue_s(k, 0);
      int pv[NQ] = {};  // P.V passes issued per query tile
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int rv = 2 * j + 1;
        if (!mbar_wait(&ring_full[slot_of(rv)], phase_of(rv))) {
          ok = false;
          break;
        }
        const uint32_t v_base = ring_base + slot_of(rv) * kTileBytes;
        for (int k = 0; ok && k < NQ; ++k) {
          const uint32_t pk = p_base + k * kTileBytes;
          for (int u = 0; u < passes; ++u, ++pv[k]) {
            if (!mbar_wait(&p_full[k], pv[k] & 1)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              const uint64_t pd = tc::sw128_desc(pk + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 1024, 1024);
              tc::mma_bf16_ss(tmem + kColO + 128 * k, pd, tc::sw128_desc(v_base + kk * 2048, kHalfBytes, 1024),
                              kIdescPV, (j > 0 || u > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit(&o_done[k]);
          }
          if (!ok) break;
          if (k == NQ - 1) tc::commit(&ring_empty[slot_of(rv)]);
          if (j + 1 < n_tiles && !issue_s(k, j + 1)) ok = false;
        }
      }
      if (!ok) flag_error(a.err, RRA_ERR_TIMEOUT);
      tc::commit(mma_done);  // every MMA issued above has completed once this arrives
      mbar_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------------ softmax: thread = row
    const int k = warp >> 2;                       // query tile of this warpgroup
    const int r = threadIdx.x & 127;               // row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t s_col = tmem + lane_base + k * kKeys, o_col = tmem + lane_base + kColO + 128 * k;
    const int tok = q0 + r;
    const int lim = min(p0 + tok, end - 1);        // last key this row attends
    const int lim_min = p0 + q0;                   // the block's smallest limit: tiles past it need the mask
    uint8_t* p_smem = smem + C::kOffP + k * kTileBytes;
    const float sl = a.scale_log2;
    float m_use = -INFINITY, l = 0.f;              // running max (log2 units) and sum
    int pv = 0;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(&s_full[k], j & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const bool diag = (j + 1) * kKeys - 1 > lim_min;  // keys past some row's limit: mask them
      const int nvis = lim - j * kKeys + 1;
      auto load_s = [&](float (&sv)[kKeys]) {
        ld_row(s_col, sv);
        if (diag) {
#pragma unroll
          for (int i = 0; i < kKeys; ++i) sv[i] = i < nvis ? sv[i] : -INFINITY;
        }
      };
      // the previous P.V pass has read the P buffer and O is stable
      auto wait_pv = [&]() -> bool {
        if (pv == 0) return true;
        if (!warp_wait(&o_done[k], (pv - 1) & 1)) return false;
        tc::fence_after_sync();
        return true;
      };
      float alpha = 1.f;
      bool rescale = false;
      {
        float sv[kKeys];
        load_s(sv);
        const float m_new = fmaxf(m_use, row_max(sv) * sl);
        rescale = m_new > m_use + kRescaleLog2;  // also the first finite max
        if (rescale) {
          alpha = ex2(m_use - m_new);
          m_use = m_new;
        }
        const float mref = m_use == -INFINITY ? 0.f : m_use;
        if (!wait_pv()) {
          ok = false;
          break;
        }
        if (k == 0 && j == n_tiles - 1 && last_valid < kKeys) {
          // keys past the end of the prompt: their V rows (stale or poisoned) become zeros so that
          // 0 * V stays 0 in the tensor core (query tile 0's P.V reads this V first)
          const int rv = 2 * j + 1;
          if (!warp_wait(&ring_full[slot_of(rv)], phase_of(rv))) {
            ok = false;
            break;
          }
          if (r >= last_valid) {
            uint8_t* vrow = smem + C::kOffRing + slot_of(rv) * kTileBytes + r * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              *reinterpret_cast<uint4*>(vrow + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(vrow + kHalfBytes + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        l = l * alpha + row_probs<false>(sv, p_smem, r, sl, mref);  // the bf16 part of P
      }
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {  // O rows whose max moved (warp-collective; alpha = 1 elsewhere)
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
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      mbar_arrive(&p_full[k]);
      ++pv;
      if (passes == 2) {  // short rows: the remainder of P in a second pass (S is still in TMEM)
        if (!wait_pv()) {
          ok = false;
          break;
        }
        float sv[kKeys];
        load_s(sv);
        row_probs<true>(sv, p_smem, r, sl, m_use == -INFINITY ? 0.f : m_use);
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        mbar_arrive(&p_full[k]);
        ++pv;
      }
      if (!ok) break;
    }
    // ------------------------------------------------------------------ epilogue: O / l
    if (ok && warp_wait(&o_done[k], (pv - 1) & 1)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                            ((static_cast<size_t>(b) * T + min(tok, T - 1)) * a.Hq + h0 + k) * kD);
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(o_col + 32 * c, v);
        tc::tmem_wait_ld();
        if (tok < T) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            out[4 * c + i] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                                        pack_bf16x2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                                        pack_bf16x2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                                        pack_bf16x2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
        }
      }
    } else {
      flag_error(a.err, RRA_ERR_TIMEOUT);
    }
    tc::fence_before_sync();
  }
  __syncthreads();
  if (warp == mma_warp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NQ, bool PAGED>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                     cudaStream_t st) {
  using C = Cfg<NQ>;
  static int done[64] = {0};
  auto kern = prefill_tc_kernel<NQ, PAGED>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(((a.gamma + kRows - 1) / kRows) * (a.Hq / NQ), 1, a.B);
  return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, st, qm, km, vm, a);
}

// Two query heads per CTA when every KV group has an even number of them, else one.
template <bool PAGED>
cudaError_t launch(const DecodeArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                   cudaStream_t st) {
  return ((a.Hq / a.Hkv) % 2 == 0) ? launch_t<2, PAGED>(a, qm, km, vm, st) : launch_t<1, PAGED>(a, qm, km, vm, st);
}

}  // namespace ptc
}  // namespace rra
