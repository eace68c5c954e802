// Split-K GQA decode attention for bf16 caches on the tensor cores (mma.sync m16n8k16).
//
// Same math and split/merge structure as decode_kernels.cuh ("Transformer推理核心：KV Cache、
// GQA与RoPE原理与工程实践" §2.1, §2.2, §4.2; "Transformer架构优化实战2026：注意力机制、KV
// Cache与推理加速完整指南" §三, §四), with the two contractions of a stage on the tensor cores:
//
//   S^T [16 tokens x 8 heads]  = K [16 tokens x D] . Q^T [D x 8 heads]       (D/16 mma)
//   O^T [D x 8 heads]         += V^T [D x 16 tokens] . P [16 tokens x 8 heads] (D/16 mma)
//
// Tokens sit on M and the CTA's query heads (up to 8 of one KV head's group, zero-padded)
// on N, so a warp keeps only O^T (D/16 fragments of 4 floats) and the scores of 16 tokens
// in registers. The softmax works on the score fragment directly (each lane owns two heads
// and two tokens of every 16); the probabilities go back to the tensor cores as the B
// operand after one movmatrix transpose per 8x8 half, never touching shared memory.
//
// Data path: the producer warp streams K and V tiles with 4-D (paged pool) or 3-D
// (contiguous cache) TMA tensor copies using the 128-byte swizzle, in 64-dim halves, into a
// 2-stage ring (three CTAs per SM); each consumer warp reads its 16-token slices with ldmatrix (K as the A
// operand, V through ldmatrix.trans as V^T), conflict-free thanks to the swizzle.
#pragma once

#include "decode_kernels.cuh"
#include "rra_device.cuh"
#include "rra_internal.h"

namespace rra {

// Two 32 KB stages per CTA and three CTAs per SM (registers <= 136, ~68 KB shared memory
// each): measured faster on GB300 than three stages at two CTAs per SM, because more CTAs
// per SM overlap one CTA's start-up and epilogue with the others' streaming.
#ifndef RRA_MMA_STAGES
#define RRA_MMA_STAGES 2
#endif
#ifndef RRA_MMA_CTAS_PER_SM
#define RRA_MMA_CTAS_PER_SM 3
#endif
// Lanes of the producer warp that issue a stage's TMA copies together (a stage of 16-token
// blocks is 16 copies): measured 2.6 % faster on the batch-64 step and 9 % on the MQA sweep than
// one lane issuing them in turn.
#ifndef RRA_MMA_ISSUE_LANES
#define RRA_MMA_ISSUE_LANES 32
#endif

template <int D>
struct MmaCfg {
  static constexpr int kRowBytes = D * 2;                 // bf16
  static constexpr int kHalves = D / 64;                  // 128-byte swizzle spans per row
  static constexpr int kTile = 16384 / kRowBytes;         // tokens per stage (K 16 KB + V 16 KB)
  static constexpr int kStages = RRA_MMA_STAGES;
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kWarpTokens = kTile / kConsumerWarps;
  static constexpr int kSteps = kWarpTokens / 16;         // 16-token mma steps per warp per stage
  static constexpr int kHalfBytes = kTile * 128;          // one 64-dim half of K or V of a stage
  static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  // after the ring: full[kStages], empty[kStages], appended (8 bytes each), the block-id
  // table, and cos/sin hi/lo [4][D/2] floats for the fused step
  static constexpr int kOffBar = kRingBytes;
  static constexpr int kOffTable = kOffBar + (2 * kStages + 1) * 8;
  static constexpr int kOffCs = kOffTable + kMmaTableEntries * 4;
  static constexpr int kSmemBytes = 1024 + kOffCs + 4 * (D / 2) * 4;
  static constexpr int kMaxHeads = 8;
  static constexpr int kKSteps = D / 16;
};

// The decode kernel with NT 8-head n-tiles per CTA (up to 8 * NT query heads of one KV head's
// group): NT = 2 serves 16 heads from every K/V tile (groups of 16 or more heads stream the KV half
// as often as with 8 heads per CTA); its larger register state runs at two CTAs per SM, with a
// 3-stage ring so that an SM still keeps 192 KB of K/V in flight.
//
// NARROW (head_dim 128, NT 1): two consumer warps, 32-token stages (16 KB) in a 3-stage ring and
// four CTAs per SM (608 on 152 SMs instead of 456), for grids of few sequences cut into more
// splits than one wave holds (a 128-split 128K step: 1024 CTAs in 1.7 waves instead of 2.25, the
// second wave of 416 CTAs still keeping 20 MB of K/V in flight).
template <int D, int NT, bool NARROW = false>
struct MmaCfgN : MmaCfg<D> {
  using B = MmaCfg<D>;
  static constexpr int kConsumerWarps = NARROW ? 2 : B::kConsumerWarps;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kTile = NARROW ? 32 : B::kTile;
  static constexpr int kWarpTokens = kTile / kConsumerWarps;
  static constexpr int kSteps = kWarpTokens / 16;
  static constexpr int kHalfBytes = kTile * 128;
  static constexpr int kStageBytes = 2 * B::kHalves * kHalfBytes;
  static constexpr int kStages = NARROW || NT == 2 ? 3 : B::kStages;
  static constexpr int kCtasPerSm = NARROW ? 4 : (NT == 1 ? RRA_MMA_CTAS_PER_SM : 2);
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kOffBar = kRingBytes;
  static constexpr int kOffTable = kOffBar + (2 * kStages + 1) * 8;
  static constexpr int kOffCs = kOffTable + kMmaTableEntries * 4;
  static constexpr int kSmemBytes = 1024 + kOffCs + 4 * (D / 2) * 4;
  static constexpr int kMaxHeads = 8 * NT;
  static_assert(!NARROW || (D == 128 && NT == 1), "narrow CTAs: head_dim 128, 8 heads");
};

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled buffer.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (r << 7) + (((c ^ r) & 7) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void tma_g2s_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                           uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int D>
struct MmaWarpState {
  float o[D / 16][4];   // O^T fragments: dims 16*i + lane/4 (+8), heads 2*(lane%4) + {0,1}
  float m[2], l[2];     // running max (log2 units) and this lane's partial sum, per owned head
};

// One 16-token slice of a stage for one warp. CHECK: tokens at or past `valid` are masked
// (their V rows are zeroed first, so NaN or stale data never reaches the tensor cores).
// HALF: bytes of one 64-dim half of K or V in the stage (rows of the tile x 128).
template <int D, bool CHECK, int HALF = MmaCfg<D>::kHalfBytes>
__device__ __forceinline__ void mma_step(MmaWarpState<D>& st, const uint32_t (&qb)[D / 16][2], uint32_t k_base,
                                         uint32_t v_base, uint8_t* v_gen, int t0, int valid, int lane,
                                         float scale_log2) {
  using C = MmaCfg<D>;
  if (CHECK) {  // zero V rows t0+i >= valid of this slice (each row: kHalves x 128 bytes)
    const int first = max(valid - t0, 0);
    if (first < 16) {
      for (int idx = lane; idx < (16 - first) * C::kHalves * 8; idx += 32) {
        const int r = t0 + first + idx / (C::kHalves * 8);
        const int h = (idx / 8) % C::kHalves, c = idx % 8;
        *reinterpret_cast<uint4*>(v_gen + h * HALF + swz(r, c)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();  // these generic writes precede the next TMA write of the stage
      __syncwarp();
    }
  }
  // scores
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int mat = lane >> 3;
    const int r = t0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < C::kKSteps; ++kk) {
      uint32_t a[4];
      ldsm_x4(k_base + (kk >> 2) * HALF + swz(r, ((kk & 3) << 1) + (mat >> 1)), a);
      mma_bf16(s, a, qb[kk][0], qb[kk][1]);
    }
  }
  // online softmax on the fragment: s[j] token t0 + lane/4, s[2 + j] token t0 + lane/4 + 8; head 2*(lane%4) + j
  const int ta = t0 + (lane >> 2), tb = ta + 8;
  float x[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    x[j][0] = (!CHECK || ta < valid) ? s[j] * scale_log2 : -INFINITY;
    x[j][1] = (!CHECK || tb < valid) ? s[2 + j] * scale_log2 : -INFINITY;
  }
  float mnew[2];
  bool grow = false;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float mx = fmaxf(x[j][0], x[j][1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mnew[j] = fmaxf(st.m[j], mx);
    grow |= mnew[j] > st.m[j];
  }
  if (__any_sync(0xffffffffu, grow)) {
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      alpha[j] = mnew[j] > st.m[j] ? exp2f(st.m[j] - mnew[j]) : 1.f;
      st.l[j] *= alpha[j];
      st.m[j] = mnew[j];
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      st.o[i][0] *= alpha[0];
      st.o[i][1] *= alpha[1];
      st.o[i][2] *= alpha[0];
      st.o[i][3] *= alpha[1];
    }
  }
  float p[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float mref = st.m[j] == -INFINITY ? 0.f : st.m[j];
    p[j][0] = exp2f(x[j][0] - mref);
    p[j][1] = exp2f(x[j][1] - mref);
    st.l[j] += p[j][0] + p[j][1];
  }
  // P as the B operand (k = token, n = head): transpose the two 8x8 token halves.
  const uint32_t b0 = movmatrix_trans(pack_bf16x2(p[0][0], p[1][0]));
  const uint32_t b1 = movmatrix_trans(pack_bf16x2(p[0][1], p[1][1]));
  {
    const int mat = lane >> 3;
    const int r = t0 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      uint32_t a[4];
      ldsm_x4_trans(v_base + (i >> 2) * HALF + swz(r, ((i & 3) << 1) + (mat & 1)), a);
      mma_bf16(st.o[i], a, b0, b1);
    }
  }
}

// Online softmax of one 8-head n-tile's score fragment (as in mma_step); returns P as the B operand.
template <int D, bool CHECK>
__device__ __forceinline__ void softmax_tile(MmaWarpState<D>& st, const float (&s)[4], int t0, int valid, int lane,
                                             float scale_log2, uint32_t& b0, uint32_t& b1) {
  const int ta = t0 + (lane >> 2), tb = ta + 8;
  float x[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    x[j][0] = (!CHECK || ta < valid) ? s[j] * scale_log2 : -INFINITY;
    x[j][1] = (!CHECK || tb < valid) ? s[2 + j] * scale_log2 : -INFINITY;
  }
  float mnew[2];
  bool grow = false;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float mx = fmaxf(x[j][0], x[j][1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mnew[j] = fmaxf(st.m[j], mx);
    grow |= mnew[j] > st.m[j];
  }
  if (__any_sync(0xffffffffu, grow)) {
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      alpha[j] = mnew[j] > st.m[j] ? exp2f(st.m[j] - mnew[j]) : 1.f;
      st.l[j] *= alpha[j];
      st.m[j] = mnew[j];
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      st.o[i][0] *= alpha[0];
      st.o[i][1] *= alpha[1];
      st.o[i][2] *= alpha[0];
      st.o[i][3] *= alpha[1];
    }
  }
  float p[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float mref = st.m[j] == -INFINITY ? 0.f : st.m[j];
    p[j][0] = exp2f(x[j][0] - mref);
    p[j][1] = exp2f(x[j][1] - mref);
    st.l[j] += p[j][0] + p[j][1];
  }
  b0 = movmatrix_trans(pack_bf16x2(p[0][0], p[1][0]));
  b1 = movmatrix_trans(pack_bf16x2(p[0][1], p[1][1]));
}

// mma_step for 16 query heads (two 8-head n-tiles, st[0] heads 0-7 and st[1] heads 8-15): each K
// and V fragment read from shared memory feeds both n-tiles, whose score chains run side by side.
template <int D, bool CHECK>
__device__ __forceinline__ void mma_step2(MmaWarpState<D> (&st)[2], const uint32_t (&qb)[2][D / 16][2],
                                          uint32_t k_base, uint32_t v_base, uint8_t* v_gen, int t0, int valid,
                                          int lane, float scale_log2) {
  using C = MmaCfg<D>;
  constexpr int HALF = C::kHalfBytes;
  if (CHECK) {  // zero V rows t0+i >= valid of this slice (each row: kHalves x 128 bytes)
    const int first = max(valid - t0, 0);
    if (first < 16) {
      for (int idx = lane; idx < (16 - first) * C::kHalves * 8; idx += 32) {
        const int r = t0 + first + idx / (C::kHalves * 8);
        const int h = (idx / 8) % C::kHalves, c = idx % 8;
        *reinterpret_cast<uint4*>(v_gen + h * HALF + swz(r, c)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
  }
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int mat = lane >> 3;
    const int r = t0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < C::kKSteps; ++kk) {
      uint32_t a[4];
      ldsm_x4(k_base + (kk >> 2) * HALF + swz(r, ((kk & 3) << 1) + (mat >> 1)), a);
      mma_bf16(s[0], a, qb[0][kk][0], qb[0][kk][1]);
      mma_bf16(s[1], a, qb[1][kk][0], qb[1][kk][1]);
    }
  }
  uint32_t b0[2], b1[2];
  softmax_tile<D, CHECK>(st[0], s[0], t0, valid, lane, scale_log2, b0[0], b1[0]);
  softmax_tile<D, CHECK>(st[1], s[1], t0, valid, lane, scale_log2, b0[1], b1[1]);
  {
    const int mat = lane >> 3;
    const int r = t0 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      uint32_t a[4];
      ldsm_x4_trans(v_base + (i >> 2) * HALF + swz(r, ((i & 3) << 1) + (mat & 1)), a);
      mma_bf16(st[0].o[i], a, b0[0], b1[0]);
      mma_bf16(st[1].o[i], a, b0[1], b1[1]);
    }
  }
}

// Fused step only: rotates the consumer lane's q fragment (raw bf16 pairs, same layout as
// the B operand) in place, with cos/sin hi/lo per frequency in `cs`.
template <int D>
__device__ __forceinline__ void rotate_q_fragment(uint32_t (&qb)[D / 16][2], const float* cs, int lane, int style) {
  constexpr int KK = D / 16, HALF = D / 2;
  const int c2 = 2 * (lane & 3);
  auto unpack = [](uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  };
  if (style == 1) {  // interleaved pairs (2i, 2i+1): the two halves of each 32-bit word
#pragma unroll
    for (int kk = 0; kk < KK; ++kk)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = (16 * kk + 8 * r + c2) >> 1;
        float x0, x1;
        unpack(qb[kk][r], x0, x1);
        const float ch = cs[i], cl = cs[HALF + i], sh = cs[2 * HALF + i], sl = cs[3 * HALF + i];
        qb[kk][r] = pack_bf16x2(rotate_diff(x0, x1, ch, cl, sh, sl), rotate_diff(x1, -x0, ch, cl, sh, sl));
      }
    return;
  }
  // half-split pairs (i, i + D/2): k-step kk and kk + KK/2 hold the two members
#pragma unroll
  for (int kk = 0; kk < KK / 2; ++kk)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float a0, a1, b0, b1;
      unpack(qb[kk][r], a0, a1);
      unpack(qb[kk + KK / 2][r], b0, b1);
      const int i0 = 16 * kk + 8 * r + c2, i1 = i0 + 1;
      const float ch0 = cs[i0], cl0 = cs[HALF + i0], sh0 = cs[2 * HALF + i0], sl0 = cs[3 * HALF + i0];
      const float ch1 = cs[i1], cl1 = cs[HALF + i1], sh1 = cs[2 * HALF + i1], sl1 = cs[3 * HALF + i1];
      qb[kk][r] = pack_bf16x2(rotate_diff(a0, b0, ch0, cl0, sh0, sl0), rotate_diff(a1, b1, ch1, cl1, sh1, sl1));
      qb[kk + KK / 2][r] =
          pack_bf16x2(rotate_diff(b0, -a0, ch0, cl0, sh0, sl0), rotate_diff(b1, -a1, ch1, cl1, sh1, sl1));
    }
}

// The fused step's append, by one warp: rotated k_new and raw v_new into slot pos of KV head g.
// Lane l holds dims E l .. E l + E - 1 (E = D / 32) of both as bf16 pairs; a half-split RoPE
// pair (i, i + D/2) sits in lanes l and l ^ 16. The rotation is the append kernel's. Every
// head-slice CTA of this chunk writes the same bytes, so their writes cannot tear one another's
// reads. Arrives on `appended` once the writes are visible to TMA reads.
template <int D, bool PAGED>
__device__ __forceinline__ void append_token_bf16(const DecodeArgs& a, const float* cs, const uint32_t (&kraw)[D / 64],
                                                  const uint32_t (&vraw)[D / 64], int phys, int b, int g, int pos,
                                                  int lane, uint64_t* appended) {
  constexpr int E = D / 32;
  size_t row = 0;
  bool ok = true;
  if constexpr (PAGED) {
    ok = phys >= 0 && phys < a.num_blocks;  // a bad id was flagged when the table was read
    row = ((static_cast<size_t>(phys) << a.log2_bs) + (pos & ((1 << a.log2_bs) - 1))) * a.Hkv + g;
  } else {
    row = (static_cast<size_t>(b) * a.Hkv + g) * a.max_len + pos;
  }
  float kx[E];
#pragma unroll
  for (int w = 0; w < E / 2; ++w) {
    kx[2 * w] = __uint_as_float(kraw[w] << 16);
    kx[2 * w + 1] = __uint_as_float(kraw[w] & 0xffff0000u);
  }
  float kr[E];
  if (a.rope_style == 1) {  // interleaved pairs (2i, 2i + 1), both in this lane
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const int i = (E * lane + e) / 2;
      const float ch = cs[i], cl = cs[D / 2 + i], sh = cs[D + i], sl = cs[3 * (D / 2) + i];
      kr[e] = rotate_diff(kx[e], kx[e + 1], ch, cl, sh, sl);
      kr[e + 1] = rotate_diff(kx[e + 1], -kx[e], ch, cl, sh, sl);
    }
  } else {  // half-split pairs (i, i + D/2): the partner is 16 lanes away
    const bool first = lane < 16;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float partner = __shfl_xor_sync(0xffffffffu, kx[e], 16);
      const int i = E * (lane & 15) + e;
      const float ch = cs[i], cl = cs[D / 2 + i], sh = cs[D + i], sl = cs[3 * (D / 2) + i];
      kr[e] = first ? rotate_diff(kx[e], partner, ch, cl, sh, sl)     // a cos - b sin
                    : rotate_diff(kx[e], -partner, ch, cl, sh, sl);   // b cos + a sin
    }
  }
  if (ok) {
    uint32_t* kd = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(const_cast<void*>(a.k)) + row * D + E * lane);
    uint32_t* vd = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(const_cast<void*>(a.v)) + row * D + E * lane);
#pragma unroll
    for (int w = 0; w < E / 2; ++w) {
      kd[w] = pack_bf16x2(kr[2 * w], kr[2 * w + 1]);
      vd[w] = vraw[w];
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // visible to the TMA that reads the slot
  __syncwarp();
  if (lane == 0 && !a.test_hold_append) mbar_arrive(appended);  // the hold: see DecodeArgs
}

template <int D, bool PAGED, bool FUSED, int NT = 1, bool NARROW = false>
__global__ void __launch_bounds__(MmaCfgN<D, NT, NARROW>::kThreads, MmaCfgN<D, NT, NARROW>::kCtasPerSm)
    decode_mma_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                      const DecodeArgs a) {
  using C = MmaCfgN<D, NT, NARROW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int n_rep = a.Hq / a.Hkv;
  const int hpc = a.hpc;
  const int slices = n_rep / hpc;
  const int split = blockIdx.x / slices;
  const int g = blockIdx.y;
  const int h0 = g * n_rep + (blockIdx.x - split * slices) * hpc;
  const int b = blockIdx.z;

  // Programmatic dependent launch: the next kernel may be scheduled now. Until the previous
  // kernel has finished, only warm L2 with this CTA's first tiles, from lengths and block ids
  // read ahead (they may still change: they only choose what to prefetch, clamped in range).
  pdl_launch_dependents();
  if (threadIdx.x == C::kConsumerWarps * 32) {
    const int Ls = min(max(FUSED ? a.positions[b] + 1 : a.seq_lens[b], 0), a.capacity);
    const int s0 = split * a.chunk;
    const int e0 = min(Ls, s0 + a.chunk);
    const int nt = s0 < Ls ? min((e0 - s0 + C::kTile - 1) / C::kTile, C::kStages) : 0;
    for (int it = 0; it < nt; ++it) {
      const int t0 = s0 + it * C::kTile;
      if constexpr (PAGED) {
        const int bs = 1 << a.log2_bs;
        const bool whole = bs <= C::kTile;
        const int nblk = whole ? (min(C::kTile, e0 - t0) + bs - 1) >> a.log2_bs : 1;
        for (int jb = 0; jb < nblk; ++jb) {
          int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (t0 >> a.log2_bs) + jb];
          phys = min(max(phys, 0), a.num_blocks - 1);
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h) {
            tma_prefetch_l2_4d(&k_map, 64 * h, g, whole ? 0 : (t0 & (bs - 1)), phys);
            tma_prefetch_l2_4d(&v_map, 64 * h, g, whole ? 0 : (t0 & (bs - 1)), phys);
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h) {
          tma_prefetch_l2_3d(&k_map, 64 * h, t0, b * a.Hkv + g);
          tma_prefetch_l2_3d(&v_map, 64 * h, t0, b * a.Hkv + g);
        }
      }
    }
  }
  pdl_wait();
  // the chunk's block ids load alongside the sequence length
  ChunkBlockIds<(kMmaTableEntries + C::kThreads - 1) / C::kThreads> pre_ids;
  if constexpr (PAGED) pre_ids.load(a, b, (split * a.chunk) >> a.log2_bs, threadIdx.x, C::kThreads);

  int L;
  if constexpr (FUSED) {
    const int pos = a.positions[b];
    if (pos < 0 || pos >= a.capacity) {  // nothing is written for this sequence
      if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) flag_error(a.err, RRA_ERR_POSITION);
      return;
    }
    L = pos + 1;
  } else {
    L = a.seq_lens[b];
    if (L < 0 || L > a.capacity) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) flag_error(a.err, RRA_ERR_SEQ_LEN);
      L = min(max(L, 0), a.capacity);
    }
  }
  const int start = split * a.chunk;
  const int n_work = (L + a.chunk - 1) / a.chunk;  // splits of this sequence that hold tokens
  if (start >= L) {
    if (L == 0 && split == 0) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(b) * a.Hq + h0) * D;
      for (int i = threadIdx.x; i < hpc * D; i += blockDim.x) out[i] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int end = min(L, start + a.chunk);
  const int n_tiles = (end - start + C::kTile - 1) / C::kTile;
  // Fused step: this CTA's chunk holds the new token, so it writes it into the cache first.
  const bool appender = FUSED && end == L;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + C::kStages;
  uint64_t* appended = empty + C::kStages;
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kOffTable);
  float* cs = reinterpret_cast<float*>(smem + C::kOffCs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    mbar_init(appended, 1);
    fence_barrier_init();
  }
  int first_blk = 0;
  if constexpr (PAGED) {
    first_blk = start >> a.log2_bs;
    const int n_blk = ((end - 1) >> a.log2_bs) - first_blk + 1;
    pre_ids.store(a, tbl, n_blk, threadIdx.x, C::kThreads);
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer
  if (warp == C::kConsumerWarps) {
    // Lane 0 waits for the stage and sets its byte count; the copies of the stage are then issued
    // by RRA_MMA_ISSUE_LANES lanes of the warp at once (a stage of 16-token blocks is 16 copies).
    constexpr int kIssueLanes = RRA_MMA_ISSUE_LANES;
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
    int issued = 0;
    for (int it = 0; it < n_tiles; ++it) {
      const int s = it % C::kStages;
      const int t0 = start + it * C::kTile;
      uint8_t* kst = smem + s * C::kStageBytes;
      uint8_t* vst = kst + C::kHalves * C::kHalfBytes;
      // copies of this stage: paged whole blocks nblk x kHalves x {K, V}; otherwise kHalves x {K, V}
      int nblk = 1, bytes = 2 * C::kHalves * C::kTile * 128;
      if constexpr (PAGED) {
        const int bs = 1 << a.log2_bs;
        if (bs <= C::kTile) {
          nblk = (min(C::kTile, end - t0) + bs - 1) >> a.log2_bs;
          bytes = 2 * C::kHalves * nblk * bs * 128;
        }
      }
      int ok = 1;
      if (lane == 0) {
        if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1)) {
          flag_error(a.err, RRA_ERR_TIMEOUT);
          ok = 0;
        } else if (appender && it == n_tiles - 1 && !mbar_wait(appended, 0)) {  // the new token is in this tile
          flag_error(a.err, RRA_ERR_TIMEOUT);
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(bytes));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane < kIssueLanes) {
        for (int c = lane; c < 2 * C::kHalves * nblk; c += kIssueLanes) {
          const int kv = c & 1, h = (c >> 1) % C::kHalves, jb = (c >> 1) / C::kHalves;
          uint8_t* dst = (kv ? vst : kst) + h * C::kHalfBytes;
          const CUtensorMap* map = kv ? &v_map : &k_map;
          if constexpr (PAGED) {
            const int bs = 1 << a.log2_bs;
            if (bs <= C::kTile) {  // whole blocks, one box of bs rows per block and half
              tma_g2s_4d(dst + jb * bs * 128, map, 64 * h, g, 0, tbl[(t0 >> a.log2_bs) - first_blk + jb], &full[s]);
            } else {  // a kTile-row window of one block
              tma_g2s_4d(dst, map, 64 * h, g, t0 & (bs - 1), tbl[(t0 >> a.log2_bs) - first_blk], &full[s]);
            }
          } else {  // contiguous: box of kTile rows of sequence b, head g (rows past max_len read as 0)
            tma_g2s_3d(dst, map, 64 * h, t0, b * a.Hkv + g, &full[s]);
          }
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    if (lane == 0)
      for (int it = issued > C::kStages ? issued - C::kStages : 0; it < issued; ++it)
        mbar_wait(&full[it % C::kStages], (it / C::kStages) & 1);
    return;
  }

  // ------------------------------------------------------------------ consumers
  constexpr int kConsumerThreads = C::kConsumerWarps * 32;
  // Q^T as the B operand: n-tile n, lane holds q[head 8n + lane/4][dims 16kk + 2(lane%4) + {0,1}] and (+8).
  uint32_t qb[NT][C::kKSteps][2];
  const int hd = lane >> 2;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                          (static_cast<size_t>(b) * a.Hq + h0 + 8 * n + hd) * D);
#pragma unroll
    for (int kk = 0; kk < C::kKSteps; ++kk) {
      qb[n][kk][0] = 8 * n + hd < hpc ? q[kk * 8 + (lane & 3)] : 0u;
      qb[n][kk][1] = 8 * n + hd < hpc ? q[kk * 8 + 4 + (lane & 3)] : 0u;
    }
  }
  if constexpr (FUSED) {
    // RoPE ("Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §3): sine and cosine of
    // pos * theta_i as float32 hi + lo pairs (rope_cos_sin) for the error-free rotation.
    const int pos = L - 1;
    // the appender warp fetches the new token's k and v (D / 32 dims per lane) and its block id
    // now, so that the loads overlap the sine / cosine below
    const bool app_warp = appender && warp == 1;
    uint32_t kraw[D / 64], vraw[D / 64];
    int phys = 0;
    if (app_warp) {
      const size_t off = (static_cast<size_t>(b) * a.Hkv + g) * D + lane * (D / 32);
      const uint32_t* kn = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.k_new) + off);
      const uint32_t* vn = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.v_new) + off);
#pragma unroll
      for (int w = 0; w < D / 64; ++w) {
        kraw[w] = kn[w];
        vraw[w] = vn[w];
      }
      if constexpr (PAGED) phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
    }
    if (threadIdx.x < D / 2) {
      rope_cos_sin(pos, a.rope_phi[threadIdx.x], cs[threadIdx.x], cs[D / 2 + threadIdx.x], cs[D + threadIdx.x],
                   cs[3 * (D / 2) + threadIdx.x]);
    }
    named_barrier_sync(1, kConsumerThreads);
#pragma unroll
    for (int n = 0; n < NT; ++n) rotate_q_fragment<D>(qb[n], cs, lane, a.rope_style);
#pragma unroll
    for (int n = 0; n < NT; ++n)
      if (warp == 0 && split == 0 && 8 * n + hd < hpc) {  // publish q_rot (rounded to bf16, as used here)
        uint32_t* qo = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.q_out) +
                                                   (static_cast<size_t>(b) * a.Hq + h0 + 8 * n + hd) * D);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk) {
          qo[kk * 8 + (lane & 3)] = qb[n][kk][0];
          qo[kk * 8 + 4 + (lane & 3)] = qb[n][kk][1];
        }
      }
    if (app_warp) append_token_bf16<D, PAGED>(a, cs, kraw, vraw, phys, b, g, pos, lane, appended);
  }
  MmaWarpState<D> st[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int i = 0; i < D / 16; ++i) st[n].o[i][0] = st[n].o[i][1] = st[n].o[i][2] = st[n].o[i][3] = 0.f;
    st[n].m[0] = st[n].m[1] = -INFINITY;
    st[n].l[0] = st[n].l[1] = 0.f;
  }

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % C::kStages;
    if (!mbar_wait(&full[s], (it / C::kStages) & 1)) {
      flag_error(a.err, RRA_ERR_TIMEOUT);
      break;
    }
    uint8_t* kst = smem + s * C::kStageBytes;
    uint8_t* vst = kst + C::kHalves * C::kHalfBytes;
    const uint32_t k_base = smem_addr(kst), v_base = smem_addr(vst);
    const int valid = min(C::kTile, end - (start + it * C::kTile));
#pragma unroll
    for (int step = 0; step < C::kSteps; ++step) {
      const int t0 = warp * C::kWarpTokens + step * 16;
      if constexpr (NT == 1) {
        if (valid == C::kTile)
          mma_step<D, false, C::kHalfBytes>(st[0], qb[0], k_base, v_base, vst, t0, valid, lane, a.scale_log2);
        else if (t0 < valid)
          mma_step<D, true, C::kHalfBytes>(st[0], qb[0], k_base, v_base, vst, t0, valid, lane, a.scale_log2);
      } else {
        if (valid == C::kTile)
          mma_step2<D, false>(st, qb, k_base, v_base, vst, t0, valid, lane, a.scale_log2);
        else if (t0 < valid)
          mma_step2<D, true>(st, qb, k_base, v_base, vst, t0, valid, lane, a.scale_log2);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ------------------------------------------------------------------ merge the 4 warps
  constexpr int kConsumers = C::kConsumerWarps * 32;
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      st[n].l[j] += __shfl_xor_sync(0xffffffffu, st[n].l[j], 4);
      st[n].l[j] += __shfl_xor_sync(0xffffffffu, st[n].l[j], 8);
      st[n].l[j] += __shfl_xor_sync(0xffffffffu, st[n].l[j], 16);
    }
  named_barrier_sync(1, kConsumers);
  // [warps][8 NT heads][D + 4]: the padded row stride puts the four heads a store instruction
  // covers in distinct banks
  constexpr int kRS = D + 4;
  static_assert(C::kConsumerWarps * C::kMaxHeads * (kRS + 4) * 4 + 2 * C::kMaxHeads * 4 <= C::kRingBytes,
                "the warp merge fits in the ring");
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + C::kConsumerWarps * C::kMaxHeads * kRS;  // [warps][8 NT heads]
  float* red_l = red_m + C::kConsumerWarps * C::kMaxHeads;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int hd0 = 8 * n + 2 * (lane & 3), dl = lane >> 2;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        red_o[(warp * C::kMaxHeads + hd0 + j) * kRS + 16 * i + dl] = st[n].o[i][j];
        red_o[(warp * C::kMaxHeads + hd0 + j) * kRS + 16 * i + 8 + dl] = st[n].o[i][2 + j];
      }
    }
    if (dl == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        red_m[warp * C::kMaxHeads + hd0 + j] = st[n].m[j];
        red_l[warp * C::kMaxHeads + hd0 + j] = st[n].l[j];
      }
    }
  }
  named_barrier_sync(1, kConsumers);
  // the warps' weights and the merged (max, sum) once per head, then the rows: a loop of
  // independent items (exp2f and the max per item would chain their latency through every item)
  float* red_w = red_l + C::kConsumerWarps * C::kMaxHeads;  // [warps][heads] weights
  float* red_ml = red_w + C::kConsumerWarps * C::kMaxHeads;  // [heads][2] merged max, sum
  for (int h = threadIdx.x; h < hpc; h += kConsumers) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, red_m[w * C::kMaxHeads + h]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) {
      const float wt = M != -INFINITY ? exp2f(red_m[w * C::kMaxHeads + h] - M) : 0.f;
      lsum = fmaf(wt, red_l[w * C::kMaxHeads + h], lsum);
      red_w[w * C::kMaxHeads + h] = wt;
    }
    red_ml[2 * h] = M;
    red_ml[2 * h + 1] = lsum;
  }
  named_barrier_sync(1, kConsumers);
#pragma unroll 4
  for (int idx = threadIdx.x; idx < hpc * D; idx += kConsumers) {
    const int h = idx / D, d = idx - h * D;
    const float M = red_ml[2 * h], lsum = red_ml[2 * h + 1];
    float osum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w)
      osum = fmaf(red_w[w * C::kMaxHeads + h], red_o[(w * C::kMaxHeads + h) * kRS + d], osum);
    const size_t bh = static_cast<size_t>(b) * a.Hq + h0 + h;
    if (n_work == 1) {
      static_cast<__nv_bfloat16*>(a.out)[bh * D + d] = __float2bfloat16_rn(lsum > 0.f ? osum / lsum : 0.f);
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
    finish_split<__nv_bfloat16, D>(a, b, h0, hpc, split, n_work, reinterpret_cast<float*>(smem), &s_last,
                                   threadIdx.x, kConsumers, C::kRingBytes);
  }
}

template <int D, bool PAGED, bool FUSED, int NT, bool NARROW = false>
cudaError_t launch_decode_mma_nt(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, int hpc,
                                 cudaStream_t st) {
  using C = MmaCfgN<D, NT, NARROW>;
  static int done[64] = {0};
  auto kern = decode_mma_kernel<D, PAGED, FUSED, NT, NARROW>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_splits * ((a.Hq / a.Hkv) / hpc), a.Hkv, a.B);
  return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, st, km, vm, a);
}

// 16 heads per CTA (two n-tiles) when hpc > 8; narrow CTAs when the plan asks for them (a.narrow).
template <int D, bool PAGED, bool FUSED>
cudaError_t launch_decode_mma_t(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, int hpc,
                                cudaStream_t st) {
  if (hpc > 8) return launch_decode_mma_nt<D, PAGED, FUSED, 2>(a, km, vm, hpc, st);
  if constexpr (D == 128)
    if (a.narrow) return launch_decode_mma_nt<D, PAGED, FUSED, 1, true>(a, km, vm, hpc, st);
  return launch_decode_mma_nt<D, PAGED, FUSED, 1>(a, km, vm, hpc, st);
}

template <bool PAGED, bool FUSED = false>
cudaError_t launch_decode_mma(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, int hpc,
                              cudaStream_t st) {
  if (a.D == 128) return launch_decode_mma_t<128, PAGED, FUSED>(a, km, vm, hpc, st);
  return launch_decode_mma_t<64, PAGED, FUSED>(a, km, vm, hpc, st);
}

}  // namespace rra
