// Split-K GQA decode attention over an INT8 KV cache with per-KV-head scales and a bf16 window
// of recent tokens, on the tensor cores.
//
// "Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §4.3: K and V cached as INT8 with
// quantisation parameters calibrated per attention head, the most recent tokens kept at high
// precision. Here a KV head g holds codes c with value c * s_g (K and V each with their own
// scale), and the W most recent tokens of every sequence also sit in a bf16 ring of W slots
// (token t in slot t mod W). Attention over L tokens reads tokens [0, L - W) as codes and the
// last min(L, W) tokens from the ring; the softmax and the split/merge are those of
// decode_mma.cuh.
//
// Work units: the INT8 tokens are cut into splits of `chunk` tokens as in the bf16 kernel. The
// CTA of the last split that holds INT8 tokens (split 0 when there are none) then streams the
// ring through the same stages as bf16 tiles of 32 tokens (D = 128), after turning its INT8
// accumulator into the bf16 fragment layout (warp shuffles, times s_V), so every CTA publishes
// one partial and the last to finish merges them.
//
// INT8 tiles (K and V codes, D-byte rows with the TMA swizzle) go through the tensor cores as
// f16: ldmatrix loads 4 codes per lane; one lop3 keeps bytes 0 and 2 (or, after a shift, 1 and
// 3), flips their sign bits and puts the f16 exponent of 1024 above them (0x64xx = 1024 + byte),
// and one f16x2 subtraction of 1152 leaves each code exactly. The dimension order inside each
// 16-dim slice is permuted so those byte pairs are already in mma fragment order:
//   scores  S^T[16 tok x 8 heads] = C_K[16 tok x D] . Q'^T   with lane (g, t) holding dims
//           4t..4t+3 of a slice, dims (4t, 4t+2) as k = (2t, 2t+1) and (4t+1, 4t+3) as
//           k = (2t+8, 2t+9) (q packed in the same order);
//   output  O^T[D x 8 heads] += C_V^T . P   with ldmatrix.trans giving lane (g, t) dims
//           2g, 2g+1 of tokens 2t, 2t+1 (and +8), so fragment row g is dim 2g and row g+8 is
//           dim 2g+1 of each 16-dim slice.
// q is taken to f16 after a per-head power-of-two scaling (largest |q| in [2^14, 2^15)), exact
// for bf16 values; the scores are multiplied by s_K * scale * log2(e) * 2^-e_h in float32 and
// the output by s_V, so the only roundings are those of the f16 probabilities and the float32
// accumulation.
//
// Pipeline: RRA_Q8_STAGES stages of RRA_Q8_STAGE_BYTES (four of 16 KB by default: 64 INT8
// tokens at D = 128, one 16-token mma step per consumer warp; or 32 bf16 ring tokens, taken by
// two of the four warps).
#pragma once

#include <cuda_fp16.h>

#include "decode_mma.cuh"

namespace rra {

template <int D, int BITS = 8>
struct Q8Cfg {
  static constexpr int kRowBytes = D * BITS / 8;         // codes of one token and head
  static constexpr int kStageBytes = RRA_Q8_STAGE_BYTES;
  static constexpr int kTileBytes = kStageBytes / 2;     // K or V codes of one stage
  static constexpr int kTile = kTileBytes / kRowBytes;   // tokens per stage
  static constexpr int kStages = RRA_Q8_STAGES;
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kWarpTokens = kTile / kConsumerWarps;
  static constexpr int kSteps = kWarpTokens / 16;
  static_assert(kSteps >= 1 && kWarpTokens % 16 == 0, "each consumer warp takes whole 16-token steps");
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kWinTile = kStageBytes / (4 * D);  // bf16 ring tokens per stage (K + V)
  static constexpr int kWinHalf = kWinTile * 128;         // one 64-dim half of a ring tile
  static_assert(kWinTile % 16 == 0 && kWinTile / 16 <= kConsumerWarps, "ring tiles: whole steps, one per warp");
  // after the ring: full[kStages], empty[kStages], appended; the block-id table; cos/sin
  // hi/lo [4][D/2] floats; the rotated q rows [8][D] bf16 (fused step)
  static constexpr int kOffBar = kRingBytes;
  static constexpr int kOffTable = kOffBar + (2 * kStages + 1) * 8;
  static constexpr int kOffCs = kOffTable + kMmaTableEntries * 4;
  static constexpr int kOffQ = kOffCs + 4 * (D / 2) * 4;
  static constexpr int kSmemBytes = 1024 + kOffQ + MmaCfg<D>::kMaxHeads * D * 2;
};

// Byte offset of 16-byte chunk c of row r in a tile of RB-byte rows written by TMA with the
// 128-byte (RB = 128) or 64-byte (RB = 64) swizzle.
template <int RB>
__device__ __forceinline__ uint32_t swz8(int r, int c) {
  if constexpr (RB == 128) return swz(r, c);
  return (r << 6) + ((((r >> 1) ^ c) & 3) << 4);
}

// INT4: nibbles 0 and 4 of w as an exact f16 pair: sign bit flipped, under the exponent of 1024
// (lop3 table 0x6a, per bit b ? a^c : c), minus 1032.
__device__ __forceinline__ uint32_t nib04_to_f16(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(w), "r"(0x000f000fu), "r"(0x64086408u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(d), "r"(0x64086408u));
  return d;
}

// INT4: nibbles 1 and 5 of w: 1024 + 16 (n ^ 8) under the same exponent, times 1/16 minus 72.
__device__ __forceinline__ uint32_t nib15_to_f16(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(w), "r"(0x00f000f0u), "r"(0x64806480u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(d), "r"(0x2c002c00u), "r"(0xd480d480u));
  return d;
}

__device__ __forceinline__ uint32_t f16x2_minus_1152(uint32_t x) {
  uint32_t y;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(x), "r"(0x64806480u));
  return y;
}

// Bytes 0 and 2 of w with their sign bits flipped, each under the f16 exponent byte 0x64:
// per bit, b ? (a ^ c) : c with b = 0x00ff00ff and c = 0x64806480 (lop3 table 0x6a).
__device__ __forceinline__ uint32_t bytes02_to_f16_biased(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(w), "r"(0x00ff00ffu), "r"(0x64806480u));
  return d;
}

// Four INT8 codes (bytes 0..3 of w) as exact f16 pairs (bytes 0, 2) and (bytes 1, 3).
__device__ __forceinline__ void s8x4_to_f16_even_odd(uint32_t w, uint32_t& ev, uint32_t& od) {
  ev = f16x2_minus_1152(bytes02_to_f16_biased(w));
  od = f16x2_minus_1152(bytes02_to_f16_biased(__umulhi(w, 0x01000000u)));  // w >> 8 on the multiply pipe
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One 16-token slice of an INT8 stage for one warp; `mult[j]` turns the raw score of owned
// head 2*(lane%4)+j into log2 units. CHECK: tokens at or past `valid` get probability 0 (the
// codes are finite whatever the bytes, so nothing needs clearing). The score sum runs as two
// independent mma chains (the two 16-dim slices of each 32-byte chunk) added at the end.
template <int D, bool CHECK>
__device__ __forceinline__ void q8_step(MmaWarpState<D>& st, const uint32_t (&qh)[D / 16][2], const float (&mult)[2],
                                        uint32_t k_base, uint32_t v_base, int t0, int valid, int lane) {
  constexpr int RB = D;
  const int mat = lane >> 3;
  const int r = t0 + (lane & 7) + ((mat & 1) << 3);  // matrices: tokens 0-7 / 8-15 of chunk 2cc, then 2cc+1
  float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t w[4], a[4];
    ldsm_x4(k_base + swz8<RB>(r, 2 * cc + (mat >> 1)), w);
    s8x4_to_f16_even_odd(w[0], a[0], a[2]);
    s8x4_to_f16_even_odd(w[1], a[1], a[3]);
    mma_f16(s, a, qh[2 * cc][0], qh[2 * cc][1]);
    s8x4_to_f16_even_odd(w[2], a[0], a[2]);
    s8x4_to_f16_even_odd(w[3], a[1], a[3]);
    mma_f16(s2, a, qh[2 * cc + 1][0], qh[2 * cc + 1][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] += s2[i];
  const int ta = t0 + (lane >> 2), tb = ta + 8;
  float x[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    x[j][0] = (!CHECK || ta < valid) ? s[j] * mult[j] : -INFINITY;
    x[j][1] = (!CHECK || tb < valid) ? s[2 + j] * mult[j] : -INFINITY;
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
  const uint32_t b0 = movmatrix_trans(pack_f16x2(p[0][0], p[1][0]));
  const uint32_t b1 = movmatrix_trans(pack_f16x2(p[0][1], p[1][1]));
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t w[4], a[4];
    ldsm_x4_trans(v_base + swz8<RB>(r, 2 * cc + (mat >> 1)), w);
    s8x4_to_f16_even_odd(w[0], a[0], a[1]);
    s8x4_to_f16_even_odd(w[1], a[2], a[3]);
    mma_f16(st.o[2 * cc], a, b0, b1);
    s8x4_to_f16_even_odd(w[2], a[0], a[1]);
    s8x4_to_f16_even_odd(w[3], a[2], a[3]);
    mma_f16(st.o[2 * cc + 1], a, b0, b1);
  }
}

// INT4 (64-byte rows, 64-byte swizzle), two 16-token slices at once (tokens t0 .. t0 + 31 of the
// stage): the two score chains are independent and interleave, one softmax update covers 32
// tokens (at most one rescale), and each output fragment takes both slices' P.
// Fragment orders: a 16-byte chunk c holds 32 dims. For the scores ldmatrix gives lane (g, t)
// dims 32c + 8t .. +7 of rows g / g+8 (nibble i = dim 8t + i); 16-dim slice 2c takes dims
// (8t, 8t+4) as k = (2t, 2t+1) and (8t+1, 8t+5) as (2t+8, 2t+9), slice 2c+1 the same after a
// shift by 8 bits (dims 8t+2, 8t+6 and 8t+3, 8t+7); q is packed to match. For the output
// ldmatrix.trans gives lane (g, t) the 16-bit column g (dims 32c + 4g .. +3) of tokens 2t, 2t+1
// (and +8): fragment rows g / g+8 of sub-tile s are dims 32c + 4g + 2s / + 2s + 1.
template <int D, bool CHECK>
__device__ __forceinline__ void q4_step32(MmaWarpState<D>& st, const uint32_t (&qh)[D / 16][2], const float (&mult)[2],
                                          uint32_t k_base, uint32_t v_base, int t0, int valid, int lane) {
  constexpr int RB = D / 2;
  constexpr uint32_t kSlice = 16 * RB;  // 16 rows further down the tile (same swizzle phase)
  const int mat = lane >> 3;
  const int r = t0 + (lane & 7) + ((mat & 1) << 3);
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int cc = 0; cc < RB / 32; ++cc) {
    uint32_t w[2][4];
    const uint32_t off = swz8<RB>(r, 2 * cc + (mat >> 1));
    ldsm_x4(k_base + off, w[0]);
    ldsm_x4(k_base + off + kSlice, w[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * cc + h;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wa = w[u][2 * h], wb = w[u][2 * h + 1];
        const uint32_t a[4] = {nib04_to_f16(wa), nib04_to_f16(wb), nib15_to_f16(wa), nib15_to_f16(wb)};
        mma_f16(s[u], a, qh[2 * c][0], qh[2 * c][1]);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wa8 = w[u][2 * h] >> 8, wb8 = w[u][2 * h + 1] >> 8;
        const uint32_t a[4] = {nib04_to_f16(wa8), nib04_to_f16(wb8), nib15_to_f16(wa8), nib15_to_f16(wb8)};
        mma_f16(s[u], a, qh[2 * c + 1][0], qh[2 * c + 1][1]);
      }
    }
  }
  // x[j][k]: head 2(lane%4)+j at token t0 + lane/4 + 8k
  const int ta = t0 + (lane >> 2);
  float x[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      x[j][k] = (!CHECK || ta + 8 * k < valid) ? s[k >> 1][2 * (k & 1) + j] * mult[j] : -INFINITY;
  float mnew[2];
  bool grow = false;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float mx = fmaxf(fmaxf(x[j][0], x[j][1]), fmaxf(x[j][2], x[j][3]));
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
  float p[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float mref = st.m[j] == -INFINITY ? 0.f : st.m[j];
#pragma unroll
    for (int k = 0; k < 4; ++k) p[j][k] = exp2f(x[j][k] - mref);
    st.l[j] += (p[j][0] + p[j][1]) + (p[j][2] + p[j][3]);
  }
  uint32_t pb[2][2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    pb[u][0] = movmatrix_trans(pack_f16x2(p[0][2 * u], p[1][2 * u]));
    pb[u][1] = movmatrix_trans(pack_f16x2(p[0][2 * u + 1], p[1][2 * u + 1]));
  }
#pragma unroll
  for (int cc = 0; cc < RB / 32; ++cc) {
    uint32_t w[2][4];
    const uint32_t off = swz8<RB>(r, 2 * cc + (mat >> 1));
    ldsm_x4_trans(v_base + off, w[0]);
    ldsm_x4_trans(v_base + off + kSlice, w[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * cc + h;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t ra = w[u][2 * h], rb = w[u][2 * h + 1];
        const uint32_t a[4] = {nib04_to_f16(ra), nib15_to_f16(ra), nib04_to_f16(rb), nib15_to_f16(rb)};
        mma_f16(st.o[2 * c], a, pb[u][0], pb[u][1]);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t ra8 = w[u][2 * h] >> 8, rb8 = w[u][2 * h + 1] >> 8;
        const uint32_t a[4] = {nib04_to_f16(ra8), nib15_to_f16(ra8), nib04_to_f16(rb8), nib15_to_f16(rb8)};
        mma_f16(st.o[2 * c + 1], a, pb[u][0], pb[u][1]);
      }
    }
  }
}

// Moves an INT8-phase accumulator (fragment rows g / g+8 = dims 2g / 2g+1 of each 16-dim slice,
// in code units) into the bf16 layout (rows g / g+8 = dims g / g+8), times the V scale.
template <int D>
__device__ __forceinline__ void q8_acc_to_bf16_layout(MmaWarpState<D>& st, float vs, int lane) {
  const int dl = lane >> 2, t = lane & 3;
  const int src0 = ((dl >> 1) << 2) | t, src1 = (((dl >> 1) + 4) << 2) | t;  // owners of dims dl, dl + 8
  const bool odd = dl & 1;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float e0 = __shfl_sync(0xffffffffu, st.o[i][j], src0), o0 = __shfl_sync(0xffffffffu, st.o[i][2 + j], src0);
      const float e1 = __shfl_sync(0xffffffffu, st.o[i][j], src1), o1 = __shfl_sync(0xffffffffu, st.o[i][2 + j], src1);
      st.o[i][j] = (odd ? o0 : e0) * vs;
      st.o[i][2 + j] = (odd ? o1 : e1) * vs;
    }
  }
}

// The INT4 version: fragment rows g / g+8 of sub-tile s of chunk c are dims 32c + 4g + 2s / + 1.
template <int D>
__device__ __forceinline__ void q4_acc_to_bf16_layout(MmaWarpState<D>& st, float vs, int lane) {
  const int dl = lane >> 2, t = lane & 3;
  const int s_sel = (dl >> 1) & 1, e_sel = dl & 1;  // sub-tile and row half of dims dl, dl + 8 in a chunk
  float res[D / 16][4];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    const int c = i >> 1;
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      const int rem = 16 * (i & 1) + dl + 8 * f;   // dim within chunk c
      const int src = ((rem >> 2) << 2) | t;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float v00 = __shfl_sync(0xffffffffu, st.o[2 * c][j], src);
        const float v01 = __shfl_sync(0xffffffffu, st.o[2 * c][2 + j], src);
        const float v10 = __shfl_sync(0xffffffffu, st.o[2 * c + 1][j], src);
        const float v11 = __shfl_sync(0xffffffffu, st.o[2 * c + 1][2 + j], src);
        const float v = s_sel ? (e_sel ? v11 : v10) : (e_sel ? v01 : v00);
        res[i][2 * f + j] = v * vs;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < D / 16; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) st.o[i][k] = res[i][k];
}

// The fused step's append, by one warp: quantised k (rotated, rounded to bf16) and v into cache
// slot pos of KV head g, and with a window their bf16 values into ring slot pos % window. Lane l
// holds dims E l .. E l + E - 1 (E = D / 32) of k_new and v_new as bf16 pairs; a half-split
// RoPE pair (i, i + D/2) sits in lanes l and l ^ 16. The rotation and the codes are those of the
// append kernel. `phys`: the sequence's block id for pos (paged). Every head-slice CTA of this
// unit writes the same bytes. Arrives on `appended` once the writes are visible to TMA reads.
template <int D, int BITS, bool PAGED>
__device__ __forceinline__ void append_token_q8(const DecodeArgs& a, const float* cs, const uint32_t (&kraw)[D / 64],
                                                const uint32_t (&vraw)[D / 64], int phys, int b, int g, int pos,
                                                bool has_win, int lane, uint64_t* appended) {
  constexpr int E = D / 32;
  size_t row = 0;
  bool ok = true;
  if constexpr (PAGED) {
    ok = phys >= 0 && phys < a.num_blocks;  // a bad id was flagged when the table was read
    row = ((static_cast<size_t>(phys) << a.log2_bs) + (pos & ((1 << a.log2_bs) - 1))) * a.Hkv + g;
  } else {
    row = (static_cast<size_t>(b) * a.Hkv + g) * a.max_len + pos;
  }
  float kx[E], vx[E];
#pragma unroll
  for (int w = 0; w < E / 2; ++w) {
    kx[2 * w] = __uint_as_float(kraw[w] << 16);
    kx[2 * w + 1] = __uint_as_float(kraw[w] & 0xffff0000u);
    vx[2 * w] = __uint_as_float(vraw[w] << 16);
    vx[2 * w + 1] = __uint_as_float(vraw[w] & 0xffff0000u);
  }
  __nv_bfloat16 kr[E];
  if (a.rope_style == 1) {  // interleaved pairs (2i, 2i + 1), both in this lane
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const int i = (E * lane + e) / 2;
      const float ch = cs[i], cl = cs[D / 2 + i], sh = cs[D + i], sl = cs[3 * (D / 2) + i];
      kr[e] = __float2bfloat16_rn(rotate_diff(kx[e], kx[e + 1], ch, cl, sh, sl));
      kr[e + 1] = __float2bfloat16_rn(rotate_diff(kx[e + 1], -kx[e], ch, cl, sh, sl));
    }
  } else {  // half-split pairs (i, i + D/2): the partner is 16 lanes away
    const bool first = lane < 16;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float partner = __shfl_xor_sync(0xffffffffu, kx[e], 16);
      const int i = E * (lane & 15) + e;
      const float ch = cs[i], cl = cs[D / 2 + i], sh = cs[D + i], sl = cs[3 * (D / 2) + i];
      kr[e] = __float2bfloat16_rn(first ? rotate_diff(kx[e], partner, ch, cl, sh, sl)     // a cos - b sin
                                        : rotate_diff(kx[e], -partner, ch, cl, sh, sl));  // b cos + a sin
    }
  }
  const float ks = a.k_scale[g], vs = a.v_scale[g];
  if (ok) {
    if constexpr (BITS == 8) {
      uint32_t kc = 0, vc = 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        kc |= static_cast<uint32_t>(static_cast<uint8_t>(quantize_code(__bfloat162float(kr[e]), ks))) << (8 * e);
        vc |= static_cast<uint32_t>(static_cast<uint8_t>(quantize_code(vx[e], vs))) << (8 * e);
      }
      int8_t* kd = static_cast<int8_t*>(const_cast<void*>(a.k)) + row * D + E * lane;
      int8_t* vd = static_cast<int8_t*>(const_cast<void*>(a.v)) + row * D + E * lane;
      if constexpr (E == 4) {
        *reinterpret_cast<uint32_t*>(kd) = kc;
        *reinterpret_cast<uint32_t*>(vd) = vc;
      } else {
        *reinterpret_cast<uint16_t*>(kd) = static_cast<uint16_t>(kc);
        *reinterpret_cast<uint16_t*>(vd) = static_cast<uint16_t>(vc);
      }
    } else {  // codes of dims 2j, 2j+1 in byte j, the even one in the low nibble
      uint32_t kc = 0, vc = 0;
#pragma unroll
      for (int j = 0; j < E / 2; ++j) {
        kc |= static_cast<uint32_t>(pack_nibbles(quantize_code4(__bfloat162float(kr[2 * j]), ks),
                                                 quantize_code4(__bfloat162float(kr[2 * j + 1]), ks)))
              << (8 * j);
        vc |= static_cast<uint32_t>(pack_nibbles(quantize_code4(vx[2 * j], vs), quantize_code4(vx[2 * j + 1], vs)))
              << (8 * j);
      }
      uint8_t* kd = static_cast<uint8_t*>(const_cast<void*>(a.k)) + row * (D / 2) + (E / 2) * lane;
      uint8_t* vd = static_cast<uint8_t*>(const_cast<void*>(a.v)) + row * (D / 2) + (E / 2) * lane;
      static_assert(E == 4, "INT4 caches: head dim 128");
      *reinterpret_cast<uint16_t*>(kd) = static_cast<uint16_t>(kc);
      *reinterpret_cast<uint16_t*>(vd) = static_cast<uint16_t>(vc);
    }
  }
  if (has_win) {
    const size_t wrow = ((static_cast<size_t>(b) * a.Hkv + g) * a.window + pos % a.window) * D + E * lane;
    uint32_t kw[E / 2];
#pragma unroll
    for (int w = 0; w < E / 2; ++w)
      kw[w] = static_cast<uint32_t>(__bfloat16_as_ushort(kr[2 * w])) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(kr[2 * w + 1])) << 16);
    uint32_t* kwd = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.k_win) + wrow);
    uint32_t* vwd = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.v_win) + wrow);
#pragma unroll
    for (int w = 0; w < E / 2; ++w) {
      kwd[w] = kw[w];
      vwd[w] = vraw[w];
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // visible to the TMA that reads the slot
  __syncwarp();
  if (lane == 0) mbar_arrive(appended);
}

template <int D, int BITS, bool PAGED, bool FUSED>
__global__ void __launch_bounds__(Q8Cfg<D, BITS>::kThreads, RRA_Q8_CTAS_PER_SM)
    decode_q8_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                     const __grid_constant__ CUtensorMap kw_map, const __grid_constant__ CUtensorMap vw_map,
                     const DecodeArgs a) {
  using C = Q8Cfg<D, BITS>;
  using M = MmaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int n_rep = a.Hq / a.Hkv;
  const int hpc = a.hpc;
  const int slices = n_rep / hpc;
  const int split = blockIdx.x / slices;
  const int g = blockIdx.y;
  const int h0 = g * n_rep + (blockIdx.x - split * slices) * hpc;
  const int b = blockIdx.z;
  const bool has_win = a.window > 0;

  // Programmatic dependent launch, as in decode_mma_kernel: warm L2 with this CTA's first INT8
  // tiles from lengths and block ids read ahead (clamped), then wait for the previous kernel.
  pdl_launch_dependents();
  if (threadIdx.x == C::kConsumerWarps * 32) {
    const int Ls = min(max(FUSED ? a.positions[b] + 1 : a.seq_lens[b], 0), a.capacity);
    const int Lqs = Ls - (has_win ? min(Ls, a.window) : 0);
    const int s0 = split * a.chunk;
    const int e0 = min(Lqs, s0 + a.chunk);
    const int nt = s0 < Lqs ? min((e0 - s0 + C::kTile - 1) / C::kTile, C::kStages) : 0;
    for (int it = 0; it < nt; ++it) {
      const int t0 = s0 + it * C::kTile;
      if constexpr (PAGED) {
        const int bs = 1 << a.log2_bs;
        const bool whole = bs <= C::kTile;
        const int nblk = whole ? (min(C::kTile, e0 - t0) + bs - 1) >> a.log2_bs : 1;
        for (int jb = 0; jb < nblk; ++jb) {
          int phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (t0 >> a.log2_bs) + jb];
          phys = min(max(phys, 0), a.num_blocks - 1);
          tma_prefetch_l2_4d(&k_map, 0, g, whole ? 0 : (t0 & (bs - 1)), phys);
          tma_prefetch_l2_4d(&v_map, 0, g, whole ? 0 : (t0 & (bs - 1)), phys);
        }
      } else {
        tma_prefetch_l2_3d(&k_map, 0, t0, b * a.Hkv + g);
        tma_prefetch_l2_3d(&v_map, 0, t0, b * a.Hkv + g);
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
  const int Lw = has_win ? min(L, a.window) : 0;  // tokens read from the ring
  const int Lq = L - Lw;                          // tokens read as INT8 codes
  const int nq = (Lq + a.chunk - 1) / a.chunk;
  const int n_work = max(nq, Lw > 0 ? 1 : 0);     // one partial per CTA with tokens
  const bool ring_owner = Lw > 0 && split == max(nq - 1, 0);
  const int start = split * a.chunk;
  if (start >= Lq && !ring_owner) {
    if (L == 0 && split == 0) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(b) * a.Hq + h0) * D;
      for (int i = threadIdx.x; i < hpc * D; i += blockDim.x) out[i] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int end = min(Lq, start + a.chunk);
  const int n_q8 = start < Lq ? (end - start + C::kTile - 1) / C::kTile : 0;
  const int wrows = min(C::kWinTile, max(a.window, 1));   // ring rows per tile
  const int n_win = ring_owner ? (Lw + wrows - 1) / wrows : 0;
  const int n_tiles = n_q8 + n_win;
  // Fused step: the CTA that reads the new token writes it first (the ring owner, else the CTA
  // whose INT8 chunk ends at L); the CTA whose warp 0 publishes q_rot always has tokens.
  const bool appender = FUSED && (has_win ? ring_owner : end == L);
  const bool publisher = FUSED && (has_win ? ring_owner : split == 0);

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + C::kStages;
  uint64_t* appended = empty + C::kStages;
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kOffTable);
  float* cs = reinterpret_cast<float*>(smem + C::kOffCs);
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + C::kOffQ);
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
  if (PAGED && n_q8 > 0) {
    first_blk = start >> a.log2_bs;
    const int n_blk = ((end - 1) >> a.log2_bs) - first_blk + 1;
    pre_ids.store(a, tbl, n_blk, threadIdx.x, C::kThreads);
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer
  if (warp == C::kConsumerWarps) {
    // Lane 0 waits for the stage and sets its byte count; a stage of whole paged blocks (8 or 16
    // copies) is then issued by all lanes at once, other stages by lane 0.
    if (lane == 0) {
      if (n_q8 > 0) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
      }
      if (n_win > 0) {
        prefetch_tensormap(&kw_map);
        prefetch_tensormap(&vw_map);
      }
    }
    int issued = 0;
    for (int it = 0; it < n_tiles; ++it) {
      const int s = it % C::kStages;
      uint8_t* kst = smem + s * C::kStageBytes;
      const bool ring = it >= n_q8;
      const int t0 = ring ? (it - n_q8) * wrows : start + it * C::kTile;
      int nblk = 0;  // > 0: whole paged blocks of this stage, issued by the warp
      uint32_t bytes = ring ? 2 * M::kHalves * wrows * 128 : 2 * C::kTileBytes;
      if constexpr (PAGED) {
        const int bs = 1 << a.log2_bs;
        if (!ring && bs <= C::kTile) {
          nblk = (min(C::kTile, end - t0) + bs - 1) >> a.log2_bs;
          bytes = 2 * nblk * bs * C::kRowBytes;
        }
      }
      int ok = 1;
      if (lane == 0) {
        if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1)) {
          flag_error(a.err, RRA_ERR_TIMEOUT);
          ok = 0;
        } else if (appender && it == (has_win ? n_q8 : n_q8 - 1) && !mbar_wait(appended, 0)) {
          // the new token: in the ring (before its first tile) or in the appender's last INT8 tile
          flag_error(a.err, RRA_ERR_TIMEOUT);
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&full[s], bytes);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (nblk > 0) {  // whole blocks, one box of bs rows per block
        const int bs = 1 << a.log2_bs;
        const int j0 = (t0 >> a.log2_bs) - first_blk;
        for (int c = lane; c < 2 * nblk; c += 32) {
          const int jb = c >> 1;
          uint8_t* dst = (c & 1 ? kst + C::kTileBytes : kst) + jb * bs * C::kRowBytes;
          tma_g2s_4d(dst, c & 1 ? &v_map : &k_map, 0, g, 0, tbl[j0 + jb], &full[s]);
        }
      } else if (lane == 0) {
        if (ring) {  // bf16 ring rows [t0, t0 + wrows) of (b, g) in 64-dim halves
          uint8_t* vst = kst + M::kHalves * C::kWinHalf;
          const int bg = b * a.Hkv + g;
#pragma unroll
          for (int h = 0; h < M::kHalves; ++h) {
            tma_g2s_3d(kst + h * C::kWinHalf, &kw_map, 64 * h, t0, bg, &full[s]);
            tma_g2s_3d(vst + h * C::kWinHalf, &vw_map, 64 * h, t0, bg, &full[s]);
          }
        } else {
          uint8_t* vst = kst + C::kTileBytes;
          if constexpr (PAGED) {  // a kTile-row window of one block
            const int bs = 1 << a.log2_bs;
            const int phys = tbl[(t0 >> a.log2_bs) - first_blk];
            const int off = t0 & (bs - 1);
            tma_g2s_4d(kst, &k_map, 0, g, off, phys, &full[s]);
            tma_g2s_4d(vst, &v_map, 0, g, off, phys, &full[s]);
          } else {  // contiguous: rows [t0, t0 + kTile) of (b, g); rows past max_len read as 0
            const int bg = b * a.Hkv + g;
            tma_g2s_3d(kst, &k_map, 0, t0, bg, &full[s]);
            tma_g2s_3d(vst, &v_map, 0, t0, bg, &full[s]);
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
  constexpr int kConsumers = C::kConsumerWarps * 32;
  const int hd = lane >> 2;
  const __nv_bfloat16* q_in = static_cast<const __nv_bfloat16*>(a.q) + (static_cast<size_t>(b) * a.Hq + h0) * D;
  const __nv_bfloat16* q_rows = q_in;  // rotated q rows: q_rot in memory, or the fused step's own
  // q as the bf16 B operand (lane holds q[head lane/4][dims 16kk + 2(lane%4) + {0,1}] and (+8))
  auto load_qb = [&](const __nv_bfloat16* rows, uint32_t (&qb)[M::kKSteps][2]) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(rows + hd * D);
#pragma unroll
    for (int kk = 0; kk < M::kKSteps; ++kk) {
      qb[kk][0] = hd < hpc ? q[kk * 8 + (lane & 3)] : 0u;
      qb[kk][1] = hd < hpc ? q[kk * 8 + 4 + (lane & 3)] : 0u;
    }
  };
  if constexpr (FUSED) {
    uint32_t qb[M::kKSteps][2];
    load_qb(q_in, qb);
    // RoPE ("Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §3) as in decode_mma_kernel
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
    named_barrier_sync(1, kConsumers);
    rotate_q_fragment<D>(qb, cs, lane, a.rope_style);
    if (warp == 0 && hd < hpc) {  // rotated q rows (bf16) for this CTA, and q_rot for the caller
      uint32_t* qo = reinterpret_cast<uint32_t*>(qs + hd * D);
      uint32_t* qg = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.q_out) +
                                                 (static_cast<size_t>(b) * a.Hq + h0 + hd) * D);
#pragma unroll
      for (int kk = 0; kk < M::kKSteps; ++kk) {
        qo[kk * 8 + (lane & 3)] = qb[kk][0];
        qo[kk * 8 + 4 + (lane & 3)] = qb[kk][1];
        if (publisher) {
          qg[kk * 8 + (lane & 3)] = qb[kk][0];
          qg[kk * 8 + 4 + (lane & 3)] = qb[kk][1];
        }
      }
    }
    q_rows = qs;
    named_barrier_sync(1, kConsumers);  // the rotated rows in shared memory are complete
    // the appender warp writes the new token after the barrier: the other warps start streaming
    if (app_warp)
      append_token_q8<D, BITS, PAGED>(a, cs, kraw, vraw, phys, b, g, pos, has_win, lane, appended);
  }

  MmaWarpState<D> st;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;

  if (n_q8 > 0) {
    // q in the INT8 fragment order: lane holds dims 16c + 4(lane%4) + {0..3} of head lane/4,
    // scaled by 2^e so that the head's largest |q| lies in [2^14, 2^15), then rounded to f16.
    uint32_t qh[D / 16][2];
    float down;
    {
      float xq[D / 16][4];
      float amax = 0.f;
      // INT8: row c = dims 16c + 4t .. +3; INT4: rows 2c', 2c'+1 = dims 32c' + 8t .. +3, + 4 .. +7
      const __nv_bfloat16* qr = q_rows + hd * D + (BITS == 8 ? 4 : 8) * (lane & 3);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        uint2 w = make_uint2(0u, 0u);
        const int off = BITS == 8 ? 16 * c : 32 * (c >> 1) + 4 * (c & 1);
        if (hd < hpc) w = *reinterpret_cast<const uint2*>(qr + off);
        xq[c][0] = __uint_as_float(w.x << 16);
        xq[c][1] = __uint_as_float(w.x & 0xffff0000u);
        xq[c][2] = __uint_as_float(w.y << 16);
        xq[c][3] = __uint_as_float(w.y & 0xffff0000u);
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(xq[c][e]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int e = 0;
      if (amax > 0.f && amax <= 3.4e38f) e = min(max(14 - (static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127), -126), 126);
      const float up = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
      down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        if constexpr (BITS == 8) {
          qh[c][0] = pack_f16x2(xq[c][0] * up, xq[c][2] * up);   // dims 4t, 4t+2 as k = 2t, 2t+1
          qh[c][1] = pack_f16x2(xq[c][1] * up, xq[c][3] * up);   // dims 4t+1, 4t+3 as k = 2t+8, 2t+9
        } else {  // slice c of chunk c/2: dims 8t + 2(c&1) + {0, 4} and + {1, 5} (xq rows hold 4 dims)
          const int base = (c >> 1) * 2;   // xq row pair holding dims 32(c/2) + 8t .. +7
          const int o = 2 * (c & 1);
          const float* lo4 = xq[base];      // dims 8t .. 8t+3
          const float* hi4 = xq[base + 1];  // dims 8t+4 .. 8t+7
          qh[c][0] = pack_f16x2(lo4[o] * up, hi4[o] * up);
          qh[c][1] = pack_f16x2(lo4[o + 1] * up, hi4[o + 1] * up);
        }
      }
    }
    float mult[2];
    {
      const float base = a.k_scale[g] * a.scale_log2;
#pragma unroll
      for (int j = 0; j < 2; ++j) mult[j] = base * __shfl_sync(0xffffffffu, down, 4 * (2 * (lane & 3) + j));
    }
    for (int it = 0; it < n_q8; ++it) {
      const int s = it % C::kStages;
      if (!mbar_wait(&full[s], (it / C::kStages) & 1)) {
        flag_error(a.err, RRA_ERR_TIMEOUT);
        break;
      }
      const uint32_t k_base = smem_addr(smem + s * C::kStageBytes), v_base = k_base + C::kTileBytes;
      const int valid = min(C::kTile, end - (start + it * C::kTile));
      if constexpr (BITS == 4 && C::kWarpTokens == 32) {
        const int t0 = warp * 32;
        if (valid == C::kTile)
          q4_step32<D, false>(st, qh, mult, k_base, v_base, t0, valid, lane);
        else if (t0 < valid)
          q4_step32<D, true>(st, qh, mult, k_base, v_base, t0, valid, lane);
      } else
#pragma unroll
      for (int step = 0; step < C::kSteps; ++step) {
        const int t0 = warp * C::kWarpTokens + step * 16;
        if (valid == C::kTile)
          q8_step<D, false>(st, qh, mult, k_base, v_base, t0, valid, lane);
        else if (t0 < valid)
          q8_step<D, true>(st, qh, mult, k_base, v_base, t0, valid, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if constexpr (BITS == 4)
      q4_acc_to_bf16_layout<D>(st, a.v_scale[g], lane);
    else
      q8_acc_to_bf16_layout<D>(st, a.v_scale[g], lane);
  }
  if (n_win > 0) {
    uint32_t qb[M::kKSteps][2];
    load_qb(q_rows, qb);
    for (int it = n_q8; it < n_tiles; ++it) {
      const int s = it % C::kStages;
      if (!mbar_wait(&full[s], (it / C::kStages) & 1)) {
        flag_error(a.err, RRA_ERR_TIMEOUT);
        break;
      }
      uint8_t* kst = smem + s * C::kStageBytes;
      uint8_t* vst = kst + M::kHalves * C::kWinHalf;
      const uint32_t k_base = smem_addr(kst), v_base = smem_addr(vst);
      const int valid = min(wrows, Lw - (it - n_q8) * wrows);
      const int t0 = warp * 16;  // one 16-token step per warp; ring tiles hold up to kWinTile tokens
      if (t0 < C::kWinTile) {
        if (valid == C::kWinTile)
          mma_step<D, false, C::kWinHalf>(st, qb, k_base, v_base, vst, t0, valid, lane, a.scale_log2);
        else if (t0 < valid)
          mma_step<D, true, C::kWinHalf>(st, qb, k_base, v_base, vst, t0, valid, lane, a.scale_log2);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }

  // ------------------------------------------------------------------ merge the 4 warps
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    st.l[j] += __shfl_xor_sync(0xffffffffu, st.l[j], 4);
    st.l[j] += __shfl_xor_sync(0xffffffffu, st.l[j], 8);
    st.l[j] += __shfl_xor_sync(0xffffffffu, st.l[j], 16);
  }
  named_barrier_sync(1, kConsumers);
  // [warps][8 heads][D + 4]: the padded row stride puts the four heads a store instruction covers
  // in distinct banks
  constexpr int kRS = D + 4;
  static_assert(C::kConsumerWarps * M::kMaxHeads * (kRS + 4) * 4 + 2 * M::kMaxHeads * 4 <= C::kRingBytes,
                "the warp merge fits in the ring");
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + C::kConsumerWarps * M::kMaxHeads * kRS;  // [warps][8 heads]
  float* red_l = red_m + C::kConsumerWarps * M::kMaxHeads;
  {
    const int hd0 = 2 * (lane & 3), dl = lane >> 2;
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        red_o[(warp * M::kMaxHeads + hd0 + j) * kRS + 16 * i + dl] = st.o[i][j];
        red_o[(warp * M::kMaxHeads + hd0 + j) * kRS + 16 * i + 8 + dl] = st.o[i][2 + j];
      }
    if (dl == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        red_m[warp * M::kMaxHeads + hd0 + j] = st.m[j];
        red_l[warp * M::kMaxHeads + hd0 + j] = st.l[j];
      }
    }
  }
  named_barrier_sync(1, kConsumers);
  // the warps' weights and the merged (max, sum) once per head, then independent row items
  float* red_w = red_l + C::kConsumerWarps * M::kMaxHeads;  // [warps][heads] weights
  float* red_ml = red_w + C::kConsumerWarps * M::kMaxHeads;  // [heads][2] merged max, sum
  for (int h = threadIdx.x; h < hpc; h += kConsumers) {
    float Mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) Mx = fmaxf(Mx, red_m[w * M::kMaxHeads + h]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) {
      const float wt = Mx != -INFINITY ? exp2f(red_m[w * M::kMaxHeads + h] - Mx) : 0.f;
      lsum = fmaf(wt, red_l[w * M::kMaxHeads + h], lsum);
      red_w[w * M::kMaxHeads + h] = wt;
    }
    red_ml[2 * h] = Mx;
    red_ml[2 * h + 1] = lsum;
  }
  named_barrier_sync(1, kConsumers);
#pragma unroll 4
  for (int idx = threadIdx.x; idx < hpc * D; idx += kConsumers) {
    const int h = idx / D, d = idx - h * D;
    const float Mx = red_ml[2 * h], lsum = red_ml[2 * h + 1];
    float osum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w)
      osum = fmaf(red_w[w * M::kMaxHeads + h], red_o[(w * M::kMaxHeads + h) * kRS + d], osum);
    const size_t bh = static_cast<size_t>(b) * a.Hq + h0 + h;
    if (n_work == 1) {
      static_cast<__nv_bfloat16*>(a.out)[bh * D + d] = __float2bfloat16_rn(lsum > 0.f ? osum / lsum : 0.f);
    } else {
      const size_t ps = bh * a.num_splits + split;
      a.ws_o[ps * D + d] = osum;
      if (d == 0) {
        a.ws_ml[2 * ps] = Mx;
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

template <int D, int BITS, bool PAGED, bool FUSED>
cudaError_t launch_decode_q8_t(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                               const CUtensorMap& kwm, const CUtensorMap& vwm, cudaStream_t st) {
  using C = Q8Cfg<D, BITS>;
  static int done[64] = {0};
  auto kern = decode_q8_kernel<D, BITS, PAGED, FUSED>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_splits * ((a.Hq / a.Hkv) / a.hpc), a.Hkv, a.B);
  return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, st, km, vm, kwm, vwm, a);
}

}  // namespace rra
