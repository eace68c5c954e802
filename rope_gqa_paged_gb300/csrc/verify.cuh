// Multi-query decode (the speculative-verify step) for bf16 caches on the tensor cores.
//
// "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南" §五: the target model checks
// gamma draft tokens in one pass. Each sequence b gets gamma new tokens at positions p_b ..
// p_b + gamma - 1 (already rotated and appended by the append kernel); query token j attends
// tokens [0, p_b + j] -- the cached ones and the new ones up to itself.
//
// One CTA serves one KV head's n_rep x gamma query rows (up to 16: hpc heads x gamma tokens;
// more heads use head slices) over a split-K chunk of the tokens, so every K/V byte read from
// HBM feeds 16 rows. The rows sit on the M dimension of mma.sync.m16n8k16 (FlashAttention-2
// order):
//   S [16 rows x 16 tokens]  = Q [16 x D] . K^T            (K rows through ldmatrix)
//   O [16 rows x D]         += P [16 x 16 tokens] . V       (V through ldmatrix.trans)
// and the score accumulator of two 8-token halves is already the A fragment of P. The causal
// limit of each row masks the new tokens it may not see. The pipeline (TMA into a ring of 32 KB
// stages of 64-dim halves, 128-byte swizzle), the 4-warp token split, the merge of the warps
// and of the splits are those of decode_mma.cuh / decode_kernels.cuh; three CTAs per SM.
#pragma once

#include "decode_mma.cuh"

namespace rra {

constexpr int kVerifyRows = 16;
// The fused verify step (RoPE of the gamma new tokens' q and k, their append and the attention in
// one launch) keeps the sines and cosines of up to this many positions in shared memory; larger
// gamma runs as two launches.
constexpr int kVerifyFusedMaxGamma = 8;

template <int D>
constexpr int verify_smem_bytes(bool fused) {
  return MmaCfg<D>::kSmemBytes + (fused ? (kVerifyFusedMaxGamma - 1) * 4 * (D / 2) * 4 : 0);
}

// Fused step only: rotates the two query rows of the lane's A fragment (rows lane/4 and lane/4 + 8,
// row r = head hh * gamma + token j at position p0 + j) in place, with cos/sin hi/lo of token j at
// cs + j * 2D. Padding rows (r >= rows) stay zero.
template <int D>
__device__ __forceinline__ void rotate_q_rows(uint32_t (&qa)[D / 16][4], const float* cs, int rows, int gamma, int lane,
                                              int style) {
  constexpr int KK = D / 16, HALF = D / 2;
  const int c2 = 2 * (lane & 3);
  auto unpack = [](uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  };
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = (lane >> 2) + 8 * i;
    if (r >= rows) continue;
    const float* c = cs + (r % gamma) * 2 * D;
    if (style == 1) {  // interleaved pairs (2f, 2f + 1): the two halves of each 32-bit word
#pragma unroll
      for (int kk = 0; kk < KK; ++kk)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t& w = qa[kk][hf ? 2 + i : i];
          const int f = (16 * kk + 8 * hf + c2) >> 1;
          float x0, x1;
          unpack(w, x0, x1);
          const float ch = c[f], cl = c[HALF + f], sh = c[2 * HALF + f], sl = c[3 * HALF + f];
          w = pack_bf16x2(rotate_diff(x0, x1, ch, cl, sh, sl), rotate_diff(x1, -x0, ch, cl, sh, sl));
        }
      continue;
    }
    // half-split pairs (f, f + D/2): k-steps kk and kk + KK/2 hold the two members
#pragma unroll
    for (int kk = 0; kk < KK / 2; ++kk)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t& wa = qa[kk][hf ? 2 + i : i];
        uint32_t& wb = qa[kk + KK / 2][hf ? 2 + i : i];
        float a0, a1, b0, b1;
        unpack(wa, a0, a1);
        unpack(wb, b0, b1);
        const int f0 = 16 * kk + 8 * hf + c2, f1 = f0 + 1;
        const float ch0 = c[f0], cl0 = c[HALF + f0], sh0 = c[2 * HALF + f0], sl0 = c[3 * HALF + f0];
        const float ch1 = c[f1], cl1 = c[HALF + f1], sh1 = c[2 * HALF + f1], sl1 = c[3 * HALF + f1];
        wa = pack_bf16x2(rotate_diff(a0, b0, ch0, cl0, sh0, sl0), rotate_diff(a1, b1, ch1, cl1, sh1, sl1));
        wb = pack_bf16x2(rotate_diff(b0, -a0, ch0, cl0, sh0, sl0), rotate_diff(b1, -a1, ch1, cl1, sh1, sl1));
      }
  }
}

template <int D>
struct VerifyState {
  float o[D / 8][4];  // n-tile nt: rows lane/4 and lane/4 + 8, dims 8 nt + 2 (lane % 4) + {0, 1}
  float m[2], l[2];   // rows lane/4 and lane/4 + 8 (running max in log2 units, lane-partial sum)
};

// (lo, hi) rounded to bf16 pairs: `hi` holds the nearest bf16 values, `lo` the bf16 rounding of
// what they leave out.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}

// One 16-token slice of a stage for one warp. t0: the slice's first row in the stage; tok0: its
// token index; lim0 / lim1: the last token rows lane/4 and lane/4 + 8 may attend (-1: padding).
// CHECK: rows at or past `valid` of the stage are not tokens of this chunk; their V rows are
// zeroed first so that no stale value reaches the tensor cores. SPLIT_P: P enters P.V as a
// bf16 part plus the bf16 rounding of its remainder (for rows that attend few tokens).
template <int D, bool CHECK, bool SPLIT_P = true>
__device__ __forceinline__ void verify_step(VerifyState<D>& st, const uint32_t (&qa)[D / 16][4], uint32_t k_base,
                                            uint32_t v_base, uint8_t* v_gen, int t0, int tok0, int valid, int lim0,
                                            int lim1, int lane, float scale_log2) {
  using C = MmaCfg<D>;
  if (CHECK) {
    const int first = max(valid - t0, 0);
    if (first < 16) {
      for (int idx = lane; idx < (16 - first) * C::kHalves * 8; idx += 32) {
        const int r = t0 + first + idx / (C::kHalves * 8);
        const int h = (idx / 8) % C::kHalves, c = idx % 8;
        *reinterpret_cast<uint4*>(v_gen + h * C::kHalfBytes + swz(r, c)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
  }
  const int mat = lane >> 3, t = lane & 3;
  // scores: matrices (tokens 0-7 | 8-15) x (dims 16kk..+7 | +8..+15) give the B fragments of both halves
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int r = t0 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t b[4];
      ldsm_x4(k_base + (kk >> 2) * C::kHalfBytes + swz(r, ((kk & 3) << 1) + (mat & 1)), b);
      mma_bf16(s[0], qa[kk], b[0], b[1]);
      mma_bf16(s[1], qa[kk], b[2], b[3]);
    }
  }
  // s[n][c]: row lane/4 (c < 2) or lane/4 + 8, token tok0 + 8n + 2t + (c & 1)
  float x[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int rel = 8 * n + 2 * t + (c & 1);
      const bool ok = tok0 + rel <= (c < 2 ? lim0 : lim1) && (!CHECK || t0 + rel < valid);
      x[n][c] = ok ? s[n][c] * scale_log2 : -INFINITY;
    }
  float mx[2] = {fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1])),
                 fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]))};
  bool grow = false;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
    mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    mx[i] = fmaxf(st.m[i], mx[i]);
    grow |= mx[i] > st.m[i];
  }
  if (__any_sync(0xffffffffu, grow)) {
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      alpha[i] = mx[i] > st.m[i] ? exp2f(st.m[i] - mx[i]) : 1.f;
      st.l[i] *= alpha[i];
      st.m[i] = mx[i];
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      st.o[nt][0] *= alpha[0];
      st.o[nt][1] *= alpha[0];
      st.o[nt][2] *= alpha[1];
      st.o[nt][3] *= alpha[1];
    }
  }
  const float mref[2] = {st.m[0] == -INFINITY ? 0.f : st.m[0], st.m[1] == -INFINITY ? 0.f : st.m[1]};
  float p[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) p[n][c] = exp2f(x[n][c] - mref[c >> 1]);
  st.l[0] += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
  st.l[1] += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
  // P as the A operand (rows x k = tokens): the two 8-token halves of the score fragment, as a
  // bf16 part and the bf16 rounding of its remainder (p = hi + lo to ~2^-17: a lone bf16 P,
  // 2^-9, shows in rows that attend only a few tokens)
  uint32_t pa[4], pl[4];
  split_bf16x2(p[0][0], p[0][1], pa[0], pl[0]);
  split_bf16x2(p[0][2], p[0][3], pa[1], pl[1]);
  split_bf16x2(p[1][0], p[1][1], pa[2], pl[2]);
  split_bf16x2(p[1][2], p[1][3], pa[3], pl[3]);
  {
    // matrices (tokens 0-7 | 8-15) x (dims 16j..+7 | +8..+15) through ldmatrix.trans: B fragments of two n-tiles
    const int r = t0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      uint32_t b[4];
      ldsm_x4_trans(v_base + (j >> 2) * C::kHalfBytes + swz(r, ((j & 3) << 1) + (mat >> 1)), b);
      mma_bf16(st.o[2 * j], pa, b[0], b[1]);
      mma_bf16(st.o[2 * j + 1], pa, b[2], b[3]);
      if (SPLIT_P) {
        mma_bf16(st.o[2 * j], pl, b[0], b[1]);
        mma_bf16(st.o[2 * j + 1], pl, b[2], b[3]);
      }
    }
  }
}

// Output row of virtual partial row vr (CTA rows are contiguous: 16 per (sequence, KV head,
// head slice)); CTA row r = hh * gamma + j is head h0 + hh of new token j.
struct VerifyRows {
  int Hq, Hkv, n_rep, slices, hpc, gamma;
  __device__ size_t operator()(size_t vr) const {
    const size_t cta = vr / kVerifyRows;
    const int r = static_cast<int>(vr - cta * kVerifyRows);
    const int slice = static_cast<int>(cta % slices);
    const size_t bg = cta / slices;
    const int g = static_cast<int>(bg % Hkv);
    const size_t b = bg / Hkv;
    const int hh = r / gamma, j = r - hh * gamma;
    return (b * gamma + j) * Hq + g * n_rep + slice * hpc + hh;
  }
};

// FUSED: the whole verify step in this launch. a.q holds the unrotated q of the gamma new tokens
// (gamma <= kVerifyFusedMaxGamma); the consumer warps take sin/cos of the gamma positions once per
// CTA (rope_cos_sin, as the decode step), rotate their query rows in registers, and split-0
// CTAs publish q_rot. A CTA whose chunk holds new tokens rotates their k_new and writes them and
// v_new into the cache, one warp per token, and its producer waits for those writes (an mbarrier
// with one arrival per token) before the TMA of the first tile that holds a new token. Head-slice
// CTAs of that chunk write identical bytes.
template <int D, bool PAGED, bool FUSED = false>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads, RRA_MMA_CTAS_PER_SM)
    decode_verify_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                         const DecodeArgs a) {
  using C = MmaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int gamma = a.gamma;
  const int n_rep = a.Hq / a.Hkv;
  const int hpc = a.hpc;
  const int slices = n_rep / hpc;
  const int split = blockIdx.x / slices;
  const int slice = blockIdx.x - split * slices;
  const int g = blockIdx.y;
  const int h0 = g * n_rep + slice * hpc;
  const int b = blockIdx.z;
  const int rows = hpc * gamma;  // real rows of this CTA (<= 16)
  const size_t vbase = ((static_cast<size_t>(b) * a.Hkv + g) * slices + slice) * kVerifyRows;
  const VerifyRows out_row{a.Hq, a.Hkv, n_rep, slices, hpc, gamma};

  pdl_launch_dependents();
  pdl_wait();  // the kernel before this one (the append, or the previous step) has finished
  // the chunk's block ids load alongside the position
  ChunkBlockIds<(kMmaTableEntries + C::kThreads - 1) / C::kThreads> pre_ids;
  if constexpr (PAGED) pre_ids.load(a, b, (split * a.chunk) >> a.log2_bs, threadIdx.x, C::kThreads);

  const int p0 = a.positions[b];
  int L = p0 + gamma;
  if (p0 < 0 || L > a.capacity) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  const int start = split * a.chunk;
  const int n_work = (L + a.chunk - 1) / a.chunk;
  if (start >= L) return;
  const int end = min(L, start + a.chunk);
  const int n_tiles = (end - start + C::kTile - 1) / C::kTile;
  // fused step: new tokens app_lo .. app_hi - 1 lie in this chunk and are appended here
  const int app_lo = FUSED ? max(p0, start) : 0, app_hi = FUSED ? min(L, end) : 0;
  const bool appender = FUSED && app_lo < app_hi;
  const int first_new_tile = appender ? (app_lo - start) / C::kTile : n_tiles;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + C::kStages;
  uint64_t* appended = empty + C::kStages;
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kOffTable);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    mbar_init(appended, appender ? app_hi - app_lo : 1);
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
    // Lane 0 waits for the stage and sets its byte count; the stage's copies then go out from
    // all lanes at once (as in decode_mma_kernel).
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
        } else if (it == first_new_tile && !mbar_wait(appended, 0)) {  // the new tokens start in this tile
          flag_error(a.err, RRA_ERR_TIMEOUT);
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(bytes));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      for (int c = lane; c < 2 * C::kHalves * nblk; c += 32) {
        const int kv = c & 1, h = (c >> 1) % C::kHalves, jb = (c >> 1) / C::kHalves;
        uint8_t* dst = (kv ? vst : kst) + h * C::kHalfBytes;
        const CUtensorMap* map = kv ? &v_map : &k_map;
        if constexpr (PAGED) {
          const int bs = 1 << a.log2_bs;
          if (bs <= C::kTile)
            tma_g2s_4d(dst + jb * bs * 128, map, 64 * h, g, 0, tbl[(t0 >> a.log2_bs) - first_blk + jb], &full[s]);
          else
            tma_g2s_4d(dst, map, 64 * h, g, t0 & (bs - 1), tbl[(t0 >> a.log2_bs) - first_blk], &full[s]);
        } else {
          tma_g2s_3d(dst, map, 64 * h, t0, b * a.Hkv + g, &full[s]);
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
  const int rg = lane >> 2, t = lane & 3;
  // Q as the A operand: rows rg and rg + 8, dims 16kk + 2t + {0,1} (and + 8)
  uint32_t qa[D / 16][4];
  int lim[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = rg + 8 * i;
    const int hh = r / gamma, j = r - hh * gamma;
    lim[i] = r < rows ? p0 + j : -1;
    const uint32_t* q = reinterpret_cast<const uint32_t*>(
        static_cast<const __nv_bfloat16*>(a.q) + ((static_cast<size_t>(b) * gamma + j) * a.Hq + h0 + hh) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][i] = r < rows ? q[kk * 8 + t] : 0u;
      qa[kk][2 + i] = r < rows ? q[kk * 8 + 4 + t] : 0u;
    }
  }
  if constexpr (FUSED) {
    // RoPE ("Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §3) at positions p0 .. p0 + gamma - 1:
    // sine and cosine of (p0 + j) * theta_i as float32 hi + lo pairs (rope_cos_sin) for the
    // error-free rotation, spread over the consumer threads; [gamma][4][D/2] floats.
    float* cs = reinterpret_cast<float*>(smem + C::kOffCs);
    for (int e = threadIdx.x; e < gamma * (D / 2); e += kConsumers) {
      const int j = e / (D / 2), i = e - j * (D / 2);
      float* c = cs + j * 2 * D;
      rope_cos_sin(p0 + j, a.rope_phi[i], c[i], c[D / 2 + i], c[D + i], c[3 * (D / 2) + i]);
    }
    named_barrier_sync(1, kConsumers);
    rotate_q_rows<D>(qa, cs, rows, gamma, lane, a.rope_style);
    if (warp == 0 && split == 0) {  // publish q_rot (rounded to bf16, as used here)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = rg + 8 * i;
        if (r >= rows) continue;
        const int hh = r / gamma, j = r - hh * gamma;
        uint32_t* qo = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.q_out) +
                                                   ((static_cast<size_t>(b) * gamma + j) * a.Hq + h0 + hh) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          qo[kk * 8 + t] = qa[kk][i];
          qo[kk * 8 + 4 + t] = qa[kk][2 + i];
        }
      }
    }
    if (appender) {  // one warp per new token of this chunk
      for (int pos = app_lo + warp; pos < app_hi; pos += C::kConsumerWarps) {
        const int j = pos - p0;
        const size_t off = ((static_cast<size_t>(b) * gamma + j) * a.Hkv + g) * D + lane * (D / 32);
        const uint32_t* kn = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.k_new) + off);
        const uint32_t* vn = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.v_new) + off);
        uint32_t kraw[D / 64], vraw[D / 64];
#pragma unroll
        for (int w = 0; w < D / 64; ++w) {
          kraw[w] = kn[w];
          vraw[w] = vn[w];
        }
        int phys = 0;
        if constexpr (PAGED) phys = a.block_table[static_cast<size_t>(b) * a.max_blocks_per_seq + (pos >> a.log2_bs)];
        append_token_bf16<D, PAGED>(a, cs + j * 2 * D, kraw, vraw, phys, b, g, pos, lane, appended);
      }
    }
  }
  // rows attend at least p0 + 1 keys: from 256 on, a bf16 P is exact enough (the split of P into
  // a bf16 part and its remainder is for rows that see a few tokens, as in the prefill kernel)
  const bool precise = p0 < 256;
  VerifyState<D> st;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) st.o[nt][0] = st.o[nt][1] = st.o[nt][2] = st.o[nt][3] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % C::kStages;
    if (!mbar_wait(&full[s], (it / C::kStages) & 1)) {
      flag_error(a.err, RRA_ERR_TIMEOUT);
      break;
    }
    uint8_t* kst = smem + s * C::kStageBytes;
    uint8_t* vst = kst + C::kHalves * C::kHalfBytes;
    const uint32_t k_base = smem_addr(kst), v_base = smem_addr(vst);
    const int tile0 = start + it * C::kTile;
    const int valid = min(C::kTile, end - tile0);
    // the causal mask only bites in tiles that reach the new tokens
    const bool edge = valid < C::kTile || tile0 + C::kTile > p0;
#pragma unroll
    for (int step = 0; step < C::kSteps; ++step) {
      const int t0 = warp * C::kWarpTokens + step * 16;
      if (!edge) {
        if (precise)
          verify_step<D, false, true>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                      a.scale_log2);
        else
          verify_step<D, false, false>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                       a.scale_log2);
      } else if (t0 < valid) {
        if (precise)
          verify_step<D, true, true>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                     a.scale_log2);
        else
          verify_step<D, true, false>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                      a.scale_log2);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ------------------------------------------------------------------ merge the 4 warps
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    st.l[i] += __shfl_xor_sync(0xffffffffu, st.l[i], 1);
    st.l[i] += __shfl_xor_sync(0xffffffffu, st.l[i], 2);
  }
  named_barrier_sync(1, kConsumers);
  // [warps][16 rows][D + 8]: the padded row stride keeps the float2 stores of a fragment's eight
  // rows in distinct banks
  constexpr int kRS = D + 8;
  static_assert(C::kConsumerWarps * kVerifyRows * (kRS + 4) * 4 + 2 * kVerifyRows * 4 <= C::kRingBytes,
                "the warp merge fits in the ring");
  float* red_o = reinterpret_cast<float*>(smem);
  float* red_m = red_o + C::kConsumerWarps * kVerifyRows * kRS;    // [warps][16 rows]
  float* red_l = red_m + C::kConsumerWarps * kVerifyRows;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    *reinterpret_cast<float2*>(&red_o[(warp * kVerifyRows + rg) * kRS + 8 * nt + 2 * t]) =
        make_float2(st.o[nt][0], st.o[nt][1]);
    *reinterpret_cast<float2*>(&red_o[(warp * kVerifyRows + rg + 8) * kRS + 8 * nt + 2 * t]) =
        make_float2(st.o[nt][2], st.o[nt][3]);
  }
  if (t == 0) {
    red_m[warp * kVerifyRows + rg] = st.m[0];
    red_m[warp * kVerifyRows + rg + 8] = st.m[1];
    red_l[warp * kVerifyRows + rg] = st.l[0];
    red_l[warp * kVerifyRows + rg + 8] = st.l[1];
  }
  named_barrier_sync(1, kConsumers);
  // the warps' weights and the merged (max, sum) once per row, then independent row items
  float* red_w = red_l + C::kConsumerWarps * kVerifyRows;   // [warps][16 rows] weights
  float* red_ml = red_w + C::kConsumerWarps * kVerifyRows;  // [16 rows][2] merged max, sum
  for (int r = threadIdx.x; r < rows; r += kConsumers) {
    float Mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) Mx = fmaxf(Mx, red_m[w * kVerifyRows + r]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) {
      const float wt = Mx != -INFINITY ? exp2f(red_m[w * kVerifyRows + r] - Mx) : 0.f;
      lsum = fmaf(wt, red_l[w * kVerifyRows + r], lsum);
      red_w[w * kVerifyRows + r] = wt;
    }
    red_ml[2 * r] = Mx;
    red_ml[2 * r + 1] = lsum;
  }
  named_barrier_sync(1, kConsumers);
#pragma unroll 2
  for (int idx = threadIdx.x; idx < rows * D; idx += kConsumers) {
    const int r = idx / D, d = idx - r * D;
    const float Mx = red_ml[2 * r], lsum = red_ml[2 * r + 1];
    float osum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w)
      osum = fmaf(red_w[w * kVerifyRows + r], red_o[(w * kVerifyRows + r) * kRS + d], osum);
    if (n_work == 1) {
      static_cast<__nv_bfloat16*>(a.out)[out_row(vbase + r) * D + d] = __float2bfloat16_rn(lsum > 0.f ? osum / lsum : 0.f);
    } else {
      const size_t ps = (vbase + r) * a.num_splits + split;
      a.ws_o[ps * D + d] = osum;
      if (d == 0) {
        a.ws_ml[2 * ps] = Mx;
        a.ws_ml[2 * ps + 1] = lsum;
      }
    }
  }
  if (n_work > 1) {
    __shared__ int s_last;
    finish_split_rows<__nv_bfloat16, D, VerifyRows, false>(a, vbase, rows, split, n_work,
                                                           reinterpret_cast<float*>(smem), &s_last, threadIdx.x,
                                                           kConsumers, out_row, C::kRingBytes);
  }
}

template <int D, bool PAGED, bool FUSED>
cudaError_t launch_decode_verify_t(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                                   cudaStream_t st) {
  using C = MmaCfg<D>;
  constexpr int kSmem = verify_smem_bytes<D>(FUSED);
  static int done[64] = {0};
  auto kern = decode_verify_kernel<D, PAGED, FUSED>;
  cudaError_t e = ensure_smem(kern, kSmem, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_splits * ((a.Hq / a.Hkv) / a.hpc), a.Hkv, a.B);
  return launch_pdl(kern, grid, dim3(C::kThreads), kSmem, st, km, vm, a);
}

}  // namespace rra
