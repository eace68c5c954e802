// Prefill: causal attention of a whole prompt (or of a chunk of one after a cached prefix) on the
// tensor cores, FlashAttention-style.
//
// "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南" §三: FlashAttention computes
// softmax(Q K^T / sqrt(d)) V block by block with a running max and sum, never writing the
// T x T score matrix, which is what lets a 128K prompt fit (the page's FA-2 vs standard figure).
// Here the T prompt tokens of sequence b sit at positions p_b .. p_b + T - 1, are already rotated
// and in the cache (the append kernel with gamma = T), and token t attends tokens [0, p_b + t].
//
// One CTA owns 64 query rows of one KV head (hpc heads x 64/hpc tokens; hpc divides n_rep and
// 64), four consumer warps with 16 rows each; every warp takes every 16-token slice of each
// 64-token K/V stage (the same TMA pipeline as the decode kernels) with the verify kernel's
// warp step, so each K/V byte brought into shared memory serves 64 rows. The CTA streams keys
// [0, its last row's position]: the slices past a warp's own last row are skipped, and the
// query blocks are launched longest first. No split-K: each warp normalises and writes its rows.
// Whole 32-token windows go through a two-slice step (more independent mma chains per warp);
// two CTAs per SM leave the registers for it.
#pragma once

#include "verify.cuh"

namespace rra {

constexpr int kPrefillRows = 64;

// 32 tokens of a stage for one warp (rows t0 .. t0+31, all within the chunk), bf16 P: the
// verify step on two 16-token slices at once -- four independent score chains instead of two,
// one softmax reduction and at most one rescale per 32 tokens. lim0 / lim1 as in verify_step.
template <int D>
__device__ __forceinline__ void prefill_step32(VerifyState<D>& st, const uint32_t (&qa)[D / 16][4], uint32_t k_base,
                                               uint32_t v_base, int t0, int tok0, int lim0, int lim1, int lane,
                                               float scale_log2) {
  using C = MmaCfg<D>;
  const int mat = lane >> 3, t = lane & 3;
  float s[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
  {
    const int r = t0 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t b[4], c[4];
      const uint32_t off = (kk >> 2) * C::kHalfBytes;
      ldsm_x4(k_base + off + swz(r, ((kk & 3) << 1) + (mat & 1)), b);
      ldsm_x4(k_base + off + swz(r + 16, ((kk & 3) << 1) + (mat & 1)), c);
      mma_bf16(s[0], qa[kk], b[0], b[1]);
      mma_bf16(s[1], qa[kk], b[2], b[3]);
      mma_bf16(s[2], qa[kk], c[0], c[1]);
      mma_bf16(s[3], qa[kk], c[2], c[3]);
    }
  }
  float x[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = tok0 + 8 * n + 2 * t + (c & 1);
      x[n][c] = tok <= (c < 2 ? lim0 : lim1) ? s[n][c] * scale_log2 : -INFINITY;
    }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    mx[0] = fmaxf(mx[0], fmaxf(x[n][0], x[n][1]));
    mx[1] = fmaxf(mx[1], fmaxf(x[n][2], x[n][3]));
  }
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
  uint32_t pa[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float p[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) p[n][c] = exp2f(x[2 * h + n][c] - mref[c >> 1]);
    st.l[0] += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
    st.l[1] += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
    pa[h][0] = pack_bf16x2(p[0][0], p[0][1]);
    pa[h][1] = pack_bf16x2(p[0][2], p[0][3]);
    pa[h][2] = pack_bf16x2(p[1][0], p[1][1]);
    pa[h][3] = pack_bf16x2(p[1][2], p[1][3]);
  }
  {
    const int r = t0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      uint32_t b[4], c[4];
      const uint32_t off = (j >> 2) * C::kHalfBytes;
      ldsm_x4_trans(v_base + off + swz(r, ((j & 3) << 1) + (mat >> 1)), b);
      ldsm_x4_trans(v_base + off + swz(r + 16, ((j & 3) << 1) + (mat >> 1)), c);
      mma_bf16(st.o[2 * j], pa[0], b[0], b[1]);
      mma_bf16(st.o[2 * j + 1], pa[0], b[2], b[3]);
      mma_bf16(st.o[2 * j], pa[1], c[0], c[1]);
      mma_bf16(st.o[2 * j + 1], pa[1], c[2], c[3]);
    }
  }
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                   const DecodeArgs a) {
  using C = MmaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int T = a.gamma;
  const int n_rep = a.Hq / a.Hkv;
  const int hpc = a.hpc;
  const int qt = kPrefillRows / hpc;  // prompt tokens per CTA
  const int slices = n_rep / hpc;
  const int n_qb = (T + qt - 1) / qt;
  // One CTA per (query block, KV head, head slice), in index order: band by band of KV heads
  // whose K and V fit in L2 together, the longest causal blocks of a band first.
  const int hs_band = (a.kv_band > 0 ? a.kv_band : a.Hkv) * slices;  // (KV head, slice) pairs per band
  const int band_ctas = n_qb * hs_band;
  const int band = static_cast<int>(blockIdx.x) / band_ctas;
  const int j = static_cast<int>(blockIdx.x) - band * band_ctas;
  const int qb = n_qb - 1 - j / hs_band;
  const int hs = band * hs_band + j % hs_band;
  const int slice = hs % slices;
  const int g = hs / slices;
  const int h0 = g * n_rep + slice * hpc;
  const int b = blockIdx.z;
  const int q0 = qb * qt;

  pdl_launch_dependents();
  pdl_wait();  // the append kernel before this one wrote the prompt's K, V and q_rot

  const int p0 = a.positions[b];
  if (p0 < 0 || p0 + T > a.capacity) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.err, RRA_ERR_POSITION);
    return;
  }
  const int q_end = min(T, q0 + qt);
  const int end = p0 + q_end;  // keys [0, end)
  const int n_tiles = (end + C::kTile - 1) / C::kTile;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + C::kStages;
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kOffTable);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer
  if (warp == C::kConsumerWarps) {
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      const int32_t* row = PAGED ? a.block_table + static_cast<size_t>(b) * a.max_blocks_per_seq : nullptr;
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1)) {
          flag_error(a.err, RRA_ERR_TIMEOUT);
          break;
        }
        const int t0 = it * C::kTile;
        uint8_t* kst = smem + s * C::kStageBytes;
        uint8_t* vst = kst + C::kHalves * C::kHalfBytes;
        if constexpr (PAGED) {
          const int bs = 1 << a.log2_bs;
          auto block_id = [&](int j) {
            int id = row[j];
            if (id < 0 || id >= a.num_blocks) {
              flag_error(a.err, RRA_ERR_BLOCK_ID);
              id = 0;
            }
            return id;
          };
          if (bs <= C::kTile) {
            const int n = min(C::kTile, end - t0);
            const int nblk = (n + bs - 1) >> a.log2_bs;
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * C::kHalves * nblk * bs * 128));
            for (int jb = 0; jb < nblk; ++jb) {
              const int phys = block_id((t0 >> a.log2_bs) + jb);
#pragma unroll
              for (int h = 0; h < C::kHalves; ++h) {
                tma_g2s_4d(kst + h * C::kHalfBytes + jb * bs * 128, &k_map, 64 * h, g, 0, phys, &full[s]);
                tma_g2s_4d(vst + h * C::kHalfBytes + jb * bs * 128, &v_map, 64 * h, g, 0, phys, &full[s]);
              }
            }
          } else {
            const int phys = block_id(t0 >> a.log2_bs);
            const int off = t0 & (bs - 1);
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * C::kHalves * C::kTile * 128));
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
              tma_g2s_4d(kst + h * C::kHalfBytes, &k_map, 64 * h, g, off, phys, &full[s]);
              tma_g2s_4d(vst + h * C::kHalfBytes, &v_map, 64 * h, g, off, phys, &full[s]);
            }
          }
        } else {
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * C::kHalves * C::kTile * 128));
          const int bg = b * a.Hkv + g;
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h) {
            tma_g2s_3d(kst + h * C::kHalfBytes, &k_map, 64 * h, t0, bg, &full[s]);
            tma_g2s_3d(vst + h * C::kHalfBytes, &v_map, 64 * h, t0, bg, &full[s]);
          }
        }
        issued = it + 1;
      }
      for (int it = issued > C::kStages ? issued - C::kStages : 0; it < issued; ++it)
        mbar_wait(&full[it % C::kStages], (it / C::kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int rg = lane >> 2, t = lane & 3;
  // this warp's 16 rows: CTA rows 16 warp + r, r = tt * hpc + hh -> prompt token q0 + tt, head h0 + hh
  uint32_t qa[D / 16][4];
  int lim[2];
  int last = -1;  // the last key any of this warp's rows attends
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = 16 * warp + rg + 8 * i;
    const int tt = r / hpc, hh = r - tt * hpc;
    const bool real = q0 + tt < T;
    lim[i] = real ? p0 + q0 + tt : -1;
    const uint32_t* q = reinterpret_cast<const uint32_t*>(
        static_cast<const __nv_bfloat16*>(a.q) + ((static_cast<size_t>(b) * T + q0 + tt) * a.Hq + h0 + hh) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][i] = real ? q[kk * 8 + t] : 0u;
      qa[kk][2 + i] = real ? q[kk * 8 + 4 + t] : 0u;
    }
  }
  {
    const int r_last = min(16 * warp + 15, qt * hpc - 1);
    last = min(p0 + q0 + r_last / hpc, end - 1);
  }
  // rows that see few keys keep P to ~2^-17 (bf16 part + bf16 remainder); the rest use bf16 P
  const bool precise = p0 + q0 < 256;
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
    const int tile0 = it * C::kTile;
    const int valid = min(C::kTile, end - tile0);
#pragma unroll 1
    for (int t0 = 0; t0 < valid && tile0 + t0 <= last;) {
      if (!precise && t0 + 32 <= valid) {  // two whole slices at once
        prefill_step32<D>(st, qa, k_base, v_base, t0, tile0 + t0, lim[0], lim[1], lane, a.scale_log2);
        t0 += 32;
        continue;
      }
      const bool partial = t0 + 16 > valid;
      if (precise) {
        if (partial)
          verify_step<D, true, true>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                     a.scale_log2);
        else
          verify_step<D, false, true>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                      a.scale_log2);
      } else {
        if (partial)
          verify_step<D, true, false>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                      a.scale_log2);
        else
          verify_step<D, false, false>(st, qa, k_base, v_base, vst, t0, tile0 + t0, valid, lim[0], lim[1], lane,
                                       a.scale_log2);
      }
      t0 += 16;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ------------------------------------------------------------------ this warp's rows
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    st.l[i] += __shfl_xor_sync(0xffffffffu, st.l[i], 1);
    st.l[i] += __shfl_xor_sync(0xffffffffu, st.l[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = 16 * warp + rg + 8 * i;
    const int tt = r / hpc, hh = r - tt * hpc;
    if (q0 + tt >= T) continue;
    const float inv = st.l[i] > 0.f ? 1.f / st.l[i] : 0.f;
    uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) +
                                                ((static_cast<size_t>(b) * T + q0 + tt) * a.Hq + h0 + hh) * D);
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) out[4 * nt + t] = pack_bf16x2(st.o[nt][2 * i] * inv, st.o[nt][2 * i + 1] * inv);
  }
}

template <int D, bool PAGED>
cudaError_t launch_prefill_t(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t st) {
  using C = MmaCfg<D>;
  static int done[64] = {0};
  auto kern = prefill_kernel<D, PAGED>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const int qt = kPrefillRows / a.hpc;
  const dim3 grid(((a.gamma + qt - 1) / qt) * (a.Hkv * ((a.Hq / a.Hkv) / a.hpc)), 1, a.B);
  return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, st, km, vm, a);
}

}  // namespace rra
