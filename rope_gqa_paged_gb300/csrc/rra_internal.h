// Launch interface between the C ABI (rra_abi.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rra.h"

namespace rra {

constexpr int kMaxHeadDim = 512;
constexpr int kMaxDecodeHeadDim = 128;

struct RopeArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  const int32_t* positions;
  void* q_out;
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;  // nullptr: contiguous cache
  int max_blocks_per_seq;
  int log2_bs;
  int num_blocks;
  int max_len;
  int B, Hq, Hkv, D;
  int rope_style;
  int32_t* err;
  int gamma;                    // new tokens per sequence (0 or 1: one); q/k_new/v_new/q_out [B*gamma, H, D]
  // INT8 caches only: k_cache / v_cache hold int8 codes, quantised with these per-KV-head
  // scales; with window > 0 the bf16 values also go to ring slot pos % window.
  const float* k_scale;
  const float* v_scale;
  void* k_win;                  // bf16 [B, Hkv, window, D]
  void* v_win;
  int window;
  uint32_t rope_phi[kMaxHeadDim / 2][3];  // theta_i / 2pi as 96-bit fractions (fill_rope_phi)
};

struct DecodeArgs {
  const void* q;                // q_rot [B, Hq, D]
  const void* k;                // contiguous caches [B, Hkv, max_len, D] (paged: pools, read via tensor maps)
  const void* v;
  const int32_t* seq_lens;      // [B]
  const int32_t* block_table;   // [B, max_blocks_per_seq] (paged only)
  int max_blocks_per_seq;
  int log2_bs;
  int num_blocks;
  void* out;                    // [B, Hq, D]
  float* ws_o;                  // [B, Hq, splits, D] unnormalised partial outputs
  float* ws_ml;                 // [B, Hq, splits, 2] (running max in log2 units, running sum)
  float* ws2_o;                 // [B, Hq, num_groups, D] level-2 partials (groups of kMergeFanIn splits)
  float* ws2_ml;                // [B, Hq, num_groups, 2]
  int* counters;                // [B, Hq] arrivals per (sequence, first head of a CTA's head slice)
  int* group_counters;          // [B, Hq, num_groups] arrivals per group of splits
  int num_groups;               // ceil(num_splits / kMergeFanIn)
  int B, Hq, Hkv, D;
  int max_len;                  // contiguous row stride in tokens
  int capacity;                 // tokens a sequence can hold
  int hpc;                      // query heads per CTA (divides Hq / Hkv)
  int num_splits;               // effective split count
  int chunk;                    // tokens per split (a multiple of the tile)
  int narrow;                   // bf16 decode kernel: 2 consumer warps, 32-token stages, 4 CTAs per SM
  float scale_log2;             // softmax scale * log2(e)
  int32_t* err;
  // Fused step (RoPE + append inside the decode kernel). When `positions` is set, L_b =
  // positions[b] + 1 and seq_lens is unused; the fused kernel also reads unrotated q,
  // rotates it, writes q_out, and appends rotated k_new / raw v_new at the position.
  const int32_t* positions;
  // Test of the timeout path (rra_test_hold_append): the append warp of a fused bf16 step writes
  // the new token but never arrives on the append barrier, so the producer's bounded wait for it
  // runs out and RRA_ERR_TIMEOUT is set. 0 in every ordinary call.
  int test_hold_append;
  const void* k_new;            // [B, Hkv, D]
  const void* v_new;            // [B, Hkv, D]
  void* q_out;                  // [B, Hq, D], must not overlap q
  int rope_style;
  // INT8 caches (decode_q8.cuh): k / v hold codes with these per-KV-head scales; with
  // window > 0 the `window` most recent tokens are read from the bf16 rings instead, and the
  // last of the num_splits partial slots belongs to the ring.
  const float* k_scale;
  const float* v_scale;
  void* k_win;                  // bf16 [B, Hkv, window, D]
  void* v_win;
  int window;
  int code_bits;                // 8 (INT8 codes) or 4 (INT4, two per byte)
  // Speculative verify (verify.cuh): gamma new tokens per sequence at positions[b] ..
  // positions[b] + gamma - 1; q and out are [B, gamma, Hq, D].
  int gamma;
  // Prefill: CTAs run band by band, a band being kv_band KV groups (0: all of them) whose keys
  // and values fit in L2 together, longest query blocks first within a band.
  int kv_band;
  uint32_t rope_phi[kMaxDecodeHeadDim / 2][3];  // theta_i / 2pi as 96-bit fractions (fill_rope_phi)
};

// Tokens per pipeline stage for a head_dim and element size: K + V tiles of 16 KB.
inline int decode_tile_tokens(int D, int elem_bytes) { return 8192 / (D * elem_bytes); }
// Most block-table entries one split may need (bounds the per-CTA table copy).
constexpr int kMaxTableEntries = 2048;
// Most splits per sequence (the CTA that merges them stages 2 x 8 heads x splits floats in
// shared memory).
constexpr int kMaxSplits = 1024;
// Splits merged by one CTA in one level; more splits are merged in two levels: groups of
// merge_fanin(splits) splits (about the square root of the split count, at least 8), then the
// groups, so that the merge of a group and the merge of the groups read about as many partials
// each (one group of 32 then 2 groups read 34 rows per head at 57 splits; 8 then 8 read 16).
constexpr int kMergeFanIn = 32;
__host__ __device__ inline int merge_fanin(int splits) {
  if (splits <= kMergeFanIn) return kMergeFanIn;
  int f = 8;
  while (f < kMergeFanIn && f * f < splits) ++f;
  return f;
}
__host__ __device__ inline int merge_groups(int splits) {
  const int f = merge_fanin(splits);
  return (splits + f - 1) / f;
}

// rra_decode_attn_paged with the split arrival counters at `counters` (decode_counter_ints
// int32s, all zero when the kernel starts) and only the partial arrays (decode_partial_bytes)
// in `workspace`. counters == nullptr: exactly rra_decode_attn_paged.
int decode_attn_paged_ext(const void* q_rot, const void* k_pool, const void* v_pool, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* seq_lens, int block_size, int num_blocks, void* out,
                          int B, int Hq, int Hkv, int D, float scale, int num_splits, void* workspace,
                          size_t ws_bytes, int* counters, rra_dtype dt, int32_t* err_flag, void* stream);
// Bytes of the partial arrays, and int32 arrival counters, of a decode with an effective split
// count (both 0 when splits <= 1).
size_t decode_partial_bytes(int B, int Hq, int D, int splits);
size_t decode_counter_ints(int B, int Hq, int splits);

// theta_i / 2pi (theta_i = base^(-2i/D), i < D/2, float64) as 96-bit binary fractions, least
// significant 32-bit word first: the angle tables of rope_cos_sin.
void fill_rope_phi(uint32_t (*phi)[3], int D, double base);

// Stores the text rra_last_cuda_error() returns on this thread.
void record_cuda_error(cudaError_t e, const char* where);

cudaError_t launch_rope_append(const RopeArgs& a, rra_dtype dt, cudaStream_t stream);
// RoPE + append into an INT8 cache (bf16 q / k_new / v_new; a.k_scale etc. set).
cudaError_t launch_rope_append_q8(const RopeArgs& a, cudaStream_t stream);
// The same into an INT4 cache (head_dim 128, at most 32 KV heads).
cudaError_t launch_rope_append_q4(const RopeArgs& a, cudaStream_t stream);
// Tokens per stage of the tensor-core (bf16) decode kernel: K + V tiles of 32 KB.
inline int decode_mma_tile_tokens(int D) { return 16384 / (D * 2); }
// Most block-table entries one work item of the tensor-core kernel may span.
constexpr int kMmaTableEntries = 256;

// use_mma: the bf16 tensor-core kernel (tensor maps with the 128-byte swizzle); otherwise the
// CUDA-core kernel (contiguous: 1-D bulk copies, maps unused; paged: unswizzled maps).
cudaError_t launch_decode_contig(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                 rra_dtype dt, bool use_mma, cudaStream_t stream);
cudaError_t launch_decode_paged(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                rra_dtype dt, bool use_mma, cudaStream_t stream);
// The whole step in the tensor-core kernel (a.positions, a.k_new, a.v_new, a.q_out set).
cudaError_t launch_decode_step_contig(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                      cudaStream_t stream);
cudaError_t launch_decode_step_paged(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                     cudaStream_t stream);
// The tcgen05 decode kernel (bf16, head_dim 128, query groups of 16 to 128 heads: one CTA per
// (split, KV head, sequence) serving the whole group, key tiles of 128 tokens); the whole step
// when `fused` (a.positions, a.k_new, a.v_new, a.q_out set).
cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                             bool fused, cudaStream_t stream);
constexpr int kDecodeTcTile = 128;
// Tokens per stage of the narrow bf16 decode CTAs (head_dim 128).
constexpr int kDecodeNarrowTile = 32;

// Pipeline of the INT8 decode kernel: RRA_Q8_STAGES stages of RRA_Q8_STAGE_BYTES (K + V codes).
#ifndef RRA_Q8_STAGES
#define RRA_Q8_STAGES 4
#endif
#ifndef RRA_Q8_STAGE_BYTES
#define RRA_Q8_STAGE_BYTES 16384
#endif
// Resident CTAs per SM of the INT8 / INT4 decode kernel (its launch bounds and the split plan).
#ifndef RRA_Q8_CTAS_PER_SM
#define RRA_Q8_CTAS_PER_SM 3
#endif
// Speculative verify: attention of gamma new tokens per sequence (a.gamma, a.positions set).
// fused: the whole step (a.q unrotated; a.k_new, a.v_new, a.q_out, a.rope_style, a.rope_phi set;
// gamma <= 8).
cudaError_t launch_decode_verify(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                                 bool fused, cudaStream_t stream);
// Largest gamma of the one-launch verify step.
constexpr int kVerifyFusedMaxGammaHost = 8;
// Prefill: causal attention of the T = a.gamma prompt tokens of each sequence (a.positions: the
// first one's position); 64 query rows (a.hpc heads x 64 / a.hpc tokens) per CTA.
cudaError_t launch_prefill(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, bool paged,
                           cudaStream_t stream);
// Prefill on the tcgen05 tensor cores (head_dim 128): 128 prompt tokens of one query head per
// CTA; q_map covers q_rot as {D, Hq, B*T} with boxes of 64 dims x 1 head x 128 tokens.
cudaError_t launch_prefill_tc(const DecodeArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                              const CUtensorMap& v_map, bool paged, cudaStream_t stream);
// Tokens per stage of the INT8 (bits 8) / INT4 (bits 4) decode kernel.
inline int decode_q8_tile_tokens(int D, int bits = 8) { return RRA_Q8_STAGE_BYTES / 2 / (D * bits / 8); }
// INT8 caches: attention only (a.seq_lens) or the fused step (a.positions, a.k_new, ...).
// k_map / v_map cover the code caches, kw_map / vw_map the bf16 rings (unused without a window).
cudaError_t launch_decode_q8(const DecodeArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                             const CUtensorMap& kw_map, const CUtensorMap& vw_map, bool paged, bool fused,
                             cudaStream_t stream);

}  // namespace rra
