/*
 * rra.h — C ABI of the single-token RoPE + GQA decode-attention step (GB300, sm_103a).
 *
 * The step, per layer and per sequence b of a batch:
 *   1. rotate the new token's q [Hq, D] and k [Hkv, D] at its absolute position pos_b
 *      (RoPE, theta_i = base^(-2i/D), i = 0..D/2-1);
 *   2. write the rotated k and the unrotated v into cache slot pos_b;
 *   3. for every query head h: out[b,h] = softmax(q_rot[b,h] . K^T * scale) . V over
 *      the first L_b cached tokens of KV head h / n_rep (n_rep = Hq / Hkv).
 *
 * Sources (pages, by title and section):
 *   [KVC-GQA-RoPE] "Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践":
 *       §2.1 attention formula and decode shapes, §2.2 GQA / repeat_interleave,
 *       §3 RoPE, §4.1 cache layout and paging, §5.1 the per-layer decode order.
 *   [SelfAttn-Step] "4. 自注意力机制推理：单步计算、KV Cache的引入与原理":
 *       §4.3 KV cache, §4.5 preallocated cache written by index at slot `step`.
 *   [Opt-2026] "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南":
 *       §三 default scale 1/sqrt(d_k), §四 KVCache.update / PagedKVCache /
 *       cache-size formula, §六 GQA (n_q_heads must be a multiple of n_kv_heads).
 *
 * Conventions shared by every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or keeps them. Every tensor pointer must be 16-byte aligned.
 *   - Tensors are dense, row-major, with the element type `dt` (bf16 or fp32);
 *     positions, seq_lens and block tables are int32.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous on it; a return of RRA_OK means the work was enqueued.
 *   - Errors the host can see return a negative rra_status before anything is
 *     enqueued. Errors only the device can see (a position or length beyond the
 *     cache, a block id outside the pool, a pipeline wait that ran out) set bits of
 *     *err_flag (a device int32 the caller zeroes and reads back; may be NULL) and
 *     the affected work is skipped or clamped; no kernel traps.
 *   - Shapes: B = batch, Hq / Hkv = query / KV heads (Hq % Hkv == 0), D = head_dim
 *     (64 or 128). B == 0 is a no-op.
 */
#ifndef RRA_H
#define RRA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RRA_API __attribute__((visibility("default")))
#else
#define RRA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RRA_F32 = 0, RRA_BF16 = 1 } rra_dtype;

typedef enum {
  RRA_OK = 0,
  RRA_EINVAL = -1,        /* null pointer, bad shape, Hq % Hkv != 0, misaligned pointer */
  RRA_EUNSUPPORTED = -2,  /* D not in {64,128}, unknown dtype, block_size not a power of two */
  RRA_ERANGE = -3,        /* a size beyond what the kernels index (e.g. B > 65535) */
  RRA_EWORKSPACE = -4,    /* workspace missing or smaller than rra_decode_workspace_bytes() */
  RRA_ECUDA = -5          /* a CUDA runtime/driver call failed (see rra_last_cuda_error) */
} rra_status;

/* Bits the kernels OR into *err_flag. */
enum {
  RRA_ERR_POSITION = 1,   /* positions[b] < 0 or >= cache capacity: that sequence was not written */
  RRA_ERR_BLOCK_ID = 2,   /* a block-table entry outside [0, num_blocks): block 0 was used instead */
  RRA_ERR_SEQ_LEN = 4,    /* seq_lens[b] < 0 or > capacity: clamped into [0, capacity] */
  RRA_ERR_TIMEOUT = 8,    /* an in-kernel pipeline wait gave up (~1 s): results are invalid */
  RRA_ERR_WORKSPACE = 16  /* the workspace's split counters were not zero: results are invalid */
};

/* Steps 1-2: RoPE on q and k_new at positions[b], then append rotated k and raw v.
 *
 * [KVC-GQA-RoPE] §3 (frequencies base^(-2(i-1)/d), i = 1..d/2; the cache keeps
 * rotated K so only the new token is rotated), §5.1 b.ii-iii; [SelfAttn-Step] §4.5
 * (write slot `step`); [Opt-2026] §四 (KVCache.update; PagedKVCache block table).
 *
 *   q        [B, Hq, D]   input;  q_out [B, Hq, D] output (may alias q)
 *   k_new    [B, Hkv, D]  input, rotated before it is stored
 *   v_new    [B, Hkv, D]  input, stored unrotated
 *   positions[B] int32    absolute position of the new token = its cache slot
 *   Contiguous cache (block_table == NULL): k_cache, v_cache [B, Hkv, max_len, D];
 *     slot pos of (b, g) is row ((b*Hkv + g)*max_len + pos).
 *   Paged cache (block_table != NULL): k_cache, v_cache are pools
 *     [num_blocks, block_size, Hkv, D]; block_table [B, max_blocks_per_seq] int32 lists
 *     each sequence's physical blocks in logical order; token pos of sequence b lives
 *     in block block_table[b][pos / block_size] at slot pos % block_size. The caller
 *     must have allocated that block. block_size must be a power of two.
 *   rope_base  RoPE base (10000 for the pages' models; > 1)
 *   rope_style 0 = half-split pairs (i, i + D/2) ("rotate_half"), 1 = interleaved (2i, 2i+1)
 * theta_i is formed in float64; the angle pos * theta_i is taken exactly (theta_i / 2pi as a
 * 96-bit fraction, see rra_rope_phi), its sine and cosine to about 2^-44 as float32 hi + lo
 * pairs, the rotation with error-free float32 products, and the result is rounded once to dt
 * (nearest even). Hq + Hkv must not exceed 524280.
 */
RRA_API int rra_rope_append(const void* q, const void* k_new, const void* v_new,
                    const int32_t* positions, void* q_out,
                    void* k_cache, void* v_cache,
                    const int32_t* block_table, int max_blocks_per_seq,
                    int block_size, int num_blocks, int max_len,
                    int B, int Hq, int Hkv, int D, double rope_base, int rope_style,
                    rra_dtype dt, int32_t* err_flag, void* stream);

/* Step 3 on a contiguous cache [B, Hkv, max_len, D]:
 *   out[b,h,:] = softmax(q_rot[b,h,:] . K[b, h/n_rep, 0:L_b, :]^T * scale) . V[b, h/n_rep, 0:L_b, :]
 * [KVC-GQA-RoPE] §2.1, §2.2 (repeat_interleave: query head h reads KV head h / n_rep);
 * [SelfAttn-Step] §4.1, §4.5 (K_eff = K_cache[:, :, :step+1]); [Opt-2026] §三 (scale).
 *
 *   q_rot     [B, Hq, D]   rotated queries (rra_rope_append's q_out)
 *   seq_lens  [B] int32    L_b, attended tokens INCLUDING the new one (pos_b + 1);
 *                          L_b == 0 gives a zero output row
 *   out       [B, Hq, D]   written in dt (nearest even)
 *   scale     <= 0 selects 1/sqrt(D)
 *   num_splits  split-K chunks per sequence (flash-decoding); 0 = chosen by the library
 *               from the SM count, B, Hkv and the cache capacity. The effective count is
 *               rra_decode_num_splits(); with more than one split the partial results
 *               go to `workspace` and a second kernel merges them.
 *   workspace, ws_bytes  device scratch of at least rra_decode_workspace_bytes() bytes
 *               (may be NULL when that is 0). It must be zero-filled before its first use;
 *               every call leaves it ready for the next one (its split counters back at
 *               zero). Calls sharing a workspace must not overlap on the GPU.
 * Softmax runs online in float32 per split (running max, running sum, rescaled
 * accumulator); each split publishes its partial and the last split of a sequence to
 * finish merges them by log-sum-exp in the same kernel. The result equals the plain
 * two-pass softmax up to float32 rounding.
 */
RRA_API int rra_decode_attn_contig(const void* q_rot, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, void* out,
                           int B, int Hq, int Hkv, int D, int max_len, float scale,
                           int num_splits, void* workspace, size_t ws_bytes,
                           rra_dtype dt, int32_t* err_flag, void* stream);

/* Step 3 on a paged cache: pools [num_blocks, block_size, Hkv, D], block_table
 * [B, max_blocks_per_seq] int32 ([Opt-2026] §四 PagedKVCache.get_kv_for_attention:
 * the logical K/V is the table-ordered concatenation of the blocks, cut to L_b).
 * Only entries 0 .. ceil(L_b / block_size) - 1 of row b are read. Blocks may be
 * shared between sequences (prefix sharing); they are only read. Other arguments
 * as in rra_decode_attn_contig.
 */
RRA_API int rra_decode_attn_paged(const void* q_rot, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, int block_size, int num_blocks,
                          void* out, int B, int Hq, int Hkv, int D, float scale,
                          int num_splits, void* workspace, size_t ws_bytes,
                          rra_dtype dt, int32_t* err_flag, void* stream);

/* The whole step in one call: RoPE on q and k_new at positions[b], append of rotated k and
 * raw v at that slot, and the attention of every query head over the L_b = positions[b] + 1
 * tokens now in the cache ([KVC-GQA-RoPE] §5.1 b.ii-vi; [SelfAttn-Step] §4.5). For bf16
 * caches (paged blocks of at least 8 tokens, or contiguous caches of at least 64 tokens for
 * D = 128) it is a single kernel: the CTA whose chunk holds the new token writes it into
 * the cache before reading that tile, and every CTA rotates its own query heads; otherwise
 * it runs rra_rope_append and then the decode kernel.
 *   q        [B, Hq, D] unrotated queries; q_out [B, Hq, D] receives q_rot and must not
 *            overlap q.
 *   positions[B]: slot of the new token; positions outside the cache set RRA_ERR_POSITION and
 *            leave that sequence's outputs unwritten.
 * Other arguments as in rra_rope_append and rra_decode_attn_contig / rra_decode_attn_paged
 * (same workspace and split rules). */
RRA_API int rra_decode_step_contig(const void* q, const void* k_new, const void* v_new,
                                   const int32_t* positions, void* q_out, void* k_cache, void* v_cache,
                                   int max_len, void* out, int B, int Hq, int Hkv, int D,
                                   double rope_base, int rope_style, float scale, int num_splits,
                                   void* workspace, size_t ws_bytes, rra_dtype dt, int32_t* err_flag,
                                   void* stream);
RRA_API int rra_decode_step_paged(const void* q, const void* k_new, const void* v_new,
                                  const int32_t* positions, void* q_out, void* k_pool, void* v_pool,
                                  const int32_t* block_table, int max_blocks_per_seq, int block_size,
                                  int num_blocks, void* out, int B, int Hq, int Hkv, int D,
                                  double rope_base, int rope_style, float scale, int num_splits,
                                  void* workspace, size_t ws_bytes, rra_dtype dt, int32_t* err_flag,
                                  void* stream);

/* --- INT8 KV cache with per-head scales and a bf16 window of recent tokens ---
 *
 * [KVC-GQA-RoPE] §4.3: K and V cached as INT8 instead of BF16 (half the bytes), with
 * quantisation parameters calibrated per attention head, and the most recent tokens kept at
 * high precision. The page gives no formula; these calls implement:
 *   - codes: int8 c = clamp(round_half_even(x / s_g), -127, 127) for a value x of KV head g,
 *     the quotient an IEEE float32 division; the value is c * s_g. x is the rotated k rounded
 *     to bf16, or v. -128 is never written. k_scale, v_scale: float32 [Hkv] on the device,
 *     positive and finite (calibrated by the caller; not checked).
 *   - code caches: contiguous (block_table == NULL) k_codes, v_codes int8 [B, Hkv, max_len, D]
 *     (max_len at least 16384 / D tokens), or paged pools int8 [num_blocks, block_size, Hkv, D]
 *     (block_size a power of two >= 8) addressed through block_table as in the bf16 calls.
 *   - window W (0, or a multiple of 8 up to 65536): k_win, v_win bf16 [B, Hkv, W, D] rings;
 *     token t of sequence b lives in slot t % W. Every appended token is quantised into its
 *     cache slot AND, with W > 0, written in bf16 to its ring slot. Attention over L_b tokens
 *     reads tokens [0, L_b - W) from the codes and the last min(L_b, W) tokens from the ring.
 *     With W == 0 the rings are not used (may be NULL).
 *   - q, k_new, v_new, q_out, out are bf16; everything else as in the bf16 calls.
 */

/* rra_rope_append on an INT8 cache: RoPE on q and k_new at positions[b], then the quantised
 * rotated k and v into cache slot positions[b] and their bf16 values into ring slot
 * positions[b] % W. */
RRA_API int rra_rope_append_q8(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                               void* q_out, void* k_codes, void* v_codes, const float* k_scale,
                               const float* v_scale, void* k_win, void* v_win, int window,
                               const int32_t* block_table, int max_blocks_per_seq, int block_size,
                               int num_blocks, int max_len, int B, int Hq, int Hkv, int D, double rope_base,
                               int rope_style, int32_t* err_flag, void* stream);

/* Attention of q_rot over the L_b = seq_lens[b] tokens of the mixed-precision cache (codes
 * times scales, then the window's bf16 tokens), split-K as rra_decode_attn_paged. The INT8
 * tokens are cut into splits (num_splits, 0 = chosen by the library); the split holding the
 * last INT8 tokens also reads the ring. The workspace must hold rra_decode_workspace_bytes(B,
 * Hq, D, rra_decode_q8_num_splits(...)) bytes, with the same zero-fill rule. */
RRA_API int rra_decode_attn_q8(const void* q_rot, const void* k_codes, const void* v_codes, const float* k_scale,
                               const float* v_scale, const void* k_win, const void* v_win, int window,
                               const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                               int block_size, int num_blocks, int max_len, void* out, int B, int Hq, int Hkv,
                               int D, float scale, int num_splits, void* workspace, size_t ws_bytes,
                               int32_t* err_flag, void* stream);

/* The whole step on an INT8 cache in one kernel: RoPE on q and k_new at positions[b], the
 * quantised append (and ring write) of the new token, and the attention over L_b =
 * positions[b] + 1 tokens. q_out receives q_rot and must not overlap q. */
RRA_API int rra_decode_step_q8(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                               void* q_out, void* k_codes, void* v_codes, const float* k_scale,
                               const float* v_scale, void* k_win, void* v_win, int window,
                               const int32_t* block_table, int max_blocks_per_seq, int block_size,
                               int num_blocks, int max_len, void* out, int B, int Hq, int Hkv, int D,
                               double rope_base, int rope_style, float scale, int num_splits, void* workspace,
                               size_t ws_bytes, int32_t* err_flag, void* stream);

/* Effective INT8 split count of rra_decode_attn_q8 / rra_decode_step_q8: the `splits`
 * argument of rra_decode_workspace_bytes. max_tokens and block_size as in
 * rra_decode_num_splits. Negative rra_status on bad arguments. */
RRA_API int rra_decode_q8_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size,
                                     int num_splits, int window);

/* INT4 codes ([KVC-GQA-RoPE] §4.3: INT8 or INT4): the same four calls with 4-bit codes
 * clamp(round_half_even(x / s_g), -7, 7) (float32 quotient; -8 never written), two per byte:
 * dims 2j and 2j+1 in byte j, the even one in the low nibble, as 4-bit two's complement. The
 * code caches hold D / 2 bytes per token and head ([B, Hkv, max_len, D/2] or pools
 * [num_blocks, block_size, Hkv, D/2]); head_dim 128 only; rra_rope_append_q4 takes at most 32
 * KV heads. Contiguous caches need at least 128 tokens. Everything else as for INT8. */
RRA_API int rra_rope_append_q4(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                               void* q_out, void* k_codes, void* v_codes, const float* k_scale,
                               const float* v_scale, void* k_win, void* v_win, int window,
                               const int32_t* block_table, int max_blocks_per_seq, int block_size,
                               int num_blocks, int max_len, int B, int Hq, int Hkv, int D, double rope_base,
                               int rope_style, int32_t* err_flag, void* stream);
RRA_API int rra_decode_attn_q4(const void* q_rot, const void* k_codes, const void* v_codes, const float* k_scale,
                               const float* v_scale, const void* k_win, const void* v_win, int window,
                               const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                               int block_size, int num_blocks, int max_len, void* out, int B, int Hq, int Hkv,
                               int D, float scale, int num_splits, void* workspace, size_t ws_bytes,
                               int32_t* err_flag, void* stream);
RRA_API int rra_decode_step_q4(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                               void* q_out, void* k_codes, void* v_codes, const float* k_scale,
                               const float* v_scale, void* k_win, void* v_win, int window,
                               const int32_t* block_table, int max_blocks_per_seq, int block_size,
                               int num_blocks, int max_len, void* out, int B, int Hq, int Hkv, int D,
                               double rope_base, int rope_style, float scale, int num_splits, void* workspace,
                               size_t ws_bytes, int32_t* err_flag, void* stream);
RRA_API int rra_decode_q4_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size,
                                     int num_splits, int window);

/* --- Multi-query decode: the speculative-verify step ---
 *
 * [Opt-2026] §五: the target model checks gamma draft tokens (gamma = 4 on the page) in one pass.
 * Sequence b gets gamma new tokens at positions p_b .. p_b + gamma - 1 (positions[b] = p_b);
 * each is rotated at its own position and appended at that slot, and query token j attends
 * tokens [0, p_b + j] -- the cached ones and the new ones up to itself -- exactly what
 * decoding the tokens one at a time gives. q, k_new, v_new, q_out and out are laid out
 * [B, gamma, H, D]; caches, block tables and the other arguments as in the decode calls
 * (contiguous when block_table is NULL; paged blocks of at least 8 tokens, contiguous caches of
 * at least 16384 / (2 D) tokens; bf16 only for the attention). gamma is 1..16.
 */

/* rra_rope_append for gamma new tokens per sequence (token j at positions[b] + j). With
 * gamma == 1 it is rra_rope_append; bf16 or fp32. */
RRA_API int rra_rope_append_verify(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                                   void* q_out, void* k_cache, void* v_cache, const int32_t* block_table,
                                   int max_blocks_per_seq, int block_size, int num_blocks, int max_len, int B,
                                   int gamma, int Hq, int Hkv, int D, double rope_base, int rope_style, rra_dtype dt,
                                   int32_t* err_flag, void* stream);

/* out[b, j, h] = softmax(q_rot[b, j, h] . K[b, h / n_rep, 0 : p_b + j + 1]^T * scale) . V[...] for
 * bf16 caches that already hold the new tokens. One CTA serves up to 16 query rows (heads x new
 * tokens) of a KV head, so each K/V byte read serves all of them; split-K with the same merge
 * as the decode calls. The workspace must hold rra_verify_workspace_bytes(B, gamma, Hq, Hkv, D,
 * rra_verify_num_splits(...)) bytes, zero-filled before its first use (left zeroed by every
 * call). Positions with p_b + gamma beyond the cache set RRA_ERR_POSITION and skip b. */
RRA_API int rra_verify_attn(const void* q_rot, const void* k_cache, const void* v_cache, const int32_t* block_table,
                            int max_blocks_per_seq, const int32_t* positions, int block_size, int num_blocks,
                            int max_len, void* out, int B, int gamma, int Hq, int Hkv, int D, float scale,
                            int num_splits, void* workspace, size_t ws_bytes, int32_t* err_flag, void* stream);

/* The whole verify step: RoPE of the gamma new tokens' q and k at positions p_b .. p_b + gamma - 1,
 * their append, and the attention of rra_verify_attn, with q_rot also written to q_out. Up to
 * gamma 8 this is ONE kernel: each CTA rotates its query rows in registers (sines and cosines
 * of the gamma positions as in rra_rope_append, once per CTA), and the CTAs whose chunk holds new tokens
 * write them into the cache before their own TMA reads the tile that holds them. Above gamma 8
 * it runs rra_rope_append_verify then rra_verify_attn on q_out (two kernels). Same results
 * either way. bf16. q_out must not overlap q. ("Transformer架构优化实战2026：注意力机制、KV
 * Cache与推理加速完整指南" §五; RoPE as in rra_rope_append.) */
RRA_API int rra_verify_step(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                            void* q_out, void* k_cache, void* v_cache, const int32_t* block_table,
                            int max_blocks_per_seq, int block_size, int num_blocks, int max_len, void* out, int B,
                            int gamma, int Hq, int Hkv, int D, double rope_base, int rope_style, float scale,
                            int num_splits, void* workspace, size_t ws_bytes, int32_t* err_flag, void* stream);

/* Effective split count of rra_verify_attn (max_tokens and block_size as in
 * rra_decode_num_splits); negative rra_status on bad arguments. */
RRA_API int rra_verify_num_splits(int B, int gamma, int Hq, int Hkv, int D, int64_t max_tokens, int block_size,
                                  int num_splits);

/* Workspace bytes of rra_verify_attn for an effective split count; 0 when splits <= 1. */
RRA_API size_t rra_verify_workspace_bytes(int B, int gamma, int Hq, int Hkv, int D, int splits);

/* --- Prefill: causal attention of a whole prompt (or a chunk of one after a cached prefix) ---
 *
 * [Opt-2026] §三 (FlashAttention: softmax(Q K^T / sqrt(d)) V by blocks with a running max and
 * sum, never materialising the T x T scores). The T prompt tokens of sequence b sit at
 * positions p_b .. p_b + T - 1 (positions[b] = p_b; p_b = 0 for a fresh prompt), and token t
 * attends tokens [0, p_b + t]: the definition of the verify calls with gamma = T.
 * rra_rope_append_verify(..., gamma = T, ...) rotates and appends them; then: */

/* out[b, t, h] = softmax(q_rot[b, t, h] . K[b, h / n_rep, 0 : p_b + t + 1]^T * scale) . V[...],
 * bf16, q_rot and out [B, T, Hq, D], caches as in the decode calls (paged blocks of at least 8
 * tokens, contiguous caches of at least 16384 / (2 D) tokens). No workspace. Head dim 128 runs
 * on the tcgen05 tensor cores (128 prompt tokens of one or two query heads per CTA, one CTA per
 * SM, scores and outputs in Tensor Memory; q_rot and out 16-byte aligned, as checked); head dim
 * 64 on mma.sync (64 query rows per CTA). RRA_ERANGE when (T / 64 + 1) * Hq exceeds 2^31 - 1
 * (the CTA count of one sequence). A prompt that runs past the cache sets RRA_ERR_POSITION
 * and skips b; a pipeline wait that runs out sets RRA_ERR_TIMEOUT. */
RRA_API int rra_prefill_attn(const void* q_rot, const void* k_cache, const void* v_cache, const int32_t* block_table,
                             int max_blocks_per_seq, const int32_t* positions, int block_size, int num_blocks,
                             int max_len, void* out, int B, int T, int Hq, int Hkv, int D, float scale,
                             int32_t* err_flag, void* stream);

/* rra_rope_append_verify with gamma = T, then rra_prefill_attn on q_out. bf16. q_out must not
 * overlap q. */
RRA_API int rra_prefill_step(const void* q, const void* k_new, const void* v_new, const int32_t* positions,
                             void* q_out, void* k_cache, void* v_cache, const int32_t* block_table,
                             int max_blocks_per_seq, int block_size, int num_blocks, int max_len, void* out, int B,
                             int T, int Hq, int Hkv, int D, double rope_base, int rope_style, float scale,
                             int32_t* err_flag, void* stream);

/* Bytes of a K+V cache: 2 * n_layers * n_kv_heads * head_dim * seq_len * batch * dtype_bytes
 * ([Opt-2026] §四 memory formula; [KVC-GQA-RoPE] §5.3). Host only; returns 0 when an
 * argument is negative or the product overflows 64 bits. */
RRA_API uint64_t rra_kv_bytes(int n_layers, int n_kv_heads, int head_dim, int64_t seq_len,
                      int batch, int dtype_bytes);

/* --- Helpers (host only; no counterpart on the pages) --- */

/* Effective split count the decode entry points use for these arguments
 * (max_tokens = max_len for contiguous, max_blocks_per_seq * block_size for paged;
 * block_size = 0 for contiguous). Negative rra_status on bad arguments. Queries the
 * current device's SM count when num_splits == 0. */
RRA_API int rra_decode_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size,
                          int num_splits, rra_dtype dt);

/* Workspace bytes for B sequences, Hq heads, head_dim D and an EFFECTIVE split count
 * (from rra_decode_num_splits); 0 when splits <= 1. */
RRA_API size_t rra_decode_workspace_bytes(int B, int Hq, int D, int splits);

/* Static text for an rra_status value. */
RRA_API const char* rra_status_str(int status);

/* Text of the last CUDA error an entry point saw on this thread ("" if none). */
RRA_API const char* rra_last_cuda_error(void);

/* Test hook for the bounded-wait timeout path (no counterpart on the pages). While `hold` is
 * nonzero, the fused bf16 steps (rra_decode_step_*, rra_verify_step up to gamma 8) launched
 * from any thread write the new tokens but never release the barrier their TMA producer waits
 * on before loading the tile that holds them: that wait, and the consumers' wait for the tile,
 * run out after about a second each, the kernel sets RRA_ERR_TIMEOUT and finishes (its outputs
 * are invalid), and the context stays usable. Nothing faults, traps or hangs. 0 restores normal
 * operation. Always returns RRA_OK. */
RRA_API int rra_test_hold_append(int hold);

/* The library links its own copy of the CUDA runtime, whose current device is separate
 * from the caller's: every entry point launches on the device selected here for the
 * calling thread (device 0 until set), and `stream` must belong to that device. */
RRA_API int rra_use_device(int device);

/* --- RoPE angle tables (no counterpart on the pages: how every kernel here forms the sine and
 *     cosine of m * theta_i, [KVC-GQA-RoPE] §3, exposed so that tests can check it) ---
 * The kernels carry theta_i / 2pi (theta_i = rope_base^(-2i/head_dim), i < head_dim/2, formed in
 * float64) as a 96-bit binary fraction phi_i, take m * phi_i mod 1 in integer arithmetic and
 * evaluate cos and sin of that many turns in float32 as hi + lo pairs (absolute error below
 * about 2^-44). */

/* phi_i for i < head_dim/2 into phi[3 * i + w], w = 0 the least significant 32-bit word. Host
 * only. RRA_EINVAL for a null phi, an odd head_dim or one outside [2, 512], or a rope_base that is
 * not positive and finite. */
RRA_API int rra_rope_phi(int head_dim, double rope_base, uint32_t* phi);

/* cos and sin of 2pi * (position * phi mod 1) for one phi (3 words as above) on the host, by the
 * same float32 operations as the kernels: out[0] + out[1] = cos, out[2] + out[3] = sin. RRA_EINVAL
 * for a null pointer or a negative position. */
RRA_API int rra_rope_cos_sin_host(int position, const uint32_t* phi, float* out);

/* The same on the device for positions[p] (device int32, p < n) and every i < head_dim/2: out
 * (device float32 [n, 4, head_dim/2]) holds the rows cos hi, cos lo, sin hi, sin lo; NaN for a
 * negative position. Asynchronous on `stream`. RRA_EINVAL or RRA_ERANGE on bad arguments,
 * RRA_ECUDA if the launch fails. */
RRA_API int rra_rope_cos_sin(const int32_t* positions, int n, int head_dim, double rope_base, float* out,
                             void* stream);

/* --- Decode without a caller workspace (the pages have no counterpart: this exists for
 *     callers that must not allocate device memory when they run a step) ---
 *
 * rra_decode_attn_paged_noalloc is rra_decode_attn_paged with the split-K scratch taken
 * from a fixed array inside the library instead of a caller workspace. It is meant for
 * callers that cannot call cudaMalloc when they decode: code with no allocator of its own
 * because a host framework owns all device memory, and loops that forbid allocation after
 * start-up because allocating can block, fail or fragment memory mid-run. It allocates
 * nothing and calls no allocating routine.
 *   - The array holds rra_noalloc_scratch_bytes() (16 MiB) on every GPU that loads the
 *     library, kept until the process exits: its first 1 MiB holds the split merge's
 *     arrival counters (at the same place for every shape), the other 15 MiB the split
 *     partials. A step whose effective split count needs more than that (for instance
 *     rra_decode_workspace_bytes above 15 MiB) returns RRA_EWORKSPACE before anything is
 *     enqueued; ask for fewer splits then.
 *   - The counters must be zero when the kernel starts: every call clears the ones it
 *     uses with a cudaMemsetAsync on `stream` before its launch (this allocates nothing),
 *     so each call is independent of what earlier calls, of any shape, left in the array.
 *   - All calls on a device share the array: calls whose kernels overlap on the GPU race
 *     and give wrong results. Keep them on one stream or serialise them.
 *   - The first call on each device (with that device current) looks up the array's
 *     device address; make that first call before any stream capture starts.
 * Arguments as in rra_decode_attn_paged, without workspace and ws_bytes. */
RRA_API int rra_decode_attn_paged_noalloc(const void* q_rot, const void* k_pool, const void* v_pool,
                                          const int32_t* block_table, int max_blocks_per_seq,
                                          const int32_t* seq_lens, int block_size, int num_blocks,
                                          void* out, int B, int Hq, int Hkv, int D, float scale,
                                          int num_splits, rra_dtype dt, int32_t* err_flag, void* stream);

/* Bytes of the fixed scratch array rra_decode_attn_paged_noalloc uses (16 MiB). */
RRA_API size_t rra_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* RRA_H */
