// The extern "C" entry points declared in include/rra.h: argument checks, split
// planning, tensor-map encoding for the paged pools, and kernel dispatch.
// Nothing here allocates device memory; every buffer belongs to the caller.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "rra_internal.h"

namespace {

thread_local char g_cuda_error[256] = "";
// rra_test_hold_append: while set, fused bf16 steps launched from any thread hold their append
// barrier (a test of the bounded waits' timeout path).
std::atomic<int> g_test_hold_append{0};

int cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return RRA_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
int elem_bytes(rra_dtype dt) { return dt == RRA_BF16 ? 2 : 4; }

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// How the decode work is cut: kernel, query heads per CTA, token chunk per split, split count.
struct Plan {
  int ctas_per_sm = 0;  // resident CTAs per SM of the kernel (0: 3 for the tensor-core kernels, else 2)
  bool mma = false;  // bf16 tensor-core kernel
  bool tc = false;   // bf16 tcgen05 kernel for query groups of 16..128 heads (head_dim 128)
  bool narrow = false;  // bf16 mma.sync kernel with 2 consumer warps, 32-token stages, 4 CTAs per SM
  int hpc = 1;
  int tile = 0;
  int chunk = 0;
  int splits = 1;
  int max_chunk_tokens = 2048;  // longest chunk the many-sequence plan gives one CTA
};

// The tensor-core kernel takes bf16 with TMA destinations on 1024-byte swizzle atoms:
// contiguous caches at least one tile long, paged blocks of at least 8 tokens.
bool use_mma_kernel(rra_dtype dt, int D, int64_t max_tokens, int block_size) {
  if (dt != RRA_BF16) return false;
  if (block_size > 0) return block_size >= 8;
  return max_tokens >= rra::decode_mma_tile_tokens(D);
}

int heads_per_cta(int n_rep, bool mma) {
  if (mma) {
    if (n_rep <= 8) return n_rep;
    for (int h = 8; h > 1; --h)
      if (n_rep % h == 0) return h;
    return 1;
  }
  return n_rep % 4 == 0 ? 4 : (n_rep % 2 == 0 ? 2 : 1);
}

// The bf16 decode kernel: 16 query heads per CTA (two 8-head n-tiles, two CTAs per SM) for query
// groups of a multiple of 16 heads, so each K/V tile serves 16 of them; otherwise up to 8.
int decode_mma_hpc(int n_rep) { return n_rep % 16 == 0 ? 16 : heads_per_cta(n_rep, true); }

int check_shapes(int B, int Hq, int Hkv, int D, rra_dtype dt) {
  if (dt != RRA_F32 && dt != RRA_BF16) return RRA_EUNSUPPORTED;
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return RRA_EINVAL;
  if (D != 64 && D != 128) return RRA_EUNSUPPORTED;
  if (B > 65535) return RRA_ERANGE;
  return RRA_OK;
}

// Chunk and split count for a per-sequence capacity of max_tokens, once p->mma, p->hpc and
// p->tile are set.
// extra_units: CTAs per (sequence, head slice) beyond the splits (the INT8 kernel's ring unit).
// short_splits: with few sequences x heads, chunks may go below 256 tokens (down to one tile) so
// that a short capacity still gets this many splits.
int plan_splits(int B, int Hkv, int n_rep, int64_t max_tokens, int block_size, int requested, Plan* p,
                int extra_units = 0, int short_splits = 0) {
  const int64_t tiles = std::max<int64_t>(1, (max_tokens + p->tile - 1) / p->tile);
  // A paged split copies its block ids to shared memory: at most kMaxTableEntries of them.
  int64_t max_chunk_tiles = tiles;
  if (block_size > 0) {
    const int entries = p->mma ? rra::kMmaTableEntries : rra::kMaxTableEntries;
    max_chunk_tiles = std::max<int64_t>(1, (int64_t(entries - 1) * block_size) / p->tile);
  }
  int64_t chunk_tiles;
  if (requested > 0) {
    chunk_tiles = (tiles + requested - 1) / requested;
  } else {
    // CTAs that fit on the GPU at once: 3 per SM for the mma kernel, 2 otherwise.
    const int64_t resident = (p->ctas_per_sm ? p->ctas_per_sm : (p->mma ? 3 : 2)) * int64_t(std::max(1, sm_count()));
    const int64_t units = std::max<int64_t>(1, int64_t(B) * Hkv * (n_rep / p->hpc));  // CTAs per split
    if (2 * units <= resident) {
      // Few sequences x heads: as many splits as fit in ONE wave (a second wave that is barely
      // started costs a whole CTA time), each at least 256 tokens long.
      const int64_t splits_one_wave = std::max<int64_t>(1, resident / units - extra_units);
      chunk_tiles = (tiles + splits_one_wave - 1) / splits_one_wave;
      int64_t min_tiles = std::max(1, 256 / p->tile);
      if (short_splits > 0) min_tiles = std::min<int64_t>(min_tiles, (tiles + short_splits - 1) / short_splits);
      chunk_tiles = std::max<int64_t>(chunk_tiles, std::max<int64_t>(1, min_tiles));
    } else {
      // Many sequences x heads: about two waves, each CTA streaming 128..2048 tokens; fewer,
      // longer CTAs pay start-up and epilogue less often, two waves keep ragged tails short.
      const int64_t target = 2 * resident;
      chunk_tiles = (tiles * units + target - 1) / target;
      const int64_t lo = std::max(1, 128 / p->tile), hi = std::max(1, p->max_chunk_tokens / p->tile);
      chunk_tiles = std::min(std::max(chunk_tiles, lo), hi);
    }
  }
  chunk_tiles = std::min(std::max<int64_t>(chunk_tiles, 1), max_chunk_tiles);
  chunk_tiles = std::max<int64_t>(chunk_tiles, (tiles + rra::kMaxSplits - 1) / rra::kMaxSplits);
  if (chunk_tiles > max_chunk_tiles) return RRA_ERANGE;
  const int64_t splits = (tiles + chunk_tiles - 1) / chunk_tiles;
  if (splits * (n_rep / p->hpc) > int64_t(INT32_MAX) / 2) return RRA_ERANGE;
  p->chunk = static_cast<int>(chunk_tiles * p->tile);
  p->splits = static_cast<int>(splits);
  return RRA_OK;
}

// Smallest query group (heads per KV head) the bf16 decode at head_dim 128 runs on the tcgen05
// kernel (one CTA per group) instead of the mma.sync kernel (16 heads per CTA, the group in
// slices). Measured on one KV head, 16 sequences of 8192 tokens: 128 heads 64.6 us (tcgen05)
// against 101.6 us; 64 heads 46.1 against 44.8 us; 32 heads 37.2 against 32.6 us; 16 heads 33.7
// against 31.4 us.
#ifndef RRA_TC_MIN_NREP
#define RRA_TC_MIN_NREP 96
#endif

// max_tokens: per-sequence capacity; block_size: 0 for a contiguous cache.
int make_plan(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int requested, rra_dtype dt,
              Plan* p) {
  int st = check_shapes(B, Hq, Hkv, D, dt);
  if (st != RRA_OK) return st;
  if (requested < 0 || max_tokens < 0) return RRA_EINVAL;
  if (max_tokens > (int64_t(1) << 30)) return RRA_ERANGE;
  const int n_rep = Hq / Hkv;
  p->mma = use_mma_kernel(dt, D, max_tokens, block_size);
  if (p->mma && D == 128 && n_rep >= RRA_TC_MIN_NREP && n_rep <= 128 &&
      (block_size > 0 || max_tokens >= rra::kDecodeTcTile)) {
    // one CTA per (split, KV head, sequence) serving the whole query group on the tcgen05 cores
    p->tc = true;
    p->hpc = n_rep;
    p->ctas_per_sm = 1;
    p->tile = rra::kDecodeTcTile;
    return plan_splits(B, Hkv, n_rep, max_tokens, block_size, requested, p);
  }
  p->hpc = p->mma ? decode_mma_hpc(n_rep) : heads_per_cta(n_rep, false);
  if (p->hpc > 8) p->ctas_per_sm = 2;
  if (static_cast<int64_t>(Hkv) * (n_rep / p->hpc) > 65535) return RRA_ERANGE;
  p->tile = p->mma ? rra::decode_mma_tile_tokens(D) : rra::decode_tile_tokens(D, elem_bytes(dt));
  // bf16 tensor-core decode: at least 8 splits for short capacities (one sequence, 32q/8kv, 1K
  // tokens: 11.4 us at 8 splits of 128 tokens against 12.8 us at 4 of 256; at 4K the 256-token
  // floor stays, 13.8 us at 16 splits against 14.7 us at 32)
  st = plan_splits(B, Hkv, n_rep, max_tokens, block_size, requested, p, 0, p->mma ? 8 : 0);
  if (st != RRA_OK || !p->mma || D != 128 || p->hpc > 8 || requested == 0) return st;
  // A requested split count that takes few (sequence, KV head) units past one wave of the
  // 3-per-SM kernel: narrow CTAs, four per SM, so the grid needs fewer and fuller waves.
  const int64_t resident = 3 * int64_t(std::max(1, sm_count()));
  const int64_t units = int64_t(B) * Hkv * (n_rep / p->hpc);
  if (2 * units > resident || units * p->splits <= resident) return st;
  Plan q = *p;
  q.narrow = true;
  q.ctas_per_sm = 4;
  q.tile = rra::kDecodeNarrowTile;
  if (plan_splits(B, Hkv, n_rep, max_tokens, block_size, requested, &q) == RRA_OK) *p = q;
  return st;
}

// INT8 caches: the INT8 tokens split like the bf16 tensor-core kernel's (tiles of
// decode_q8_tile_tokens(D) tokens); the window's ring is streamed by the CTA of the last split,
// so it adds no split. Paged blocks must hold at least 8 tokens and a contiguous cache at least
// one tile; the window is a multiple of 8.
int make_plan_q8(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int requested, int window,
                 Plan* p, int bits = 8) {
  int st = check_shapes(B, Hq, Hkv, D, RRA_BF16);
  if (st != RRA_OK) return st;
  if (bits == 4 && D != 128) return RRA_EUNSUPPORTED;  // INT4 tiles: 64-byte rows
  if (requested < 0 || max_tokens < 0 || window < 0) return RRA_EINVAL;
  if (max_tokens > (int64_t(1) << 30)) return RRA_ERANGE;
  if (window % 8 != 0 || window > 65536) return RRA_EUNSUPPORTED;
  const int n_rep = Hq / Hkv;
  p->mma = true;
  p->hpc = heads_per_cta(n_rep, true);
  if (static_cast<int64_t>(Hkv) * (n_rep / p->hpc) > 65535) return RRA_ERANGE;
  p->tile = rra::decode_q8_tile_tokens(D, bits);
  p->ctas_per_sm = RRA_Q8_CTAS_PER_SM;
  // INT4 CTAs stream half an INT8 CTA's bytes per token for the same start-up and merge costs
  // (per-CTA traces: ~7 us before the first tile and ~4 us merging around ~19 us of streaming), so
  // the many-sequence plan gives them chunks of up to 3072 tokens: the batch-64 INT4 step 108.5 /
  // 109.0 us at 3 splits against 112.4 / 112.6 us at 4; INT8 keeps 2048 (127.4 us at 4 splits
  // against 130.4 us at 3).
  if (bits == 4) p->max_chunk_tokens = 3072;
  if (block_size > 0 ? block_size < 8 : max_tokens < p->tile) return RRA_EUNSUPPORTED;
  return plan_splits(B, Hkv, n_rep, max_tokens, block_size, requested, p);
}

// Speculative verify: one CTA serves hpc heads x gamma new tokens (at most 16 query rows) of one
// KV head; hpc is the largest divisor of n_rep with hpc * gamma <= 16. Three CTAs per SM.
int verify_hpc(int n_rep, int gamma) {
  for (int h = std::min(n_rep, 16 / gamma); h > 1; --h)
    if (n_rep % h == 0) return h;
  return 1;
}

int make_plan_verify(int B, int gamma, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int requested,
                     Plan* p) {
  int st = check_shapes(B, Hq, Hkv, D, RRA_BF16);
  if (st != RRA_OK) return st;
  if (requested < 0 || max_tokens < 0 || gamma < 1) return RRA_EINVAL;
  if (gamma > 16) return RRA_EUNSUPPORTED;
  if (max_tokens > (int64_t(1) << 30) || int64_t(B) * gamma > (int64_t(1) << 24)) return RRA_ERANGE;
  const int n_rep = Hq / Hkv;
  p->mma = true;
  p->hpc = verify_hpc(n_rep, gamma);
  if (static_cast<int64_t>(Hkv) * (n_rep / p->hpc) > 65535) return RRA_ERANGE;
  p->tile = rra::decode_mma_tile_tokens(D);
  if (block_size > 0 ? block_size < 8 : max_tokens < p->tile) return RRA_EUNSUPPORTED;
  return plan_splits(B, Hkv, n_rep, max_tokens, block_size, requested, p);
}

// Prefill: 64 query rows per CTA, hpc heads x 64 / hpc prompt tokens; hpc divides n_rep and 64.
int prefill_hpc(int n_rep) {
  for (int h = std::min(n_rep, 64); h > 1; --h)
    if (n_rep % h == 0 && 64 % h == 0) return h;
  return 1;
}

// Limits of a prefill launch, checked before anything is enqueued: a capacity of at most 2^30
// tokens, head groups within the grid's second dimension, and the CTAs of one sequence (query
// blocks of at least 64 / hpc prompt tokens x head groups, or 128 tokens x pairs of heads) within
// its first: at most (T / 64 + 1) * Hq.
int check_prefill_limits(int T, int Hq, int Hkv, int64_t capacity) {
  if (capacity > (int64_t(1) << 30)) return RRA_ERANGE;
  const int n_rep = Hq / Hkv;
  if (int64_t(Hkv) * (n_rep / prefill_hpc(n_rep)) > 65535) return RRA_ERANGE;
  if ((int64_t(T) / 64 + 1) * Hq > int64_t(INT32_MAX)) return RRA_ERANGE;
  return RRA_OK;
}

// KV groups per prefill scheduling band: as many as have their prompt's K and V (T x D x 2 x
// 2 bytes each, bf16) within 64 MB, half of the L2, and divide Hkv; at least one.
int prefill_kv_band(int T, int Hkv, int D) {
  const int64_t per_group = int64_t(T) * D * 4;
  int g = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(Hkv, (int64_t(64) << 20) / per_group)));
  while (Hkv % g != 0) --g;
  return g;
}

// Partial rows of the verify kernel: 16 per (sequence, KV head, head slice).
int64_t verify_rows(int B, int gamma, int Hq, int Hkv) {
  return int64_t(B) * Hkv * ((Hq / Hkv) / verify_hpc(Hq / Hkv, gamma)) * 16;
}

// Workspace layout, each part 256-byte aligned (R = B*Hq, G = merge_groups(splits)):
// partials o [R, splits, D] and (max, sum) [R, splits, 2] floats, level-2 partials o [R, G, D]
// and (max, sum) [R, G, 2] floats, counters [R] and group counters [R, G] int32.
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t o, ml, o2, ml2, cnt, gcnt, total;
};

WsLayout ws_layout(int B, int Hq, int D, int splits) {
  const size_t R = size_t(B) * Hq, G = size_t(rra::merge_groups(splits));
  WsLayout l{};
  l.o = 0;
  l.ml = l.o + align256(R * splits * D * sizeof(float));
  l.o2 = l.ml + align256(R * splits * 2 * sizeof(float));
  l.ml2 = l.o2 + align256(R * G * D * sizeof(float));
  l.cnt = l.ml2 + align256(R * G * 2 * sizeof(float));
  l.gcnt = l.cnt + align256(R * sizeof(int));
  l.total = l.gcnt + R * G * sizeof(int);
  return l;
}

size_t workspace_bytes(int B, int Hq, int D, int splits) {
  if (splits <= 1 || B <= 0) return 0;
  return ws_layout(B, Hq, D, splits).total;
}

// The partial arrays alone (everything before the counters), and the counters alone in int32s.
size_t partial_bytes(int B, int Hq, int D, int splits) {
  if (splits <= 1 || B <= 0) return 0;
  return ws_layout(B, Hq, D, splits).cnt;
}

size_t counter_ints(int B, int Hq, int splits) {
  if (splits <= 1 || B <= 0) return 0;
  const size_t R = size_t(B) * Hq, G = size_t(rra::merge_groups(splits));
  return R + R * G;
}

// Tiled tensor map over `base` (rank 3 or 4, dims innermost first, strides in bytes of dims 1..).
int encode_map_typed(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box, CUtensorMapDataType type, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled unavailable");
    return RRA_ECUDA;
  }
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(map, type, rank, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
    return RRA_ECUDA;
  }
  return RRA_OK;
}

int encode_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box, rra_dtype dt, bool swizzle128) {
  return encode_map_typed(map, base, rank, dims, strides, box,
                          dt == RRA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// INT8 code caches: rows of D bytes with the 128-byte (D = 128) or 64-byte (D = 64) swizzle.
// Paged pools [num_blocks, block_size, Hkv, D] as {D, Hkv, block_size, num_blocks} with boxes of
// one head's `box_rows` rows; contiguous caches [B, Hkv, max_len, D] as {D, max_len, B*Hkv}.
// RB: bytes of codes per token and head (D for INT8, D / 2 for INT4): 128 or 64.
int encode_q8_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int Hkv, int RB,
                       int box_rows) {
  const cuuint64_t dims[4] = {cuuint64_t(RB), cuuint64_t(Hkv), cuuint64_t(block_size), cuuint64_t(num_blocks)};
  const cuuint64_t strides[3] = {cuuint64_t(RB), cuuint64_t(Hkv) * RB, cuuint64_t(block_size) * Hkv * RB};
  const cuuint32_t box[4] = {cuuint32_t(RB), 1u, cuuint32_t(box_rows), 1u};
  return encode_map_typed(map, pool, 4, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                          RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

int encode_q8_contig_map(CUtensorMap* map, const void* cache, int B, int Hkv, int max_len, int RB, int tile) {
  const cuuint64_t dims[3] = {cuuint64_t(RB), cuuint64_t(max_len), cuuint64_t(B) * Hkv};
  const cuuint64_t strides[2] = {cuuint64_t(RB), cuuint64_t(max_len) * RB};
  const cuuint32_t box[3] = {cuuint32_t(RB), cuuint32_t(tile), 1u};
  return encode_map_typed(map, cache, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                          RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// Pool [num_blocks, block_size, Hkv, D] as 4-D {D, Hkv, block_size, num_blocks}; the box is
// one head's rows of one block (64-dim halves with the 128-byte swizzle for the mma kernel).
int encode_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int Hkv, int D, int box_rows,
                    rra_dtype dt, bool mma) {
  const cuuint64_t es = elem_bytes(dt);
  const cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(block_size), cuuint64_t(num_blocks)};
  const cuuint64_t strides[3] = {D * es, cuuint64_t(Hkv) * D * es, cuuint64_t(block_size) * Hkv * D * es};
  const cuuint32_t box[4] = {cuuint32_t(mma ? 64 : D), 1u, cuuint32_t(box_rows), 1u};
  return encode_map(map, pool, 4, dims, strides, box, dt, mma);
}

// Contiguous cache [B, Hkv, max_len, D] as 3-D {D, max_len, B*Hkv}, boxes of 64 dims x tile rows.
int encode_contig_map(CUtensorMap* map, const void* cache, int B, int Hkv, int max_len, int D, int tile,
                      rra_dtype dt) {
  const cuuint64_t es = elem_bytes(dt);
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(max_len), cuuint64_t(B) * Hkv};
  const cuuint64_t strides[2] = {D * es, cuuint64_t(max_len) * D * es};
  const cuuint32_t box[3] = {64u, cuuint32_t(tile), 1u};
  return encode_map(map, cache, 3, dims, strides, box, dt, true);
}

int check_workspace(const Plan& p, int B, int Hq, int D, const void* ws, size_t ws_bytes) {
  const size_t need = workspace_bytes(B, Hq, D, p.splits);
  if (need == 0) return RRA_OK;
  if (ws == nullptr || ws_bytes < need || !aligned16(ws)) return RRA_EWORKSPACE;
  return RRA_OK;
}

// counters: when set, the arrival counters live there ([B*Hq] counters, then [B*Hq, G] group
// counters) instead of inside `ws`, which then holds only the partial arrays.
rra::DecodeArgs decode_args(const Plan& p, const void* q, const void* k, const void* v, const int32_t* seq_lens,
                            void* out, int B, int Hq, int Hkv, int D, float scale, void* ws, int32_t* err,
                            int* counters = nullptr) {
  rra::DecodeArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.seq_lens = seq_lens;
  a.out = out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.hpc = p.hpc;
  a.num_splits = p.splits;
  a.chunk = p.chunk;
  const float s = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  a.scale_log2 = s * 1.4426950408889634f;
  a.err = err;
  a.num_groups = rra::merge_groups(p.splits);
  a.narrow = p.narrow ? 1 : 0;
  a.test_hold_append = g_test_hold_append.load(std::memory_order_relaxed);
  if (p.splits > 1) {
    const WsLayout l = ws_layout(B, Hq, D, p.splits);
    uint8_t* base = static_cast<uint8_t*>(ws);
    a.ws_o = reinterpret_cast<float*>(base + l.o);
    a.ws_ml = reinterpret_cast<float*>(base + l.ml);
    a.ws2_o = reinterpret_cast<float*>(base + l.o2);
    a.ws2_ml = reinterpret_cast<float*>(base + l.ml2);
    a.counters = reinterpret_cast<int*>(base + l.cnt);
    a.group_counters = reinterpret_cast<int*>(base + l.gcnt);
    if (counters != nullptr) {
      a.counters = counters;
      a.group_counters = counters + size_t(B) * Hq;
    }
  }
  return a;
}

int finish_decode(cudaError_t e) { return e == cudaSuccess ? RRA_OK : cuda_fail(e, "decode kernel launch"); }

bool overlap(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

// Checks shared by the two fused-step entry points (everything but the cache layout).
int check_step_args(const void* q, const void* k_new, const void* v_new, const int32_t* positions, const void* q_out,
                    const void* k_cache, const void* v_cache, const void* out, int B, int Hq, int D, double rope_base,
                    int rope_style, float scale, rra_dtype dt) {
  if (!(rope_base > 1.0) || !std::isfinite(rope_base) || (rope_style != 0 && rope_style != 1)) return RRA_EINVAL;
  if (!std::isfinite(scale)) return RRA_EINVAL;
  if (B == 0) return RRA_OK;
  if (!q || !k_new || !v_new || !positions || !q_out || !k_cache || !v_cache || !out) return RRA_EINVAL;
  for (const void* p : {q, k_new, v_new, q_out, k_cache, v_cache, out})
    if (!aligned16(p)) return RRA_EINVAL;
  if (overlap(q, q_out, size_t(B) * Hq * D * elem_bytes(dt))) return RRA_EINVAL;  // q is read after q_out is written
  return RRA_OK;
}

// Checks and tensor maps shared by the INT8 entry points. Contiguous (block_table == NULL):
// codes [B, Hkv, max_len, D]; paged: pools [num_blocks, block_size, Hkv, D].
struct Q8Layout {
  int64_t capacity = 0;
  int log2_bs = 0;
};

int q8_layout(const int32_t* block_table, int max_blocks_per_seq, int block_size, int num_blocks, int max_len,
              Q8Layout* l) {
  if (block_table != nullptr) {
    if (!pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
    if (max_blocks_per_seq < 1 || num_blocks < 1) return RRA_EINVAL;
    l->capacity = int64_t(max_blocks_per_seq) * block_size;
    l->log2_bs = ilog2(block_size);
  } else {
    if (max_len < 1) return RRA_EINVAL;
    l->capacity = max_len;
  }
  return RRA_OK;
}

int check_q8_buffers(const void* k_codes, const void* v_codes, const float* k_scale, const float* v_scale,
                     const void* k_win, const void* v_win, int window) {
  if (!k_codes || !v_codes || !k_scale || !v_scale) return RRA_EINVAL;
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale)) return RRA_EINVAL;
  if (window > 0 && (!k_win || !v_win || !aligned16(k_win) || !aligned16(v_win))) return RRA_EINVAL;
  return RRA_OK;
}

int q8_maps(const Plan& p, const void* k_codes, const void* v_codes, const void* k_win, const void* v_win, int window,
            const int32_t* block_table, int block_size, int num_blocks, int max_len, int B, int Hkv, int D,
            CUtensorMap* km, CUtensorMap* vm, CUtensorMap* kwm, CUtensorMap* vwm, int bits = 8) {
  int st;
  const int RB = D * bits / 8;
  if (block_table != nullptr) {
    const int box_rows = block_size < p.tile ? block_size : p.tile;
    st = encode_q8_pool_map(km, k_codes, num_blocks, block_size, Hkv, RB, box_rows);
    if (st == RRA_OK) st = encode_q8_pool_map(vm, v_codes, num_blocks, block_size, Hkv, RB, box_rows);
  } else {
    st = encode_q8_contig_map(km, k_codes, B, Hkv, max_len, RB, p.tile);
    if (st == RRA_OK) st = encode_q8_contig_map(vm, v_codes, B, Hkv, max_len, RB, p.tile);
  }
  if (st != RRA_OK || window == 0) return st;
  const int rows = std::min(window, RRA_Q8_STAGE_BYTES / (4 * D));  // ring rows per stage (K + V bf16)
  st = encode_contig_map(kwm, k_win, B, Hkv, window, D, rows, RRA_BF16);
  if (st == RRA_OK) st = encode_contig_map(vwm, v_win, B, Hkv, window, D, rows, RRA_BF16);
  return st;
}

void set_q8_args(rra::DecodeArgs* a, const Q8Layout& l, const void* k_codes, const void* v_codes, const float* k_scale,
                 const float* v_scale, void* k_win, void* v_win, int window, const int32_t* block_table,
                 int max_blocks_per_seq, int num_blocks, int max_len) {
  a->k = k_codes;
  a->v = v_codes;
  a->k_scale = k_scale;
  a->v_scale = v_scale;
  a->k_win = k_win;
  a->v_win = v_win;
  a->window = window;
  a->block_table = block_table;
  a->max_blocks_per_seq = max_blocks_per_seq;
  a->log2_bs = l.log2_bs;
  a->num_blocks = num_blocks;
  a->max_len = block_table != nullptr ? 0 : max_len;
  a->capacity = static_cast<int>(l.capacity);
}

}  // namespace

namespace rra {
void record_cuda_error(cudaError_t e, const char* where) { cuda_fail(e, where); }
}  // namespace rra

static int decode_qk_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int num_splits,
                                int window, int bits) {
  if (block_size < 0 || (block_size > 0 && !pow2(block_size))) return block_size < 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  Plan p;
  const int st = make_plan_q8(B, Hq, Hkv, D, max_tokens, block_size, num_splits, window, &p, bits);
  return st != RRA_OK ? st : p.splits;
}

static int rope_append_qk(int bits, const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                       void* k_codes, void* v_codes, const float* k_scale, const float* v_scale, void* k_win,
                       void* v_win, int window, const int32_t* block_table, int max_blocks_per_seq, int block_size,
                       int num_blocks, int max_len, int B, int Hq, int Hkv, int D, double rope_base, int rope_style,
                       int32_t* err_flag, void* stream) {
  int st = check_shapes(B, Hq, Hkv, D, RRA_BF16);
  if (st != RRA_OK) return st;
  if (!(rope_base > 1.0) || !std::isfinite(rope_base) || (rope_style != 0 && rope_style != 1)) return RRA_EINVAL;
  if (window < 0) return RRA_EINVAL;
  if (bits == 4 && (D != 128 || Hkv > 32)) return RRA_EUNSUPPORTED;
  if (window > 0 && (window % 8 != 0 || window > 65536)) return RRA_EUNSUPPORTED;
  if (int64_t(Hq) + Hkv > 8 * 65535) return RRA_ERANGE;
  Q8Layout l;
  st = q8_layout(block_table, max_blocks_per_seq, block_size, num_blocks, max_len, &l);
  if (st != RRA_OK) return st;
  if (l.capacity > (int64_t(1) << 30)) return RRA_ERANGE;
  if (B == 0) return RRA_OK;
  if (!q || !k_new || !v_new || !positions || !q_out) return RRA_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_out)) return RRA_EINVAL;
  st = check_q8_buffers(k_codes, v_codes, k_scale, v_scale, k_win, v_win, window);
  if (st != RRA_OK) return st;
  rra::RopeArgs a{};
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.positions = positions;
  a.q_out = q_out;
  a.k_cache = k_codes;
  a.v_cache = v_codes;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.log2_bs = l.log2_bs;
  a.num_blocks = num_blocks;
  a.max_len = max_len;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.rope_style = rope_style;
  a.err = err_flag;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.k_win = k_win;
  a.v_win = v_win;
  a.window = window;
  rra::fill_rope_phi(a.rope_phi, D, rope_base);
  const cudaError_t e = bits == 4 ? rra::launch_rope_append_q4(a, static_cast<cudaStream_t>(stream))
                                  : rra::launch_rope_append_q8(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RRA_OK : cuda_fail(e, "rope_append (quantised) launch");
}

static int decode_attn_qk(int bits, const void* q_rot, const void* k_codes, const void* v_codes, const float* k_scale,
                       const float* v_scale, const void* k_win, const void* v_win, int window,
                       const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens, int block_size,
                       int num_blocks, int max_len, void* out, int B, int Hq, int Hkv, int D, float scale,
                       int num_splits, void* workspace, size_t ws_bytes, int32_t* err_flag, void* stream) {
  Q8Layout l;
  int st = q8_layout(block_table, max_blocks_per_seq, block_size, num_blocks, max_len, &l);
  if (st != RRA_OK) return st;
  Plan p;
  st = make_plan_q8(B, Hq, Hkv, D, l.capacity, block_table ? block_size : 0, num_splits, window, &p, bits);
  if (st != RRA_OK) return st;
  if (!std::isfinite(scale)) return RRA_EINVAL;
  if (B == 0) return RRA_OK;
  if (!q_rot || !seq_lens || !out || !aligned16(q_rot) || !aligned16(out)) return RRA_EINVAL;
  st = check_q8_buffers(k_codes, v_codes, k_scale, v_scale, k_win, v_win, window);
  if (st != RRA_OK) return st;
  st = check_workspace(p, B, Hq, D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  CUtensorMap km{}, vm{}, kwm{}, vwm{};
  st = q8_maps(p, k_codes, v_codes, k_win, v_win, window, block_table, block_size, num_blocks, max_len, B, Hkv, D,
               &km, &vm, &kwm, &vwm, bits);
  if (st != RRA_OK) return st;
  rra::DecodeArgs a = decode_args(p, q_rot, k_codes, v_codes, seq_lens, out, B, Hq, Hkv, D, scale, workspace, err_flag);
  set_q8_args(&a, l, k_codes, v_codes, k_scale, v_scale, const_cast<void*>(k_win), const_cast<void*>(v_win), window,
              block_table, max_blocks_per_seq, num_blocks, max_len);
  a.code_bits = bits;
  return finish_decode(rra::launch_decode_q8(a, km, vm, kwm, vwm, block_table != nullptr, false,
                                             static_cast<cudaStream_t>(stream)));
}

static int decode_step_qk(int bits, const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                       void* k_codes, void* v_codes, const float* k_scale, const float* v_scale, void* k_win,
                       void* v_win, int window, const int32_t* block_table, int max_blocks_per_seq, int block_size,
                       int num_blocks, int max_len, void* out, int B, int Hq, int Hkv, int D, double rope_base,
                       int rope_style, float scale, int num_splits, void* workspace, size_t ws_bytes,
                       int32_t* err_flag, void* stream) {
  Q8Layout l;
  int st = q8_layout(block_table, max_blocks_per_seq, block_size, num_blocks, max_len, &l);
  if (st != RRA_OK) return st;
  Plan p;
  st = make_plan_q8(B, Hq, Hkv, D, l.capacity, block_table ? block_size : 0, num_splits, window, &p, bits);
  if (st != RRA_OK) return st;
  st = check_step_args(q, k_new, v_new, positions, q_out, k_codes, v_codes, out, B, Hq, D, rope_base, rope_style,
                       scale, RRA_BF16);
  if (st != RRA_OK || B == 0) return st;
  st = check_q8_buffers(k_codes, v_codes, k_scale, v_scale, k_win, v_win, window);
  if (st != RRA_OK) return st;
  st = check_workspace(p, B, Hq, D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  CUtensorMap km{}, vm{}, kwm{}, vwm{};
  st = q8_maps(p, k_codes, v_codes, k_win, v_win, window, block_table, block_size, num_blocks, max_len, B, Hkv, D,
               &km, &vm, &kwm, &vwm, bits);
  if (st != RRA_OK) return st;
  rra::DecodeArgs a = decode_args(p, q, k_codes, v_codes, nullptr, out, B, Hq, Hkv, D, scale, workspace, err_flag);
  set_q8_args(&a, l, k_codes, v_codes, k_scale, v_scale, k_win, v_win, window, block_table, max_blocks_per_seq,
              num_blocks, max_len);
  a.code_bits = bits;
  a.positions = positions;
  a.k_new = k_new;
  a.v_new = v_new;
  a.q_out = q_out;
  a.rope_style = rope_style;
  rra::fill_rope_phi(a.rope_phi, D, rope_base);
  return finish_decode(rra::launch_decode_q8(a, km, vm, kwm, vwm, block_table != nullptr, true,
                                             static_cast<cudaStream_t>(stream)));
}


namespace {

// The fused verify step's extra inputs (rra_verify_step with gamma <= 8).
struct VerifyFusedArgs {
  const void* k_new;
  const void* v_new;
  void* q_out;
  int rope_style;
  double rope_base;
};

// rra_verify_attn, or with `fused` the whole verify step in one launch.
int verify_launch(const void* q_rot, const void* k_cache, const void* v_cache, const int32_t* block_table,
                  int max_blocks_per_seq, const int32_t* positions, int block_size, int num_blocks, int max_len,
                  void* out, int B, int gamma, int Hq, int Hkv, int D, float scale, int num_splits, void* workspace,
                  size_t ws_bytes, int32_t* err_flag, void* stream, const VerifyFusedArgs* fused) {
  int64_t capacity;
  if (block_table != nullptr) {
    if (!pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
    if (max_blocks_per_seq < 1 || num_blocks < 1) return RRA_EINVAL;
    capacity = int64_t(max_blocks_per_seq) * block_size;
  } else {
    if (max_len < 1) return RRA_EINVAL;
    capacity = max_len;
  }
  Plan p;
  int st = make_plan_verify(B, gamma, Hq, Hkv, D, capacity, block_table ? block_size : 0, num_splits, &p);
  if (st != RRA_OK) return st;
  if (!std::isfinite(scale)) return RRA_EINVAL;
  if (B == 0) return RRA_OK;
  if (!q_rot || !k_cache || !v_cache || !positions || !out) return RRA_EINVAL;
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return RRA_EINVAL;
  const int64_t rows = verify_rows(B, gamma, Hq, Hkv);
  if (rows > INT32_MAX) return RRA_ERANGE;
  st = check_workspace(p, 1, static_cast<int>(rows), D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  CUtensorMap km{}, vm{};
  if (block_table != nullptr) {
    const int box_rows = block_size < p.tile ? block_size : p.tile;
    st = encode_pool_map(&km, k_cache, num_blocks, block_size, Hkv, D, box_rows, RRA_BF16, true);
    if (st == RRA_OK) st = encode_pool_map(&vm, v_cache, num_blocks, block_size, Hkv, D, box_rows, RRA_BF16, true);
  } else {
    st = encode_contig_map(&km, k_cache, B, Hkv, max_len, D, p.tile, RRA_BF16);
    if (st == RRA_OK) st = encode_contig_map(&vm, v_cache, B, Hkv, max_len, D, p.tile, RRA_BF16);
  }
  if (st != RRA_OK) return st;
  // the workspace holds `rows` partial rows: laid out as for one sequence of `rows` heads
  rra::DecodeArgs a = decode_args(p, q_rot, k_cache, v_cache, nullptr, out, 1, static_cast<int>(rows), 1, D, scale,
                                  workspace, err_flag);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.gamma = gamma;
  a.positions = positions;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.log2_bs = block_table ? ilog2(block_size) : 0;
  a.num_blocks = num_blocks;
  a.max_len = block_table ? 0 : max_len;
  a.capacity = static_cast<int>(capacity);
  if (fused != nullptr) {  // q_rot is the unrotated q: the kernel rotates it and appends the new tokens
    a.k_new = fused->k_new;
    a.v_new = fused->v_new;
    a.q_out = fused->q_out;
    a.rope_style = fused->rope_style;
    rra::fill_rope_phi(a.rope_phi, D, fused->rope_base);
  }
  return finish_decode(
      rra::launch_decode_verify(a, km, vm, block_table != nullptr, fused != nullptr, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char* rra_status_str(int status) {
  switch (status) {
    case RRA_OK: return "ok";
    case RRA_EINVAL: return "invalid argument";
    case RRA_EUNSUPPORTED: return "unsupported configuration";
    case RRA_ERANGE: return "size out of range";
    case RRA_EWORKSPACE: return "workspace missing or too small";
    case RRA_ECUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* rra_last_cuda_error(void) { return g_cuda_error; }

int rra_test_hold_append(int hold) {
  g_test_hold_append.store(hold != 0 ? 1 : 0, std::memory_order_relaxed);
  return RRA_OK;
}

int rra_use_device(int device) {
  const cudaError_t e = cudaSetDevice(device);
  return e == cudaSuccess ? RRA_OK : cuda_fail(e, "cudaSetDevice");
}

uint64_t rra_kv_bytes(int n_layers, int n_kv_heads, int head_dim, int64_t seq_len, int batch, int dtype_bytes) {
  if (n_layers < 0 || n_kv_heads < 0 || head_dim < 0 || seq_len < 0 || batch < 0 || dtype_bytes < 0) return 0;
  const uint64_t f[6] = {2u, uint64_t(n_layers), uint64_t(n_kv_heads), uint64_t(head_dim), uint64_t(batch),
                         uint64_t(dtype_bytes)};
  uint64_t r = uint64_t(seq_len);
  for (uint64_t x : f) {
    if (x != 0 && r > UINT64_MAX / x) return 0;
    r *= x;
  }
  return r;
}

int rra_decode_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int num_splits,
                          rra_dtype dt) {
  if (block_size < 0 || (block_size > 0 && !pow2(block_size))) return block_size < 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  Plan p;
  const int st = make_plan(B, Hq, Hkv, D, max_tokens, block_size, num_splits, dt, &p);
  return st != RRA_OK ? st : p.splits;
}

size_t rra_decode_workspace_bytes(int B, int Hq, int D, int splits) { return workspace_bytes(B, Hq, D, splits); }

int rra_rope_append(const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                    void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks_per_seq, int block_size,
                    int num_blocks, int max_len, int B, int Hq, int Hkv, int D, double rope_base, int rope_style,
                    rra_dtype dt, int32_t* err_flag, void* stream) {
  return rra_rope_append_verify(q, k_new, v_new, positions, q_out, k_cache, v_cache, block_table, max_blocks_per_seq,
                                block_size, num_blocks, max_len, B, 1, Hq, Hkv, D, rope_base, rope_style, dt, err_flag,
                                stream);
}

int rra_rope_append_verify(const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                           void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks_per_seq,
                           int block_size, int num_blocks, int max_len, int B, int gamma, int Hq, int Hkv, int D,
                           double rope_base, int rope_style, rra_dtype dt, int32_t* err_flag, void* stream) {
  int st = check_shapes(B, Hq, Hkv, D, dt);
  if (st != RRA_OK) return st;
  if (gamma < 1) return RRA_EINVAL;
  if (int64_t(B) * gamma > 2147483647LL) return RRA_ERANGE;
  if (!(rope_base > 1.0) || !std::isfinite(rope_base) || (rope_style != 0 && rope_style != 1)) return RRA_EINVAL;
  if (int64_t(Hq) + Hkv > 8 * 65535) return RRA_ERANGE;
  if (B == 0) return RRA_OK;
  if (!q || !k_new || !v_new || !positions || !q_out || !k_cache || !v_cache) return RRA_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_out) || !aligned16(k_cache) ||
      !aligned16(v_cache))
    return RRA_EINVAL;
  rra::RopeArgs a{};
  if (block_table != nullptr) {
    if (!pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
    if (max_blocks_per_seq < 1 || num_blocks < 1) return RRA_EINVAL;
    if (int64_t(max_blocks_per_seq) * block_size > (int64_t(1) << 30)) return RRA_ERANGE;
    a.log2_bs = ilog2(block_size);
  } else if (max_len < 1) {
    return RRA_EINVAL;
  }
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.positions = positions;
  a.q_out = q_out;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.max_len = max_len;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.gamma = gamma;
  rra::fill_rope_phi(a.rope_phi, D, rope_base);
  a.rope_style = rope_style;
  a.err = err_flag;
  const cudaError_t e = rra::launch_rope_append(a, dt, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RRA_OK : cuda_fail(e, "rope_append launch");
}

int rra_decode_attn_contig(const void* q_rot, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                           void* out, int B, int Hq, int Hkv, int D, int max_len, float scale, int num_splits,
                           void* workspace, size_t ws_bytes, rra_dtype dt, int32_t* err_flag, void* stream) {
  if (max_len < 1) return RRA_EINVAL;
  Plan p;
  int st = make_plan(B, Hq, Hkv, D, max_len, 0, num_splits, dt, &p);
  if (st != RRA_OK) return st;
  if (B == 0) return RRA_OK;
  if (!q_rot || !k_cache || !v_cache || !seq_lens || !out) return RRA_EINVAL;
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return RRA_EINVAL;
  if (!std::isfinite(scale)) return RRA_EINVAL;
  st = check_workspace(p, B, Hq, D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  CUtensorMap km{}, vm{};
  if (p.mma) {
    st = encode_contig_map(&km, k_cache, B, Hkv, max_len, D, p.tile, dt);
    if (st != RRA_OK) return st;
    st = encode_contig_map(&vm, v_cache, B, Hkv, max_len, D, p.tile, dt);
    if (st != RRA_OK) return st;
  }
  rra::DecodeArgs a = decode_args(p, q_rot, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, D, scale, workspace, err_flag);
  a.max_len = max_len;
  a.capacity = max_len;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.tc) return finish_decode(rra::launch_decode_tc(a, km, vm, false, false, s));
  return finish_decode(rra::launch_decode_contig(a, km, vm, dt, p.mma, s));
}

int rra_decode_attn_paged(const void* q_rot, const void* k_pool, const void* v_pool, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* seq_lens, int block_size, int num_blocks, void* out,
                          int B, int Hq, int Hkv, int D, float scale, int num_splits, void* workspace,
                          size_t ws_bytes, rra_dtype dt, int32_t* err_flag, void* stream) {
  return rra::decode_attn_paged_ext(q_rot, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, block_size,
                                    num_blocks, out, B, Hq, Hkv, D, scale, num_splits, workspace, ws_bytes, nullptr,
                                    dt, err_flag, stream);
}

}  // extern "C"

namespace rra {

size_t decode_partial_bytes(int B, int Hq, int D, int splits) { return partial_bytes(B, Hq, D, splits); }
size_t decode_counter_ints(int B, int Hq, int splits) { return counter_ints(B, Hq, splits); }

int decode_attn_paged_ext(const void* q_rot, const void* k_pool, const void* v_pool, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* seq_lens, int block_size, int num_blocks, void* out,
                          int B, int Hq, int Hkv, int D, float scale, int num_splits, void* workspace,
                          size_t ws_bytes, int* counters, rra_dtype dt, int32_t* err_flag, void* stream) {
  if (!pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  if (max_blocks_per_seq < 1 || num_blocks < 1) return RRA_EINVAL;
  const int64_t capacity = int64_t(max_blocks_per_seq) * block_size;
  Plan p;
  int st = make_plan(B, Hq, Hkv, D, capacity, block_size, num_splits, dt, &p);
  if (st != RRA_OK) return st;
  if (B == 0) return RRA_OK;
  if (!q_rot || !k_pool || !v_pool || !block_table || !seq_lens || !out) return RRA_EINVAL;
  if (!aligned16(q_rot) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return RRA_EINVAL;
  if (!std::isfinite(scale)) return RRA_EINVAL;
  if (counters == nullptr) {
    st = check_workspace(p, B, Hq, D, workspace, ws_bytes);
  } else if (p.splits > 1 &&
             (workspace == nullptr || !aligned16(workspace) || ws_bytes < partial_bytes(B, Hq, D, p.splits))) {
    st = RRA_EWORKSPACE;
  }
  if (st != RRA_OK) return st;
  const int box_rows = block_size < p.tile ? block_size : p.tile;
  CUtensorMap km, vm;
  st = encode_pool_map(&km, k_pool, num_blocks, block_size, Hkv, D, box_rows, dt, p.mma);
  if (st != RRA_OK) return st;
  st = encode_pool_map(&vm, v_pool, num_blocks, block_size, Hkv, D, box_rows, dt, p.mma);
  if (st != RRA_OK) return st;
  rra::DecodeArgs a =
      decode_args(p, q_rot, k_pool, v_pool, seq_lens, out, B, Hq, Hkv, D, scale, workspace, err_flag, counters);
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.log2_bs = ilog2(block_size);
  a.num_blocks = num_blocks;
  a.max_len = 0;
  a.capacity = static_cast<int>(capacity);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.tc) return finish_decode(rra::launch_decode_tc(a, km, vm, true, false, s));
  return finish_decode(rra::launch_decode_paged(a, km, vm, dt, p.mma, s));
}

}  // namespace rra

extern "C" {

int rra_decode_step_contig(const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                           void* k_cache, void* v_cache, int max_len, void* out, int B, int Hq, int Hkv, int D,
                           double rope_base, int rope_style, float scale, int num_splits, void* workspace,
                           size_t ws_bytes, rra_dtype dt, int32_t* err_flag, void* stream) {
  if (max_len < 1) return RRA_EINVAL;
  Plan p;
  int st = make_plan(B, Hq, Hkv, D, max_len, 0, num_splits, dt, &p);
  if (st != RRA_OK) return st;
  st = check_step_args(q, k_new, v_new, positions, q_out, k_cache, v_cache, out, B, Hq, D, rope_base, rope_style,
                       scale, dt);
  if (st != RRA_OK || B == 0) return st;
  st = check_workspace(p, B, Hq, D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap km{}, vm{};
  if (p.mma) {
    st = encode_contig_map(&km, k_cache, B, Hkv, max_len, D, p.tile, dt);
    if (st != RRA_OK) return st;
    st = encode_contig_map(&vm, v_cache, B, Hkv, max_len, D, p.tile, dt);
    if (st != RRA_OK) return st;
  } else {  // two kernels: RoPE + append, then the decode with L_b = positions[b] + 1
    st = rra_rope_append(q, k_new, v_new, positions, q_out, k_cache, v_cache, nullptr, 0, 0, 0, max_len, B, Hq, Hkv,
                         D, rope_base, rope_style, dt, err_flag, stream);
    if (st != RRA_OK) return st;
  }
  rra::DecodeArgs a =
      decode_args(p, p.mma ? q : q_out, k_cache, v_cache, nullptr, out, B, Hq, Hkv, D, scale, workspace, err_flag);
  a.max_len = max_len;
  a.capacity = max_len;
  a.positions = positions;
  if (!p.mma) return finish_decode(rra::launch_decode_contig(a, km, vm, dt, false, s));
  a.k_new = k_new;
  a.v_new = v_new;
  a.q_out = q_out;
  a.rope_style = rope_style;
  rra::fill_rope_phi(a.rope_phi, D, rope_base);
  if (p.tc) return finish_decode(rra::launch_decode_tc(a, km, vm, false, true, s));
  return finish_decode(rra::launch_decode_step_contig(a, km, vm, s));
}

int rra_decode_step_paged(const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                          void* k_pool, void* v_pool, const int32_t* block_table, int max_blocks_per_seq,
                          int block_size, int num_blocks, void* out, int B, int Hq, int Hkv, int D, double rope_base,
                          int rope_style, float scale, int num_splits, void* workspace, size_t ws_bytes, rra_dtype dt,
                          int32_t* err_flag, void* stream) {
  if (!pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  if (max_blocks_per_seq < 1 || num_blocks < 1) return RRA_EINVAL;
  const int64_t capacity = int64_t(max_blocks_per_seq) * block_size;
  Plan p;
  int st = make_plan(B, Hq, Hkv, D, capacity, block_size, num_splits, dt, &p);
  if (st != RRA_OK) return st;
  st = check_step_args(q, k_new, v_new, positions, q_out, k_pool, v_pool, out, B, Hq, D, rope_base, rope_style, scale,
                       dt);
  if (st != RRA_OK || B == 0) return st;
  if (!block_table) return RRA_EINVAL;
  st = check_workspace(p, B, Hq, D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int box_rows = block_size < p.tile ? block_size : p.tile;
  CUtensorMap km, vm;
  st = encode_pool_map(&km, k_pool, num_blocks, block_size, Hkv, D, box_rows, dt, p.mma);
  if (st != RRA_OK) return st;
  st = encode_pool_map(&vm, v_pool, num_blocks, block_size, Hkv, D, box_rows, dt, p.mma);
  if (st != RRA_OK) return st;
  if (!p.mma) {  // two kernels: RoPE + append, then the decode with L_b = positions[b] + 1
    st = rra_rope_append(q, k_new, v_new, positions, q_out, k_pool, v_pool, block_table, max_blocks_per_seq,
                         block_size, num_blocks, 0, B, Hq, Hkv, D, rope_base, rope_style, dt, err_flag, stream);
    if (st != RRA_OK) return st;
  }
  rra::DecodeArgs a =
      decode_args(p, p.mma ? q : q_out, k_pool, v_pool, nullptr, out, B, Hq, Hkv, D, scale, workspace, err_flag);
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.log2_bs = ilog2(block_size);
  a.num_blocks = num_blocks;
  a.max_len = 0;
  a.capacity = static_cast<int>(capacity);
  a.positions = positions;
  if (!p.mma) return finish_decode(rra::launch_decode_paged(a, km, vm, dt, false, s));
  a.k_new = k_new;
  a.v_new = v_new;
  a.q_out = q_out;
  a.rope_style = rope_style;
  rra::fill_rope_phi(a.rope_phi, D, rope_base);
  if (p.tc) return finish_decode(rra::launch_decode_tc(a, km, vm, true, true, s));
  return finish_decode(rra::launch_decode_step_paged(a, km, vm, s));
}

int rra_decode_q8_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int num_splits,
                             int window) {
  return decode_qk_num_splits(B, Hq, Hkv, D, max_tokens, block_size, num_splits, window, 8);
}

int rra_decode_q4_num_splits(int B, int Hq, int Hkv, int D, int64_t max_tokens, int block_size, int num_splits,
                             int window) {
  return decode_qk_num_splits(B, Hq, Hkv, D, max_tokens, block_size, num_splits, window, 4);
}

#define RRA_APPEND_ARGS                                                                                             \
  const void *q, const void *k_new, const void *v_new, const int32_t *positions, void *q_out, void *k_codes,         \
      void *v_codes, const float *k_scale, const float *v_scale, void *k_win, void *v_win, int window,               \
      const int32_t *block_table, int max_blocks_per_seq, int block_size, int num_blocks, int max_len, int B, int Hq, \
      int Hkv, int D, double rope_base, int rope_style, int32_t *err_flag, void *stream
#define RRA_APPEND_PASS                                                                                               \
  q, k_new, v_new, positions, q_out, k_codes, v_codes, k_scale, v_scale, k_win, v_win, window, block_table,            \
      max_blocks_per_seq, block_size, num_blocks, max_len, B, Hq, Hkv, D, rope_base, rope_style, err_flag, stream
int rra_rope_append_q8(RRA_APPEND_ARGS) { return rope_append_qk(8, RRA_APPEND_PASS); }
int rra_rope_append_q4(RRA_APPEND_ARGS) { return rope_append_qk(4, RRA_APPEND_PASS); }

#define RRA_ATTN_ARGS                                                                                                 \
  const void *q_rot, const void *k_codes, const void *v_codes, const float *k_scale, const float *v_scale,            \
      const void *k_win, const void *v_win, int window, const int32_t *block_table, int max_blocks_per_seq,           \
      const int32_t *seq_lens, int block_size, int num_blocks, int max_len, void *out, int B, int Hq, int Hkv, int D, \
      float scale, int num_splits, void *workspace, size_t ws_bytes, int32_t *err_flag, void *stream
#define RRA_ATTN_PASS                                                                                                 \
  q_rot, k_codes, v_codes, k_scale, v_scale, k_win, v_win, window, block_table, max_blocks_per_seq, seq_lens,          \
      block_size, num_blocks, max_len, out, B, Hq, Hkv, D, scale, num_splits, workspace, ws_bytes, err_flag, stream
int rra_decode_attn_q8(RRA_ATTN_ARGS) { return decode_attn_qk(8, RRA_ATTN_PASS); }
int rra_decode_attn_q4(RRA_ATTN_ARGS) { return decode_attn_qk(4, RRA_ATTN_PASS); }

#define RRA_STEP_ARGS                                                                                                 \
  const void *q, const void *k_new, const void *v_new, const int32_t *positions, void *q_out, void *k_codes,         \
      void *v_codes, const float *k_scale, const float *v_scale, void *k_win, void *v_win, int window,               \
      const int32_t *block_table, int max_blocks_per_seq, int block_size, int num_blocks, int max_len, void *out,     \
      int B, int Hq, int Hkv, int D, double rope_base, int rope_style, float scale, int num_splits, void *workspace,  \
      size_t ws_bytes, int32_t *err_flag, void *stream
#define RRA_STEP_PASS                                                                                                 \
  q, k_new, v_new, positions, q_out, k_codes, v_codes, k_scale, v_scale, k_win, v_win, window, block_table,            \
      max_blocks_per_seq, block_size, num_blocks, max_len, out, B, Hq, Hkv, D, rope_base, rope_style, scale,          \
      num_splits, workspace, ws_bytes, err_flag, stream
int rra_decode_step_q8(RRA_STEP_ARGS) { return decode_step_qk(8, RRA_STEP_PASS); }
int rra_decode_step_q4(RRA_STEP_ARGS) { return decode_step_qk(4, RRA_STEP_PASS); }

int rra_verify_num_splits(int B, int gamma, int Hq, int Hkv, int D, int64_t max_tokens, int block_size,
                          int num_splits) {
  if (block_size < 0 || (block_size > 0 && !pow2(block_size))) return block_size < 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  Plan p;
  const int st = make_plan_verify(B, gamma, Hq, Hkv, D, max_tokens, block_size, num_splits, &p);
  return st != RRA_OK ? st : p.splits;
}

size_t rra_verify_workspace_bytes(int B, int gamma, int Hq, int Hkv, int D, int splits) {
  if (B <= 0 || gamma < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || gamma > 16) return 0;
  const int64_t rows = verify_rows(B, gamma, Hq, Hkv);
  if (rows > INT32_MAX) return 0;
  return workspace_bytes(1, static_cast<int>(rows), D, splits);
}

int rra_verify_attn(const void* q_rot, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    int max_blocks_per_seq, const int32_t* positions, int block_size, int num_blocks, int max_len,
                    void* out, int B, int gamma, int Hq, int Hkv, int D, float scale, int num_splits, void* workspace,
                    size_t ws_bytes, int32_t* err_flag, void* stream) {
  return verify_launch(q_rot, k_cache, v_cache, block_table, max_blocks_per_seq, positions, block_size, num_blocks,
                       max_len, out, B, gamma, Hq, Hkv, D, scale, num_splits, workspace, ws_bytes, err_flag, stream,
                       nullptr);
}

int rra_verify_step(const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                    void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks_per_seq, int block_size,
                    int num_blocks, int max_len, void* out, int B, int gamma, int Hq, int Hkv, int D, double rope_base,
                    int rope_style, float scale, int num_splits, void* workspace, size_t ws_bytes, int32_t* err_flag,
                    void* stream) {
  // argument checks of the attention first, so that nothing is enqueued when it would refuse
  int64_t capacity = block_table ? int64_t(max_blocks_per_seq) * block_size : max_len;
  Plan p;
  if (block_table != nullptr && !pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  int st = make_plan_verify(B, gamma, Hq, Hkv, D, capacity, block_table ? block_size : 0, num_splits, &p);
  if (st != RRA_OK) return st;
  st = check_step_args(q, k_new, v_new, positions, q_out, k_cache, v_cache, out, B * gamma, Hq, D, rope_base,
                       rope_style, scale, RRA_BF16);
  if (st != RRA_OK || B == 0) return st;
  const int64_t rows = verify_rows(B, gamma, Hq, Hkv);
  st = check_workspace(p, 1, static_cast<int>(rows), D, workspace, ws_bytes);
  if (st != RRA_OK) return st;
  if (gamma <= rra::kVerifyFusedMaxGammaHost) {  // one launch: RoPE, append and attention
    const VerifyFusedArgs f{k_new, v_new, q_out, rope_style, rope_base};
    return verify_launch(q, k_cache, v_cache, block_table, max_blocks_per_seq, positions, block_size, num_blocks,
                         max_len, out, B, gamma, Hq, Hkv, D, scale, num_splits, workspace, ws_bytes, err_flag, stream,
                         &f);
  }
  st = rra_rope_append_verify(q, k_new, v_new, positions, q_out, k_cache, v_cache, block_table, max_blocks_per_seq,
                              block_size, num_blocks, max_len, B, gamma, Hq, Hkv, D, rope_base, rope_style, RRA_BF16,
                              err_flag, stream);
  if (st != RRA_OK) return st;
  return rra_verify_attn(q_out, k_cache, v_cache, block_table, max_blocks_per_seq, positions, block_size, num_blocks,
                         max_len, out, B, gamma, Hq, Hkv, D, scale, num_splits, workspace, ws_bytes, err_flag, stream);
}

int rra_prefill_attn(const void* q_rot, const void* k_cache, const void* v_cache, const int32_t* block_table,
                     int max_blocks_per_seq, const int32_t* positions, int block_size, int num_blocks, int max_len,
                     void* out, int B, int T, int Hq, int Hkv, int D, float scale, int32_t* err_flag, void* stream) {
  int st = check_shapes(B, Hq, Hkv, D, RRA_BF16);
  if (st != RRA_OK) return st;
  if (T < 1 || !std::isfinite(scale)) return RRA_EINVAL;
  int64_t capacity;
  if (block_table != nullptr) {
    if (!pow2(block_size)) return block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
    if (block_size < 8) return RRA_EUNSUPPORTED;
    if (max_blocks_per_seq < 1 || num_blocks < 1) return RRA_EINVAL;
    capacity = int64_t(max_blocks_per_seq) * block_size;
  } else {
    if (max_len < 1) return RRA_EINVAL;
    if (max_len < rra::decode_mma_tile_tokens(D)) return RRA_EUNSUPPORTED;
    capacity = max_len;
  }
  st = check_prefill_limits(T, Hq, Hkv, capacity);
  if (st != RRA_OK) return st;
  const int n_rep = Hq / Hkv;
  const int hpc = prefill_hpc(n_rep);
  if (B == 0) return RRA_OK;
  if (!q_rot || !k_cache || !v_cache || !positions || !out) return RRA_EINVAL;
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return RRA_EINVAL;
  const int tile = rra::decode_mma_tile_tokens(D);
  CUtensorMap km{}, vm{};
  if (block_table != nullptr) {
    const int box_rows = block_size < tile ? block_size : tile;
    st = encode_pool_map(&km, k_cache, num_blocks, block_size, Hkv, D, box_rows, RRA_BF16, true);
    if (st == RRA_OK) st = encode_pool_map(&vm, v_cache, num_blocks, block_size, Hkv, D, box_rows, RRA_BF16, true);
  } else {
    st = encode_contig_map(&km, k_cache, B, Hkv, max_len, D, tile, RRA_BF16);
    if (st == RRA_OK) st = encode_contig_map(&vm, v_cache, B, Hkv, max_len, D, tile, RRA_BF16);
  }
  if (st != RRA_OK) return st;
  rra::DecodeArgs a{};
  a.q = q_rot;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.hpc = hpc;
  a.gamma = T;
  a.kv_band = prefill_kv_band(T, Hkv, D);
  a.positions = positions;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.log2_bs = block_table ? ilog2(block_size) : 0;
  a.num_blocks = num_blocks;
  a.max_len = block_table ? 0 : max_len;
  a.capacity = static_cast<int>(capacity);
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  a.scale_log2 = sc * 1.4426950408889634f;
  a.err = err_flag;
  if (D == 128) {  // the tcgen05 kernel: q_rot [B*T, Hq, D] read as 128-token boxes of one head
    CUtensorMap qm{};
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(Hq), cuuint64_t(B) * T};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(Hq) * D * 2};
    const cuuint32_t box[3] = {64u, 1u, 128u};
    st = encode_map(&qm, q_rot, 3, dims, strides, box, RRA_BF16, true);
    if (st != RRA_OK) return st;
    return finish_decode(
        rra::launch_prefill_tc(a, qm, km, vm, block_table != nullptr, static_cast<cudaStream_t>(stream)));
  }
  return finish_decode(rra::launch_prefill(a, km, vm, block_table != nullptr, static_cast<cudaStream_t>(stream)));
}

int rra_prefill_step(const void* q, const void* k_new, const void* v_new, const int32_t* positions, void* q_out,
                     void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks_per_seq, int block_size,
                     int num_blocks, int max_len, void* out, int B, int T, int Hq, int Hkv, int D, double rope_base,
                     int rope_style, float scale, int32_t* err_flag, void* stream) {
  int st = check_shapes(B, Hq, Hkv, D, RRA_BF16);
  if (st != RRA_OK) return st;
  if (T < 1) return RRA_EINVAL;
  if (block_table != nullptr ? (!pow2(block_size) || block_size < 8) : max_len < rra::decode_mma_tile_tokens(D))
    return block_table != nullptr && block_size <= 0 ? RRA_EINVAL : RRA_EUNSUPPORTED;
  st = check_prefill_limits(T, Hq, Hkv,
                            block_table != nullptr ? int64_t(max_blocks_per_seq) * block_size : int64_t(max_len));
  if (st != RRA_OK) return st;
  if (int64_t(B) * T > int64_t(INT32_MAX)) return RRA_ERANGE;  // rows of q / q_out / out
  st = check_step_args(q, k_new, v_new, positions, q_out, k_cache, v_cache, out, B * T, Hq, D, rope_base, rope_style,
                       scale, RRA_BF16);
  if (st != RRA_OK || B == 0) return st;
  st = rra_rope_append_verify(q, k_new, v_new, positions, q_out, k_cache, v_cache, block_table, max_blocks_per_seq,
                              block_size, num_blocks, max_len, B, T, Hq, Hkv, D, rope_base, rope_style, RRA_BF16,
                              err_flag, stream);
  if (st != RRA_OK) return st;
  return rra_prefill_attn(q_out, k_cache, v_cache, block_table, max_blocks_per_seq, positions, block_size, num_blocks,
                          max_len, out, B, T, Hq, Hkv, D, scale, err_flag, stream);
}

}  // extern "C"
