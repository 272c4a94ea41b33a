// Internal launch parameters shared by the host library and the kernels.
// Not part of the C ABI (include/verify_attn.h is).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace va {

constexpr int kHeadDim = 256;
// Absorbed-MLA latent cache (sglang PR 34517 digest, "Implementation breakdown"
// item 1): one KV head whose rows are [latent (NOPE) | rope key (PE)]; the
// latent is also the value. The latent width is not on the pages: 512, as in
// the DeepSeek-V3 / Kimi-K2 MLA family.
constexpr int kMlaNope = 512;
constexpr int kMlaPe = 64;
constexpr int kMlaRow = kMlaNope + kMlaPe;  // 576
// Row stride of the latent path's column-major partials (a multiple of 4
// rows, so that 4 rows are one 16-byte store).
__host__ __device__ constexpr int mla_row_stride(int max_rows) { return (max_rows + 3) & ~3; }
// Index of (row, column) of piece `piece` in those partials, laid out in
// groups of four rows: [piece][row / 4][column][row % 4].
__host__ __device__ constexpr int64_t mla_acc_index(int64_t piece, int row, int col, int ldr) {
  return ((piece * (ldr / 4) + row / 4) * kMlaNope + col) * 4 + (row % 4);
}
constexpr int kPageSize = 16;
constexpr int kMaxRows = 64;  // G * max_seqlen_q packed rows per (sequence, KV head)

// Everything a kernel needs, by value. Strides are in elements.
struct Params {
  const uint16_t* q;  // bf16 bits
  int64_t q_s0, q_s1;
  const void* k;
  int64_t k_s0, k_s1, k_s2;
  const void* v;
  int64_t v_s0, v_s1, v_s2;
  const int32_t* block_table;
  int64_t bt_s0, bt_s1;
  int32_t bt_width;
  const int32_t* cu_q;
  const int32_t* seqused_k;
  const float* k_descale;  // nullable
  const float* v_descale;  // nullable
  uint16_t* out;           // bf16 bits
  int64_t o_s0, o_s1;
  int32_t out_v8;          // out and its row strides are 32-byte aligned (32-byte stores)
  int32_t num_seqs, hq, hkv, group, num_blocks, total_q, max_seqlen_q, max_seqlen_k;
  int32_t kv_fp8;
  float scale_log2;  // softmax_scale * log2(e)
  // Variants of the generic attention (sliding window, logit soft-cap, sinks).
  int32_t window_left;     // -1: none; else position i sees keys [i - window_left, i]
  float softcap_log2;      // 0: none; else softcap * log2(e): x -> c tanh(x / c) in log2 units
  const float* sinks;      // nullable, [hq]: per-head sink logits (natural log)
  // One shard of each sequence's keys (verify_attn_partial): with kv_extent,
  // draft token t of sequence b sees the shard's local keys j <= extent_b - L + t
  // (extent_b = the sequence's total keys - the shard's first key position);
  // with partial, every item goes through the merge, which writes o (fp32,
  // normalised) and lse (natural log) instead of out.
  const int32_t* kv_extent;  // nullable: extent = seqused_k
  int32_t partial;
  float* o_part;             // [total_q, hq, 256]
  int64_t op_s0, op_s1;
  float* lse_part;           // [total_q, hq]
  int64_t lse_s0, lse_s1;

  // Split-KV decomposition: one stream of key tiles over all work items
  // j = b * hkv + kvh, cut into num_splits equal ranges (one per CTA). Each
  // item also costs piece_cost units ahead of its first tile (its Q staging,
  // epilogue and pipeline refill), so a CTA that starts an item gets fewer
  // tiles.
  int32_t tile_keys, num_splits, max_rows, num_work, piece_cost;
  int32_t q_in_tmem;   // 1: the plan chose kKernelTcQTmem (used unless a variant option is set)
  int32_t dv;          // output (value) columns: kHeadDim, or kMlaNope over a latent cache
  // Limit of every bounded wait of the main kernels, in ns (kDefaultWaitLimitNs
  // unless a test shortened it to make waits run out).
  uint64_t wait_limit_ns;
  int32_t* ws_status;  // sticky error bits (a bounded wait timed out); never cleared by kernels
  int32_t* ws_meta;  // [num_work + 1]: first tile of each work item (split units), then the total
  float* ws_ml;      // [pieces][max_rows][2]: running max (log2 units), row sum
  float* ws_acc;     // [pieces][max_rows][dv]: unnormalised output rows
};

// A bounded wait of the main kernels gives up after this long (by
// %globaltimer), sets the workspace status word and lets the kernel wind down.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
// The drains on the way out (copies and MMAs in flight) wait this long at most.
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 100 ms

// Workspace layout. pieces = num_work + num_splits: a work item split over
// CTAs c0..c1 stores the partial of CTA c at piece j + c, which is unique
// because consecutive work items share at most one CTA.
struct WorkspaceLayout {
  size_t status_off, meta_off, ml_off, acc_off, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WorkspaceLayout workspace_layout(int64_t num_work, int64_t num_splits, int64_t max_rows,
                                        int64_t dv = kHeadDim) {
  WorkspaceLayout w;
  const int64_t pieces = num_work + num_splits;
  w.status_off = 0;
  w.meta_off = 256;
  w.ml_off = w.meta_off + align_up(sizeof(int32_t) * (size_t)(num_work + 1), 256);
  w.acc_off = w.ml_off + align_up(sizeof(float) * 2 * (size_t)(pieces * max_rows), 256);
  w.total = w.acc_off + align_up(sizeof(float) * (size_t)dv * (size_t)(pieces * max_rows), 256);
  return w;
}

// Main kernel (tensor cores) and its key-tile sizes. kKernelTc keeps Q in
// shared memory (FP8: two S tiles, each P written over its S); kKernelTcQTmem,
// the FP8 kernel for batches of at least kSmallSplitTiles tiles per CTA,
// takes Q and P from TMEM (one S tile) and spends the shared memory on a
// fourth K ring slot. The variant options (window, soft cap, sinks) always
// run the first layout.
enum Kernel : int32_t { kKernelTc = 1, kKernelTcQTmem = 2 };
constexpr int kTcTileKeysFp8 = 128;  // keys per tile, FP8 KV
constexpr int kTcTileKeysBf16 = 64;  // keys per tile, BF16 KV
// Split cost of starting a work item, in tiles: a CTA's boundary between two
// items (epilogue of one, Q staging and pipeline refill of the next). Swept
// over 2/3/4/6/8 on the mid- and long-context FP8 workloads: 4 is best on both.
// When the tile bound per CTA is under kSmallSplitTiles, every CTA pays a
// start-up of its own and charging it to the CTAs that start an item only
// unbalances the split: swept over 1-4 there, 1 is best (main kernel,
// gqa_32q2kv 22.5 -> 21.2 us on one box and 22.9 -> 22.7 on another,
// tiny_verify 18.7 -> 18.4).
constexpr int kPieceCostTiles = 4;
constexpr int kPieceCostTilesSmall = 1;
constexpr int64_t kSmallSplitTiles = 16;

cudaError_t launch_merge(const Params& p, cudaStream_t stream);

// Log-sum-exp merge of shard results (verify_attn_merge_partials).
constexpr int kMaxShards = 16;
struct ShardMergeParams {
  int32_t n, total_q, hq;
  const float* o[kMaxShards];
  int64_t o_s0[kMaxShards], o_s1[kMaxShards];
  const float* lse[kMaxShards];
  int64_t lse_s0[kMaxShards], lse_s1[kMaxShards];
  uint16_t* out;  // bf16 [total_q, hq, 256]
  int64_t out_s0, out_s1;
};
cudaError_t launch_merge_shards(const ShardMergeParams& m, cudaStream_t stream);

// Block table from the flat token-slot form (va_pagetable.cu). Status bits:
constexpr int32_t kBtBadPage = 1;     // a page's slots are not one aligned page in order
constexpr int32_t kBtTruncated = 2;   // a sequence has more pages than the table is wide
constexpr int32_t kBtBadIndptr = 4;   // kv_indptr decreases, is negative or passes nnz
cudaError_t launch_block_table(const int32_t* indptr, const int32_t* indices, int64_t nnz,
                               int32_t num_seqs, int32_t width, int32_t* bt, int64_t bt_s0,
                               int64_t bt_s1, int32_t* seqused, int64_t sk_s0, int32_t pad,
                               int32_t* status, cudaStream_t stream);
cudaError_t prepare_main_tc();  // once per device: opt in to its shared memory
// Latent-cache main kernel (va_mla_tc.cu): FP8 cache, 64-key tiles.
constexpr int kMlaTileKeys = 64;
// Split cost of starting an item on the latent path, in 64-key tiles: Q
// staging (576 columns) and the 128 KB partial of the previous piece, both
// through a memory system saturated by the ring. Swept over 12/18/24 on the
// mid- and long-context latent workloads (same box, back to back): 12 is
// best by ~1.5 us on both.
constexpr int kMlaPieceCostTiles = 12;
cudaError_t prepare_mla_tc();
cudaError_t launch_mla_tc(const Params& p, const CUtensorMap& tm_kv, const CUtensorMap& tm_pe,
                          cudaStream_t stream);
// Latent-cache main kernel over a BF16 cache (va_mla_bf16_tc.cu): 32-key
// tiles (36 KB, the bytes of a 64-key FP8 tile), Q in shared memory. Its
// piece cost is the FP8 kernel's in keys.
constexpr int kMlaTileKeysBf16 = 32;
constexpr int kMlaPieceCostTilesBf16 = 2 * kMlaPieceCostTiles;
cudaError_t prepare_mla_bf16_tc();
cudaError_t launch_mla_bf16_tc(const Params& p, const CUtensorMap& tm_kv, cudaStream_t stream);
cudaError_t launch_main_tc(const Params& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           cudaStream_t stream);

}  // namespace va
