// Device helpers for the split-KV decomposition shared by the main and merge
// kernels: per-sequence lengths (clamped so no access leaves its buffer), the
// key-tile count of each (sequence, KV head) work item, and the mapping from a
// global key tile to the CTA whose equal share contains it.
#pragma once

#include <cuda_bf16.h>

#include "va_internal.h"

namespace va {

// Draft tokens of sequence b, clamped to [0, max_seqlen_q] and to the rows of q.
__device__ __forceinline__ int seq_q_len(const Params& p, int b) {
  const int a = p.cu_q[b];
  const int e = p.cu_q[b + 1];
  int L = e - a;
  L = L < 0 ? 0 : L;
  L = L > p.max_seqlen_q ? p.max_seqlen_q : L;
  if (a < 0) return 0;
  const int room = p.total_q - a;
  return L > room ? (room < 0 ? 0 : room) : L;
}

// Cached tokens of sequence b, clamped to what its block-table row can address.
__device__ __forceinline__ int seq_kv_len(const Params& p, int b) {
  int S = p.seqused_k[b];
  S = S < 0 ? 0 : S;
  const int cap = p.bt_width * kPageSize;
  return S > cap ? cap : S;
}

// First key any draft token of a sequence (S cached tokens, L draft tokens)
// can see: 0, or with a sliding window the start of the first token's window.
__device__ __forceinline__ int first_key(const Params& p, int S, int L) {
  if (p.window_left < 0) return 0;
  const int k0 = S - L - p.window_left;
  return k0 > 0 ? k0 : 0;
}

// First key tile of a sequence's work (tiles wholly before the window are
// never read).
__device__ __forceinline__ int first_tile(const Params& p, int S, int L) {
  return first_key(p, S, L) / p.tile_keys;
}

// Key tiles of work item j (b = j / hkv): those from the first visible key to
// the end. A sequence without draft tokens needs no work.
__device__ __forceinline__ int work_tiles(const Params& p, int j) {
  const int b = j / p.hkv;
  const int L = seq_q_len(p, b);
  if (L == 0) return 0;
  const int S = seq_kv_len(p, b);
  const int nt = (S + p.tile_keys - 1) / p.tile_keys;
  return nt > 0 ? nt - first_tile(p, S, L) : 0;
}

// One sequence's clamped lengths as the split uses them: S cached keys, L
// draft tokens, its first Q row q0 and causal extent E (S, or a shard's
// kv_extent). A small batch's are kept in shared memory from the work scan
// on (see locate_work), so that moving to the next piece reads no global
// memory: under full HBM load each such read costs about a microsecond, and
// every role makes it at every piece boundary.
struct SeqMeta {
  int S, L, q0, E;
};
constexpr int kSeqCache = 64;  // sequences a cache holds

__device__ __forceinline__ SeqMeta seq_meta(const Params& p, const SeqMeta* cache, int b) {
  if (cache) return cache[b];
  SeqMeta m;
  m.S = seq_kv_len(p, b);
  m.L = seq_q_len(p, b);
  m.q0 = p.cu_q[b];
  m.E = m.S;
  if (p.kv_extent) {
    const int e = p.kv_extent[b];
    m.E = e > m.S ? e : m.S;
  }
  return m;
}

// Key tiles of an item whose sequence has lengths m (as work_tiles).
__device__ __forceinline__ int meta_tiles(const Params& p, const SeqMeta& m) {
  if (m.L == 0) return 0;
  const int nt = (m.S + p.tile_keys - 1) / p.tile_keys;
  return nt > 0 ? nt - first_tile(p, m.S, m.L) : 0;
}

// Split cost of work item j with nt tiles: the tiles plus the item's start-up
// cost, which comes first in split units.
__device__ __forceinline__ long long work_cost(const Params& p, int nt) {
  return nt > 0 ? (long long)nt + p.piece_cost : 0;
}

// First split unit of CTA c when N units are cut into G equal ranges.
__device__ __forceinline__ long long split_begin(long long N, int c, int G) {
  return (N * (long long)c) / G;
}

// The CTA whose range contains split unit x (0 <= x < N): the largest c with
// split_begin(c) <= x, i.e. c*N < (x+1)*G.
__device__ __forceinline__ int split_of(long long x, long long N, int G) {
  return (int)(((x + 1) * (long long)G - 1) / N);
}

// Block-wide exclusive scan of one value per thread (NT threads, NT % 32 == 0).
// Returns the exclusive prefix; *total receives the block sum. Uses 32 slots
// of shared scratch; contains __syncthreads.
template <int NT>
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* scratch,
                                                          long long* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const long long base = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[NT / 32 - 1];
  __syncthreads();
  return base + x - v;
}

// Scans the split costs of all work items. When write_meta, stores the split
// unit of the first tile of every item in ws_meta and the total at
// ws_meta[num_work]. Returns the total N.
template <int NT>
__device__ long long scan_work(const Params& p, long long* scratch, bool write_meta) {
  long long running = 0;
  for (int base = 0; base < p.num_work; base += NT) {
    const int j = base + (int)threadIdx.x;
    const int nt = j < p.num_work ? work_tiles(p, j) : 0;
    const long long v = work_cost(p, nt);
    long long tot;
    const long long ex = block_exclusive_scan<NT>(v, scratch, &tot);
    if (write_meta && j < p.num_work) p.ws_meta[j] = (int32_t)(running + ex + (v - nt));
    running += tot;
  }
  if (write_meta && threadIdx.x == 0) p.ws_meta[p.num_work] = (int32_t)running;
  return running;
}

// The block-table entry of item j's tile lt, prefetched into L2: the TMA
// producers' first load, whose latency then overlaps the CTA's setup.
__device__ __forceinline__ void prefetch_first_pages(const Params& p, int j, long long lt) {
  const int b = j / p.hkv;
  lt += first_tile(p, seq_kv_len(p, b), seq_q_len(p, b));  // lt counts from the item's first tile
  const int* bt = p.block_table + (int64_t)b * p.bt_s0 +
                  (int64_t)(lt * p.tile_keys / kPageSize) * p.bt_s1;
  asm volatile("prefetch.global.L2 [%0];" ::"l"(bt));
}

// Finds the work item whose split range contains unit x (0 <= x < N) and the
// unit of its first tile. Every thread gets the answer.
template <int NT>
__device__ void find_work(const Params& p, long long x, long long* scratch, int* s_j,
                          long long* s_ts, int* out_j, long long* out_ts) {
  long long running = 0;
  for (int base = 0; base < p.num_work; base += NT) {
    const int j = base + (int)threadIdx.x;
    const int nt = j < p.num_work ? work_tiles(p, j) : 0;
    const long long v = work_cost(p, nt);
    long long tot;
    const long long ex = block_exclusive_scan<NT>(v, scratch, &tot);
    const long long s = running + ex;
    if (j < p.num_work && v > 0 && s <= x && x < s + v) {
      *s_j = j;
      *s_ts = s + (v - nt);
      prefetch_first_pages(p, j, x > s + (v - nt) ? x - (s + (v - nt)) : 0);
    }
    running += tot;
  }
  __syncthreads();
  *out_j = *s_j;
  *out_ts = *s_ts;
}

// This CTA's split range [t0, t1) and, if it is not empty, its first work
// item and the unit of that item's first tile. With at most one item per
// thread the block scan's total is known in the same pass, so one scan does
// both jobs; larger batches scan twice. Returns N.
//
// With a non-null `cache` (kSeqCache entries of shared memory) and a batch
// small enough (at most NT items and kSeqCache sequences), the scan also
// stores every sequence's lengths there; *cached then says so (for
// next_piece's `cache` argument).
template <int NT>
__device__ long long locate_work(const Params& p, int c, long long* scratch, int* s_j,
                                 long long* s_ts, long long* t0, long long* t1, int* out_j,
                                 long long* out_ts, SeqMeta* cache = nullptr, bool* cached = nullptr) {
  if (cached) *cached = false;
  if (p.num_work > NT) {
    const long long N = scan_work<NT>(p, scratch, c == 0);
    *t0 = split_begin(N, c, p.num_splits);
    *t1 = split_begin(N, c + 1, p.num_splits);
    if (*t0 < *t1) find_work<NT>(p, *t0, scratch, s_j, s_ts, out_j, out_ts);
    return N;
  }
  const int j = (int)threadIdx.x;
  const bool fill = cache != nullptr && p.num_seqs <= kSeqCache;  // CTA-uniform
  int nt = 0;
  if (j < p.num_work) {
    const int b = j / p.hkv;
    const SeqMeta m = seq_meta(p, nullptr, b);
    nt = meta_tiles(p, m);
    if (fill && j - b * p.hkv == 0) cache[b] = m;
  }
  const long long v = work_cost(p, nt);
  long long N;
  const long long s = block_exclusive_scan<NT>(v, scratch, &N);  // its barriers publish the cache
  if (cached) *cached = fill;
  *t0 = split_begin(N, c, p.num_splits);
  *t1 = split_begin(N, c + 1, p.num_splits);
  if (c == 0 && j < p.num_work) p.ws_meta[j] = (int32_t)(s + (v - nt));
  if (c == 0 && j == 0) p.ws_meta[p.num_work] = (int32_t)N;
  if (*t0 < *t1 && j < p.num_work && v > 0 && s <= *t0 && *t0 < s + v) {
    *s_j = j;
    *s_ts = s + (v - nt);
    prefetch_first_pages(p, j, *t0 > s + (v - nt) ? *t0 - (s + (v - nt)) : 0);
  }
  __syncthreads();
  *out_j = *s_j;
  *out_ts = *s_ts;
  return N;
}

// One (sequence, KV head) item's share of this CTA. Tile indices are absolute
// within the sequence: the item's tiles are [tb, nt), this CTA's [lt0, lt1).
struct Piece {
  int j, b, kvh, S, L, q0, R, nt, tb, lt0, lt1;
  int E;  // the causal extent: S, or the shard's kv_extent (>= S)
  bool direct;
};

// Next (sequence, KV head) item with tiles in this CTA's split range [t0, t1);
// ts is the split unit of item j's first tile.
// `cache`: the sequences' lengths in shared memory (locate_work), or null.
__device__ __forceinline__ bool next_piece(const Params& p, long long t0, long long t1, int& j,
                                           long long& ts, Piece& pc, const SeqMeta* cache = nullptr) {
  while (j < p.num_work && ts < t1) {
    const int b = j / p.hkv;
    const SeqMeta m = seq_meta(p, cache, b);
    const int nt = meta_tiles(p, m);
    if (nt == 0) {
      ++j;
      continue;
    }
    pc.j = j;
    pc.b = b;
    pc.kvh = j - pc.b * p.hkv;
    pc.S = m.S;
    pc.L = m.L;
    pc.E = m.E;
    pc.q0 = m.q0;
    pc.R = p.group * pc.L;
    pc.tb = first_tile(p, pc.S, pc.L);
    pc.nt = pc.tb + nt;
    pc.lt0 = pc.tb + (int)((t0 > ts ? t0 : ts) - ts);
    pc.lt1 = pc.tb + (int)((t1 < ts + nt ? t1 : ts + nt) - ts);
    pc.direct = !p.partial && (pc.lt0 == pc.tb && pc.lt1 == pc.nt);
    ts += work_cost(p, nt);  // the next item's first tile follows its start-up units
    ++j;
    return true;
  }
  return false;
}

__device__ __forceinline__ void fail(const Params& p, volatile int* abort_flag, int code) {
  *abort_flag = 1;
  if (p.ws_status) atomicOr(p.ws_status, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

}  // namespace va
