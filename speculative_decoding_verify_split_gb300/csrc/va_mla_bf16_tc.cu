// Split-KV main kernel over an absorbed-MLA latent cache held in BF16
// (tcgen05, sm_103a). The operation is that of the FP8 latent kernel
// (va_mla_tc.cu): one KV head whose cache rows are [latent c (512) | rope key
// r (64)], logits (q_nope . c + q_pe . r) * sm_scale * k_scale, the latent c
// as the value, all Hq heads x L draft tokens (<= 64 rows) of a sequence
// sharing every cache row (sglang PR 34517 digest, "Implementation breakdown"
// item 1; its tests cover BF16 and FP8 E4M3 latent caches, item 4).
//
// Work split, roles, lazy reference max, rescale vote, bounded waits and exit
// drains follow the FP8 latent kernel. What a BF16 cache changes:
//  * Q and K are both bf16, so Q K^T runs on kind::f16 with Q as it is (no
//    hi/lo split): M = 64 packed rows (row 16q + i in TMEM lane 32q + i),
//    N = 32 keys, K = 576 in 36 steps of 16.
//  * A bf16 Q (64 rows x 1152 bytes) does not fit in TMEM beside O^T, so it
//    sits in shared memory: nine 128-byte-swizzled K-major regions (72 KB).
//  * The ring therefore holds 32-key tiles: 2 pages x nine 2 KB TMA boxes
//    (64 bf16 of 16 rows each) = 36 KB, as many bytes as a 64-key FP8 tile.
//    Its four slots form two pairs whose 128-byte regions are interleaved
//    (region c of a pair: the first tile's 32 rows, then the second's), so
//    that one Q K^T MMA spans both tiles with N = 64: a tiny N = 32 MMA costs
//    about as much as an N = 64 one. The consumers (Q K^T, softmax, P V)
//    step over such pairs of an item's tiles (64 keys); a pair whose second
//    tile lies outside the CTA's share takes a 0-byte stand-in for it.
//  * O^T = V^T P^T as in the FP8 kernel (M = 128 latent columns per chunk,
//    N = 64 rows, 256 TMEM columns), with P as one bf16 term: V^T chunk a is
//    the MN-major A operand over regions 2a and 2a + 1 of the cache tile (two
//    64-column swizzle atoms), P^T the K-major B operand (64 rows x 32 keys).
// The partials and their merge are those of the FP8 latent path.
#include <cuda_bf16.h>

#include "va_fp8.cuh"
#include "va_ptx.cuh"
#include "va_split.cuh"

namespace va {
namespace {

using namespace ptx;

constexpr int kT = kMlaTileKeysBf16;             // 32 keys per ring tile (the split unit)
constexpr int kHalves = 2;                       // ring tiles per consumer step
constexpr int kLT = kHalves * kT;                // 64 keys per consumer step
constexpr int kPagesPerTile = kT / kPageSize;    // 2
constexpr int kRegions = kMlaRow * 2 / 128;      // 9 regions of 64 bf16: latent 0-7, rope 8
constexpr int kLatentRegions = kMlaNope * 2 / 128;  // 8
constexpr int kHalfRegion = kT * 128;            // one tile's 32 rows x 128 bytes of a region
constexpr int kRegion = kLT * 128;               // 8 KB: a pair's 64 rows x 128 bytes, 128-byte swizzle
constexpr int kPairBytes = kRegions * kRegion;   // 72 KB
constexpr int kPairs = 2;
constexpr int kSlots = kPairs * kHalves;         // 4 ring slots (tiles): slot s = 2 pair + half
constexpr int kProducers = 3;                    // warps 0, 2, 3 take every third ring index
static_assert(kProducers <= kSlots, "producers exceed the ring");
constexpr int kBoxes = kPagesPerTile * kRegions;  // 18 boxes of 2 KB per tile
static_assert(kBoxes <= 32, "one box per lane");
constexpr int kSBufs = 2;                        // S tiles in TMEM (64 columns each)
constexpr int kPBuf = 64 * kLT * 2;              // P^T: 64 rows x 64 keys bf16 = 8 KB, one buffer
constexpr int kQRegion = 64 * 128;               // one 64-column region of Q: 64 rows x 128 bytes
constexpr int kQBytes = kRegions * kQRegion;     // 72 KB
constexpr int kQkSteps = kMlaRow / 16;           // 36 K-steps of 16 bf16
constexpr int kPvSteps = kT / 16;                // 2 K-steps of 16 keys per ring tile
constexpr int kChunks = kMlaNope / 128;          // 4 O^T chunks of 128 latent columns

constexpr int kOffQ = kPairs * kPairBytes;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffX = kOffP + kPBuf;           // [2 parity][2 kh][64 rows] floats
constexpr int kOffBar = kOffX + 1024;
constexpr int kSmemBytes = kOffBar + 1024;
static_assert(kSmemBytes + 1024 <= 232448, "shared memory (with the 1 KB alignment slack)");
static_assert(kPairBytes % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms");

constexpr int kThreads = 416;  // 13 warps
constexpr int kSoftmaxThreads = 256;
constexpr int kBarAllSoftmax = 5;  // named barriers: 1-4 per quadrant, 5 all softmax warps

constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdQK = instr_desc(1, 1, false, kLT, 64);       // bf16 x bf16, M = 64, N = 64 keys
constexpr uint32_t kIdPV = instr_desc(1, 1, false, 64, 128, true);  // A = V^T MN-major, N = 64 rows

// P = 2^(s - m_ref + kPShift), the reference max moved as in the FP8 latent
// kernel (a bf16 P has range to spare; the same settings keep the two paths'
// rescale behaviour alike).
constexpr float kPShift = 6.f;
constexpr float kHeadroom = 1.f;
constexpr float kHeadroomFirst = 4.f;
constexpr float kOvershoot = 2.8f;

enum : int {
  kBarFull = 0,
  kBarEmpty = kBarFull + kSlots,
  kBarSFull = kBarEmpty + kSlots,
  kBarSFree = kBarSFull + kSBufs,
  kBarPFull = kBarSFree + kSBufs,
  kBarPFree,
  kBarQFull,
  kBarQFree,
  kBarOFull,
  kBarOFree,
  kBarDrain,
  kNumBars
};
// barrier area: mbarriers | TMEM address, abort flag | scan scratch (34 x 8) |
// last tile issued into each ring slot | per-row factors [2 rounds][64] floats
constexpr int kOffTmemSlot = 8 * kNumBars;
constexpr int kOffScratch = 224;
constexpr int kOffSlotTile = kOffScratch + 34 * 8;
constexpr int kOffRowVals = 512;
static_assert(kOffTmemSlot + 8 <= kOffScratch && kOffSlotTile + 4 * kSlots <= kOffRowVals, "barrier area");

// Byte offset of element (row m, byte k) in a no-swizzle K-major operand whose
// rows are `row_bytes` long: 8-row x 16-byte core matrices, K-adjacent ones
// 128 bytes apart, 8-row groups 8 * row_bytes apart.
__device__ __forceinline__ int core_off(int m, int k, int row_bytes) {
  return (m >> 3) * (8 * row_bytes) + (k >> 4) * 128 + (m & 7) * 16 + (k & 15);
}

__global__ void __launch_bounds__(kThreads, 1)
    va_mla_bf16_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tm_kv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffBar + kOffTmemSlot + 4);
  long long* scratch = reinterpret_cast<long long*>(sm + kOffBar + kOffScratch);  // 32 slots
  long long* s_ts = scratch + 32;
  int* s_j = reinterpret_cast<int*>(scratch + 33);
  float* xch = reinterpret_cast<float*>(sm + kOffX);
  float* row_vals = reinterpret_cast<float*>(sm + kOffBar + kOffRowVals);  // [2][64]
  volatile int* slot_tile = reinterpret_cast<volatile int*>(sm + kOffBar + kOffSlotTile);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  const uint32_t sbase = smem_addr(sm);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  // The merge kernel is a programmatic dependent; it waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- setup (no global memory: runs while the stream's previous kernel ends) ---
  constexpr uint32_t kSwWarps = kSoftmaxThreads / 32;
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), kSwWarps);
    }
    mbar_init(bar(kBarPFull), kSwWarps);
    mbar_init(bar(kBarPFree), 1);
    mbar_init(bar(kBarQFull), kSwWarps);
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), kSwWarps);
    mbar_init(bar(kBarDrain), 2);
    *abort_flag = 0;
    for (int s = 0; s < kSlots; ++s) slot_tile[s] = -1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2 && lane == 0 && p.num_blocks > 0) tma_prefetch_desc(&tm_kv);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // A programmatic dependent of the stream's previous kernel (which may write
  // Q, the block table or the lengths, and may still read this workspace):
  // nothing global is read or written before its completion.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  long long t0, t1, ts_first = 0;
  int j_first = 0;
  locate_work<kThreads>(p, c, scratch, s_j, s_ts, &t0, &t1, &j_first, &ts_first);
  if (t0 >= t1) {  // CTA-uniform
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    return;
  }

  // Ring index x = 2 u + h is the h-th tile of the u-th pair this CTA
  // consumes (a pair's second tile may be a stand-in); it lives in slot
  // x % kSlots = 2 (u % kPairs) + h, and that slot's barriers name it by the
  // parity of x / kSlots.
  auto pair_base = [&](int u) { return (uint32_t)((u % kPairs) * kPairBytes); };

  if (warp == 0 || warp == 2 || warp == 3) {
    // ======================= TMA producers ======================================
    const int prod = warp == 0 ? 0 : warp - 1;
    const uint64_t kv_policy = l2_evict_first_policy();  // the cache rows are read once
    int it = 0;  // ring indices walked
    int u = 0;
    int j = j_first;
    long long ts = ts_first;
    Piece pc;
    bool ok = true;
    while (ok && next_piece(p, t0, t1, j, ts, pc)) {
      const int npages = (pc.S + kPageSize - 1) / kPageSize;
      const int* bt_row = p.block_table + (int64_t)pc.b * p.bt_s0;
      const int ntile = pc.lt1 - pc.lt0;
      int win = -1;
      int my_page = -1;
      for (int i = 0; i < ntile && ok; i += kHalves, ++u) {
        const int nh = ntile - i < kHalves ? ntile - i : kHalves;
        for (int h = 0; h < kHalves && ok; ++h, ++it) {
          if (it % kProducers != prod) continue;
          const int s = it % kSlots;
          const bool real = h < nh;  // warp-uniform
          const int lt = pc.lt0 + i + h;
          int ids[kPagesPerTile];
          uint32_t nvalid = 0;
          if (real) {
            const int pg0 = lt * kPagesPerTile;
            if (win < 0 || pg0 + kPagesPerTile > win + 32) {
              win = pg0;
              const int pg = win + lane;
              my_page = pg < npages ? bt_row[(int64_t)pg * p.bt_s1] : -1;
              if (lane == 0 && win + 32 < npages)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(bt_row + (int64_t)(win + 32) * p.bt_s1));
            }
#pragma unroll
            for (int k = 0; k < kPagesPerTile; ++k) {
              ids[k] = __shfl_sync(0xffffffffu, my_page, pg0 + k - win);
              const bool v = (pg0 + k) < npages && (unsigned)ids[k] < (unsigned)p.num_blocks;
              ids[k] = v ? ids[k] : -1;
              nvalid += v ? 1u : 0u;
            }
          }
          const bool got = __all_sync(
              0xffffffffu, mbar_wait(bar(kBarEmpty + s), ((it / kSlots) & 1) ^ 1, abort_flag, p.wait_limit_ns));
          if (!got) {
            if (lane == 0) fail(p, abort_flag, 1);
            ok = false;
            break;
          }
          // rows [32 h, +32) of every region of the pair; a stand-in brings 0 bytes
          const uint32_t dst = sbase + pair_base(u) + h * kHalfRegion;
          if (lane == 0) {
            slot_tile[s] = it;
            mbar_arrive_expect_tx(bar(kBarFull + s), nvalid * (uint32_t)(kRegions * 2048));
          }
          __syncwarp();
          if (real && lane < kBoxes) {  // lane -> (page, 64-column region)
            const int k = lane / kRegions, ch = lane % kRegions;
            const int id = k == 0 ? ids[0] : ids[1];
            if (id >= 0)
              tma_load_4d_hint(dst + ch * kRegion + k * 2048, &tm_kv, ch * 64, 0, 0, id, bar(kBarFull + s),
                               kv_policy);
          }
          __syncwarp();
        }
      }
    }
    // Copies still in flight land before the CTA goes away, also when another
    // role gave up (the window: see the GQA kernel's producers).
    if (lane == 0) {
      for (int k = (it > kSlots + kProducers - 1 ? it - kSlots - kProducers + 1 : 0); k < it; ++k) {
        if (k % kProducers != prod) continue;
        drain_ring_tile(bar(kBarFull + k % kSlots), k, kSlots, slot_tile + k % kSlots, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 12) {
    // ======================= MMA issuers ==========================================
    if (lane == 0) {
      const bool is_qk = warp == 1;
      const uint32_t qbase = sbase + kOffQ;
      const uint32_t pbuf = sbase + kOffP;
      int u = 0, piece_idx = 0;
      int j = j_first;
      long long ts = ts_first;
      Piece pc;
      bool ok = true;
      auto wait_or_fail = [&](int b, uint32_t par, int code) {
        if (!ok) return false;
        if (!mbar_wait(bar(b), par, abort_flag, p.wait_limit_ns)) {
          fail(p, abort_flag, code);
          ok = false;
        }
        return ok;
      };
      while (ok && next_piece(p, t0, t1, j, ts, pc)) {
        const int ntile = pc.lt1 - pc.lt0;
        for (int i = 0; i < ntile && ok; i += kHalves, ++u) {
          const int nh = ntile - i < kHalves ? ntile - i : kHalves;
          const uint32_t base = sbase + pair_base(u);
          const uint32_t full_par = (uint32_t)((2 * u / kSlots) & 1);
          if (is_qk) {
            if (i == 0 && !wait_or_fail(kBarQFull, piece_idx & 1, 2)) break;
            const int b = u & (kSBufs - 1);
            if (u >= kSBufs && !wait_or_fail(kBarSFree + b, ((u - kSBufs) / kSBufs) & 1, 64)) break;
            // both tiles of the pair (a stand-in lands at once)
            if (!wait_or_fail(kBarFull + 2 * (u % kPairs), full_par, 32)) break;
            if (!wait_or_fail(kBarFull + 2 * (u % kPairs) + 1, full_par, 32)) break;
            tc_fence_after();
#pragma unroll 4
            for (int k = 0; k < kQkSteps; ++k) {
              const uint32_t off = (uint32_t)((k >> 2) * kQRegion + (k & 3) * 32);
              const uint64_t a = smem_desc(qbase + off, 16, 1024, kLayoutSw128);
              const uint64_t bdesc =
                  smem_desc(base + (uint32_t)((k >> 2) * kRegion + (k & 3) * 32), 16, 1024, kLayoutSw128);
              mma_f16(tmem + kColS + b * kLT, a, bdesc, kIdQK, k ? 1u : 0u);
            }
            mma_commit(bar(kBarSFull + b));
            if (i + nh >= ntile) mma_commit(bar(kBarQFree));
          } else {
            if (!wait_or_fail(kBarPFull, u & 1, 4)) break;
            if (!wait_or_fail(kBarFull + 2 * (u % kPairs), full_par, 8)) break;
            if (!wait_or_fail(kBarFull + 2 * (u % kPairs) + 1, full_par, 8)) break;
            if (i == 0 && piece_idx > 0 && !wait_or_fail(kBarOFree, (piece_idx - 1) & 1, 16)) break;
            tc_fence_after();
            for (int h = 0; h < nh; ++h) {
#pragma unroll
              for (int kk = 0; kk < kPvSteps; ++kk) {
                // P^T: 64 rows x keys [32 h + 16 kk, +16) (two K-adjacent core matrices)
                const uint64_t bdesc = smem_desc(pbuf + (4 * h + 2 * kk) * 128, 128, 8 * kLT * 2, kLayoutNone);
#pragma unroll
                for (int a = 0; a < kChunks; ++a) {
                  // V^T chunk a: latent columns [128 a, +128) = regions 2a, 2a + 1
                  // (two 64-column atoms, kRegion apart), rows of tile h,
                  // keys [16 kk, +16)
                  const uint64_t adesc = smem_desc(base + (2 * a) * kRegion + h * kHalfRegion + kk * 2048,
                                                   kRegion, 1024, kLayoutSw128);
                  mma_f16(tmem + kColO + 64 * a, adesc, bdesc, kIdPV, (i == 0 && h == 0 && kk == 0) ? 0u : 1u);
                }
              }
            }
            // both slots are free once P V has read them (a stand-in at once)
            mma_commit(bar(kBarEmpty + 2 * (u % kPairs)));
            mma_commit(bar(kBarEmpty + 2 * (u % kPairs) + 1));
            mma_commit(bar(kBarPFree));
            if (i + nh >= ntile) mma_commit(bar(kBarOFull));
          }
        }
        ++piece_idx;
      }
      mma_commit(bar(kBarDrain));
      mbar_wait_drain(bar(kBarDrain), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ======================= softmax / epilogue ===================================
    const int q = warp & 3;              // TMEM lane quadrant
    const int kh = (warp - 4) >> 2;      // which tile of a pair (keys), half of the O^T chunks
    const int sub = lane >> 4;
    const int rl = lane & 15;
    const int r = 16 * q + rl;           // packed row
    const int qtr = 2 * kh + sub;        // 16-key quarter of a pair, quarter of Q staging
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float kd = p.k_descale ? *p.k_descale : 1.0f;
    const float cscale = p.scale_log2 * kd;
    const int G = p.group;
    unsigned char* qs = sm + kOffQ;
    int u = 0, piece_idx = 0, round = 0;
    int j = j_first;
    long long ts = ts_first;
    Piece pc;
    bool ok = true;
    // Waits are warp-uniform; after a failure the warp walks the same pieces
    // and pairs "dry" so that every named barrier still sees all its threads.
    auto wait_or_fail = [&](int b, uint32_t par, int code) {
      if (!ok) return false;
      const bool got = __all_sync(0xffffffffu, mbar_wait(bar(b), par, abort_flag, p.wait_limit_ns));
      if (!got) {
        if (lane == 0) fail(p, abort_flag, code);
        ok = false;
      }
      return ok;
    };
    // Row-wide combine over the row's four threads (lanes t, t ^ 16 of this
    // warp and of the quadrant's other warp), as in the GQA kernel.
    int xround = 0;
    auto exchange = [&](float v, bool is_max) {
      v = is_max ? fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16)) : v + __shfl_xor_sync(0xffffffffu, v, 16);
      const int par = xround & 1;
      ++xround;
      if (sub == 0) xch[(par * 2 + kh) * 64 + r] = v;
      named_bar(1 + q, 64);
      const float other = xch[(par * 2 + (kh ^ 1)) * 64 + r];
      return is_max ? fmaxf(v, other) : v + other;
    };
    // Q of piece pq into the K-major 128-byte-swizzled A operand: this
    // thread copies 16-byte pieces [18 qtr, +18) of row r's 72 (bf16 as it
    // is). Returns the row's logit scale.
    auto stage_q = [&](const Piece& pq, int qidx) -> float {
      if (qidx > 0) wait_or_fail(kBarQFree, (qidx - 1) & 1, 128);
      const bool row_ok = r < pq.R;
      const int tq = row_ok ? r / G : 0;
      const int gq = row_ok ? r - tq * G : 0;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (int64_t)(pq.q0 + tq) * p.q_s0 + (int64_t)gq * p.q_s1);
      if (ok) {
#pragma unroll 6
        for (int k = 0; k < 18; ++k) {
          const int pi = 18 * qtr + k;           // 16-byte piece of the row (8 bf16)
          const int region = pi >> 3, p16 = pi & 7;
          const uint4 v = row_ok ? src[pi] : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(qs + region * kQRegion + r * 128 + ((p16 ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQFull));
      }
      return row_ok ? cscale : 0.f;
    };
    float rs_next = 0.f;
    bool staged_next = false;
    while (next_piece(p, t0, t1, j, ts, pc)) {
      Piece pn;
      int jn = j;
      long long tsn = ts;
      const bool has_next = next_piece(p, t0, t1, jn, tsn, pn);
      const float rs = staged_next ? rs_next : stage_q(pc, piece_idx);
      staged_next = false;
      const bool row_ok = r < pc.R;
      const int tq = row_ok ? r / G : 0;

      float m_ref = -INFINITY;
      float l = 0.f;
      const int vis_end = pc.S - pc.L + tq;  // last visible key of this row
      const int ntile = pc.lt1 - pc.lt0;
      for (int i = 0; i < ntile; i += kHalves, ++u) {
        const int nh = ntile - i < kHalves ? ntile - i : kHalves;
        const int lt = pc.lt0 + i;           // the pair's first tile
        const int b = u & (kSBufs - 1);
        if (i + nh >= ntile && has_next) {
          rs_next = stage_q(pn, piece_idx + 1);
          staged_next = true;
        }
        float x[16];  // logits of keys [16 qtr, +16) of this pair (tile kh), this row
#pragma unroll
        for (int k = 0; k < 16; ++k) x[k] = -INFINITY;
        if (wait_or_fail(kBarSFull + b, (u / kSBufs) & 1, 256)) {
          tc_fence_after();
          if (kh < nh) {  // warp-uniform: a stand-in tile's columns are never read
            // lanes 0-15 of the quadrant hold rows 16q + i; this warp reads
            // keys [32 kh, +32), the half-warps 16 each
            uint32_t v[16];
            tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kColS + b * kLT + 32 * kh, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) x[k] = __uint_as_float(v[k]) * rs;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarSFree + b));
          const int key0 = lt * kT + 16 * qtr;
          if ((lt + nh) * kT - 1 > pc.S - pc.L) {  // tail: causal mask
#pragma unroll
            for (int k = 0; k < 16; ++k)
              if (key0 + k > vis_end) x[k] = -INFINITY;
          }
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < 16; k += 2) tmax = fmaxf(tmax, fmaxf(x[k], x[k + 1]));
        tmax = exchange(tmax, true);

        const bool need = ok && tmax > m_ref + kOvershoot;
        const float m_new = need ? tmax + (m_ref == -INFINITY ? kHeadroomFirst : kHeadroom) : m_ref;
        const bool rescale = need && (m_ref != -INFINITY) && (i > 0);
        const float alpha = rescale ? ex2(m_ref - m_new) : 1.f;
        // O^T keeps a row in a column across all 128 lanes: every softmax
        // warp scales its lanes' part of the rows that moved, so the decision
        // is taken by all of them at once
        float* al = row_vals + (round & 1) * 64;
        ++round;
        if (kh == 0 && sub == 0) al[r] = alpha;
        const bool any = named_bar_or(kBarAllSoftmax, kSoftmaxThreads, rescale);
        if (!ok) continue;

        // the P buffer was last read by P V(u - 1), which has also put its
        // tiles into O^T before a rescale
        if (u > 0 && !wait_or_fail(kBarPFree, (u - 1) & 1, 512)) continue;
        tc_fence_after();
        const float mref_s = m_new - kPShift;
        const bool live = m_new != -INFINITY;
        uint32_t pw[8];
        float ls = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float a = live ? ex2(x[2 * k] - mref_s) : 0.f;
          const float bb = live ? ex2(x[2 * k + 1] - mref_s) : 0.f;
          ls += a + bb;
          pw[k] = pack_bf16x2(a, bb);
        }
        // P^T operand: row r, keys [16 qtr, +16) = 32 bytes, two core-matrix rows
        unsigned char* pbuf = sm + kOffP;
        *reinterpret_cast<uint4*>(pbuf + core_off(r, 32 * qtr, kLT * 2)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(pbuf + core_off(r, 32 * qtr + 16, kLT * 2)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
        // then the rows that moved (P V(u - 1) is in O^T: waited above)
        if (any) {
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kColO + 64 * (2 * kh + (k >> 1)) + 32 * (k & 1);
            tmem_ld_32x32b_x32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int c2 = 0; c2 < 32; ++c2) o[c2] = __float_as_uint(__uint_as_float(o[c2]) * al[32 * (k & 1) + c2]);
            tmem_st_32x32b_x32(ta, o);
          }
          tmem_wait_st();
        }
        l = l * alpha + ls;
        m_ref = m_new;
        // latent rows past S in the item's last tile (a partial page, a page
        // never loaded) are zeroed so that 0 * garbage cannot reach O; Q K^T
        // of this pair has completed (S was full)
        const int hl = pc.nt - 1 - lt;  // the tile of the pair that ends the item, if any
        if (hl >= 0 && hl < nh && (pc.S % kT) != 0) {
          const int zt0 = pc.S - (lt + hl) * kT;
          unsigned char* vst = sm + pair_base(u) + hl * kHalfRegion;
          for (int idx = tid - 128; idx < (kT - zt0) * kLatentRegions * 8; idx += kSoftmaxThreads) {
            const int row = zt0 + idx / (kLatentRegions * 8);
            const int rem = idx % (kLatentRegions * 8);
            *reinterpret_cast<uint4*>(vst + (rem >> 3) * kRegion + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        tc_fence_before();  // the O^T rescale, before the arrive
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull));
      }

      // -- epilogue: as in the FP8 latent kernel. This thread's lane holds
      // latent column 128 a + 32 q + lane of chunks a = 2 kh, 2 kh + 1, for
      // all packed rows; every piece leaves (m, l) and its unnormalised O^T in
      // groups of four rows (mla_acc_index) for the merge kernel.
      const float lrow = exchange(l, false);
      wait_or_fail(kBarOFull, piece_idx & 1, 4096);
      tc_fence_after();
      ++piece_idx;
      if (!ok) continue;
      const int64_t piece = (int64_t)pc.j + c;
      const int ldr = mla_row_stride(p.max_rows);
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int a = 2 * kh + (k >> 1);
        const int r0 = 32 * (k & 1);
        if (r0 >= pc.R) continue;  // warp-uniform
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kColO + 64 * a + r0, o);
        tmem_wait_ld();
        const int col = 128 * a + 32 * q + lane;
        const int nrow = ldr - r0 < 32 ? ldr - r0 : 32;
#pragma unroll
        for (int w = 0; w < 8; ++w)
          if (4 * w < nrow)
            *reinterpret_cast<float4*>(p.ws_acc + mla_acc_index(piece, r0 + 4 * w, col, ldr)) =
                make_float4(__uint_as_float(o[4 * w]), __uint_as_float(o[4 * w + 1]),
                            __uint_as_float(o[4 * w + 2]), __uint_as_float(o[4 * w + 3]));
      }
      if (row_ok && kh == 0 && sub == 0) {
        p.ws_ml[(piece * p.max_rows + r) * 2 + 0] = (m_ref == -INFINITY) ? -INFINITY : m_ref - kPShift;
        p.ws_ml[(piece * p.max_rows + r) * 2 + 1] = lrow;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t prepare_mla_bf16_tc() {
  return cudaFuncSetAttribute(va_mla_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes + 1024);
}

cudaError_t launch_mla_bf16_tc(const Params& p, const CUtensorMap& tm_kv, cudaStream_t stream) {
  // a programmatic dependent of the stream's previous kernel (see the kernel)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, va_mla_bf16_tc_kernel, p, tm_kv);
}

}  // namespace va
