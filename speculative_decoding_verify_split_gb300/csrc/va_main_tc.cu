// Split-KV main kernel on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA per SM takes an equal share of the batch's key tiles (128 keys for
// an FP8 cache, 64 for BF16; each (sequence, KV head) item is also charged a
// start-up cost in the split), and for every item in its share packs all G
// query heads x L draft tokens (<= 64 rows) into one MMA tile, so each KV page
// is read from HBM once per KV head (sglang PR 30105 digest, "Implementation
// breakdown" item 2; sglang PR 34517 digest, "Motivation": one KV load shared
// by the heads of a group).
//
// KV pages are TMA-loaded as 128-byte-swizzled boxes (16 tokens x 128 bytes
// of one KV head) into separate K and V rings of 32 KB tiles and fed to the
// tensor cores as they are. The loads carry an L2 evict_first policy: the
// cache is read once per call, and its stream should not push Q, the block
// table or the split partials out of L2.
//
// Launch order: the kernel is a programmatic dependent of the stream's
// previous kernel. It sets up (barriers, TMEM, descriptor prefetch) before
// griddepcontrol.wait and touches global memory only after it; its merge
// kernel is its own programmatic dependent and lets the next call launch, so
// back-to-back calls overlap a merge with the next call's launch and setup.
//  * FP8 E4M3 cache, kind::f8f6f4. Q (bf16) is scaled per row by an exact
//    power of two 2^e and split into two e4m3 terms, Qh = e4m3(Q 2^e) and
//    Ql = e4m3(Q 2^e - Qh); P is split the same way. The two terms are
//    stacked in one M=128 MMA: packed row 16q + i uses A rows 32q + i (hi)
//    and 32q + 16 + i (lo), so the hi and lo results land in lanes i and
//    16 + i of the same TMEM lane quadrant; two 16-lane TMEM loads hand each
//    softmax thread both terms of its own keys, which it adds.
//    Q K^T and P V take their A operands (Q, P) from TMEM: Q is staged there
//    by the softmax warps, P written there beside the one S tile, which is
//    free again once the softmax has loaded it. The shared memory this
//    leaves to the rings holds 4 K + 3 V slots. The variant kernel, whose
//    soft cap can make the softmax the bottleneck, keeps Q in shared memory
//    and two S tiles, each P written over its S (3 K + 3 V). K and V are
//    never dequantised.
//  * BF16 cache, kind::f16, M=64 (packed row 16q + i in lane 32q + i); P goes
//    through four smem buffers; rings 3 K + 2 V.
// V is the MN-major B operand of O += P V. The k/v descales fold into the
// logit scale and the output scale.
//
// Roles (416 threads):
//  warps 0,2,3 TMA producers: warp 0 streams K tiles into the K ring (freed
//              once Q K^T has read them), warps 2 and 3 alternate on V tiles
//              (V ring, freed after P V). Block-table walk with 32 page ids
//              per lane load, read before waiting for the ring slot; one
//              2 KB box per lane.
//  warp 1      TMEM owner; one thread issues Q K^T into the S buffer(s).
//  warp 12     one thread issues P V into O.
//  warps 4-11  softmax, two warps per TMEM lane quadrant q = w % 4 (both on
//              the same SMSP). Warp half kh = (w - 4) / 4 takes half of each
//              tile's keys and O columns [128 kh, 128 kh + 128); lane bit 4
//              splits those again. The two warps of a quadrant combine row
//              maxima and sums through shared memory around a per-quadrant
//              named barrier. They also stage Q (the next item's during the
//              current item's last tile) and write the epilogue.
// Online softmax in log2 units keeps a per-row reference m_ref and computes
// P = 2^(s - m_ref + 6) <= 2^8.8; m_ref moves (and O, l are rescaled in
// TMEM) only when a tile's max exceeds it by more than 2.8, and a row's first
// m_ref sits 4 above its first tile's max, so rescales are rare. The tile
// max is taken over the raw dot products and the (positive) row scale
// applied inside the FMA of P's exponent. The VAR instantiation adds the
// generic attention's variants (sliding
// window, logit soft cap, sinks). Waits are bounded in time and warp-uniform:
// on a timeout the kernel sets the workspace status word, stops issuing
// work, drains and frees its TMEM. The epilogue writes split partials as
// fp32 with 32-byte stores (whole L2 sectors), each thread of a hi/lo lane
// pair summing and writing half of every 32-column chunk. A batch of at most
// 64 sequences keeps its lengths in shared memory for the piece walk.
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "va_fp8.cuh"
#include "va_ptx.cuh"
#include "va_split.cuh"

namespace va {
namespace {

using namespace ptx;

template <bool FP8, bool VAR, bool QTM>
struct Cfg {
  static constexpr int kT = FP8 ? kTcTileKeysFp8 : kTcTileKeysBf16;  // keys per tile: 128 / 64
  static constexpr int kPagesPerTile = kT / kPageSize;
  static constexpr int kKpt = kT / 4;                      // keys per softmax thread per tile
  // FP8 has two TMEM layouts. QTM (the plain kernel on batches of many
  // tiles per CTA) takes Q and P from TMEM (one S tile, two P tiles of their
  // own) and spends the shared memory on a fourth K ring slot. Otherwise Q
  // stays in shared memory with two S tiles, P written over its S tile: with
  // one S tile every tile's Q K^T waits on the softmax's load of the
  // previous S, which a CTA of few tiles pays as latency, and which a soft
  // cap (the softmax then the bottleneck, its ALU work slowing the MMA issue
  // on the same sub-partitions) pays per tile (soft cap 30 on
  // long_context_fp8: 146.3 us against 137.0 us with two S tiles).
  static_assert(FP8 || !QTM, "Q in TMEM is an FP8 layout");
  static_assert(!(VAR && QTM), "the variant kernel keeps Q in shared memory");
  static constexpr bool kQInTmem = QTM;
  static constexpr bool kPOverS = FP8 && !QTM;
  static constexpr int kSBufs = FP8 ? (kQInTmem ? 1 : 2) : 4;  // S tiles in TMEM
  static constexpr int kPBufs = FP8 ? 2 : 4;               // P buffers: TMEM (fp8) / smem (bf16)
  static constexpr int kEsize = FP8 ? 1 : 2;               // bytes per KV element
  static constexpr int kChunks = kHeadDim * kEsize / 128;  // 128-byte d chunks (2 or 4)
  static constexpr int kRegion = kT * 128;                 // one d chunk of a K or V tile
  static constexpr int kTensorBytes = kChunks * kRegion;   // a K or V tile: 16 KB / 32 KB
  // Separate K and V rings of 32 KB tiles (a K slot is free again once Q K^T
  // has read it, a V slot only after P V). A slot turns over in about DRAM
  // latency + hold + producer reaction (~3500 + 1500 + 500 cycles at full HBM
  // load), so the tile rate is slots / that. FP8 with Q in TMEM has room for
  // 4 K + 3 V slots (224 KB): with one S tile, Q K^T of a tile waits for the
  // softmax to load the previous S, which lengthens a K slot's hold
  // (measured: 4 K + 3 V beats 3 K + 4 V by 1.8 us on a 128 us call); with
  // Q in shared memory, 3 K + 3 V (192 KB). BF16 keeps Q and its P buffers in
  // shared memory and has room for 3 K + 2 V (160 KB).
  static constexpr bool kPInTmem = FP8;
  static constexpr int kKSlots = kQInTmem ? 4 : 3;
  static constexpr int kVSlots = FP8 ? 3 : 2;
  static constexpr int kRingBytes = (kKSlots + kVSlots) * 32768;
  // Producer warps: one streams K, two alternate on V's tiles. A producer's
  // wait for a slot relies on its own previous wait (kVProducers tiles back)
  // to keep that slot's empty barrier within one phase of the wanted
  // completion, which holds while the producers of a ring <= its slots.
  static constexpr int kVProducers = 2;
  static_assert(kVProducers <= kVSlots, "V producers exceed the V ring");
  static constexpr int kPageBytes = kChunks * 2048;        // one page of one tensor
  static constexpr int kM = FP8 ? 128 : 64;                // MMA rows
  static constexpr int kQRegion = kM * 128;                // one 128-byte d chunk of Q
  static constexpr int kPRowBytes = kT * kEsize;           // 128 bytes
  static constexpr int kPSbo = 8 * kPRowBytes;             // 8-row group stride, no swizzle (smem P)
  static_assert(kPSbo % 128 == 0, "P core-matrix group stride");
  static constexpr int kPBuf = kM * kPRowBytes;            // 16 KB (fp8) / 8 KB (bf16)
  static constexpr int kQkSteps = 4 * kChunks;             // K-steps of 32 bytes over d
  static constexpr int kPvSteps = kT * kEsize / 32;        // K-steps of 32 bytes over keys
  static constexpr int kKeysPerPvStep = 32 / kEsize;
  static constexpr uint32_t kFmt = FP8 ? 0u : 1u;          // e4m3 / bf16
  static constexpr uint32_t kIdQK = instr_desc(kFmt, kFmt, false, kT, kM);
  static constexpr uint32_t kIdPV = instr_desc(kFmt, kFmt, true, kHeadDim, kM);
  static_assert(kTensorBytes == 32768, "ring slot size");
  // shared memory: rings | Q (smem Q only) | P buffers (smem P only) | row
  // exchange | barriers
  static constexpr int kOffQ = kRingBytes;
  static constexpr int kOffP = kOffQ + (kQInTmem ? 0 : 32768);
  static constexpr int kOffX = kOffP + (kPInTmem ? 0 : 32768);  // [2 parity][2 kh][64 rows] floats
  static constexpr int kOffBar = kOffX + 1024;
  static constexpr int kOffSeqs = kOffBar + 1024;  // the batch's lengths (SeqMeta, kSeqCache)
  static constexpr int kSmemBytes = kOffSeqs + 16 * kSeqCache;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kChunks * kQRegion == 32768, "Q size");
  static_assert(kPInTmem || kPBufs * kPBuf == 32768, "P buffers");
  static_assert(kSBufs * kT == (kQInTmem ? 128 : 256), "S buffers");
  static_assert(!kPOverS || kSBufs == kPBufs, "a P over its S tile shares that tile's index and barriers");
  static_assert(!kQInTmem || kPInTmem, "the TMEM layout below");
  static_assert(kPagesPerTile * kChunks <= 32, "one TMA box per lane");
};

constexpr int kMaxSBufs = 4;
constexpr int kMaxPBufs = 4;
constexpr int kThreads = 416;  // 13 warps
constexpr int kSoftmaxThreads = 256;

// TMEM columns. O [0, 256), then BF16: four 64-column S tiles; FP8 with Q
// in shared memory: two 128-column S tiles, each P (32 columns) written over
// its S; FP8 with Q in TMEM: one 128-column S tile, two P tiles of 32 columns
// (128 keys of e4m3, hi row in lane 32q + i, lo row in lane 32q + 16 + i, as
// S) and the Q A operand (64 columns: 256 e4m3 bytes of each hi and lo row).
constexpr uint32_t kColO = 0;    // 256 fp32 columns
constexpr uint32_t kColS = 256;
constexpr uint32_t kColP = 384;  // FP8, Q in TMEM
constexpr uint32_t kColQ = 448;  // FP8, Q in TMEM
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPShift = 6.f;      // P = 2^(s - m_ref + kPShift)
constexpr float kHeadroom = 1.f;    // m_ref = tile max + kHeadroom when it moves
constexpr float kHeadroomFirst = 4.f;  // ... and + kHeadroomFirst for a row's first reference
constexpr float kOvershoot = 2.8f;  // move only if the tile max > m_ref + kOvershoot (P <= 2^8.8 < 448)


constexpr int kMaxSlots = 5;
// Barrier slots (8 bytes each) after kOffBar.
enum : int {
  kBarFullK = 0,
  kBarEmptyK = kBarFullK + kMaxSlots,
  kBarFullV = kBarEmptyK + kMaxSlots,
  kBarEmptyV = kBarFullV + kMaxSlots,
  kBarSFull = kBarEmptyV + kMaxSlots,
  kBarSFree = kBarSFull + kMaxSBufs,
  kBarPFull = kBarSFree + kMaxSBufs,
  kBarPFree = kBarPFull + kMaxPBufs,
  kBarQFull = kBarPFree + kMaxPBufs,
  kBarQFree,
  kBarOFull,
  kBarOFree,
  kBarDrain,
  kNumBars
};
static_assert(8 * kNumBars + 16 + 34 * 8 + 4 * 2 * kMaxSlots <= 1024, "barrier area");

template <bool FP8>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (FP8)
    mma_f8f6f4(d, a, b, idesc, acc);
  else
    mma_f16(d, a, b, idesc, acc);
}

// VAR: compiled with the sliding-window / soft-cap / sink code (the plain path
// is compiled without it). QTM: the FP8 layout with Q and P in TMEM (Cfg).
template <bool FP8, bool VAR, bool QTM>
__global__ void __launch_bounds__(kThreads, 1)
    va_main_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<FP8, VAR, QTM>;
  constexpr int kT = C::kT;
  constexpr int kSBufs = C::kSBufs;
  constexpr int kPBufs = C::kPBufs;
  constexpr int kPagesPerTile = C::kPagesPerTile;
  constexpr int kKpt = C::kKpt;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffBar + 8 * kNumBars + 4);
  long long* scratch = reinterpret_cast<long long*>(sm + C::kOffBar + 8 * kNumBars + 16);  // 32 slots
  long long* s_ts = scratch + 32;
  int* s_j = reinterpret_cast<int*>(scratch + 33);
  // last tile issued into each ring slot: [K slots | V slots], for the drain
  volatile int* slot_tile = reinterpret_cast<volatile int*>(scratch + 34);
  float* xch = reinterpret_cast<float*>(sm + C::kOffX);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  const uint32_t sbase = smem_addr(sm);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  // The merge kernel is a programmatic dependent: let it be scheduled now; it
  // waits for this grid's completion before reading the workspace.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- setup (no global memory: runs while the stream's previous kernel ends) ---
  constexpr uint32_t kSwWarps = kSoftmaxThreads / 32;
  if (tid == 0) {
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(bar(kBarFullK + s), 1);
      mbar_init(bar(kBarEmptyK + s), 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) {
      mbar_init(bar(kBarFullV + s), 1);
      mbar_init(bar(kBarEmptyV + s), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), kSwWarps);
    }
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(bar(kBarPFull + i), kSwWarps);
      mbar_init(bar(kBarPFree + i), 1);
    }
    mbar_init(bar(kBarQFull), kSwWarps);
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), kSwWarps);
    mbar_init(bar(kBarDrain), 2);
    *abort_flag = 0;
    for (int s = 0; s < 2 * kMaxSlots; ++s) slot_tile[s] = -1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2 && lane == 0 && p.num_blocks > 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This kernel is itself a programmatic dependent of the stream's previous
  // kernel (which may write Q, the block table or the lengths, and may still
  // read this workspace): nothing global is read or written before its
  // completion.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- work range (all threads) -------------------------------------------------
  long long t0, t1, ts_first = 0;
  int j_first = 0;
  bool seqs_cached = false;
  locate_work<kThreads>(p, c, scratch, s_j, s_ts, &t0, &t1, &j_first, &ts_first,
                        reinterpret_cast<SeqMeta*>(sm + C::kOffSeqs), &seqs_cached);
  const SeqMeta* seqs = seqs_cached ? reinterpret_cast<const SeqMeta*>(sm + C::kOffSeqs) : nullptr;
  if (t0 >= t1) {  // CTA-uniform
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    return;
  }

  if (warp == 0 || warp == 2 || warp == 3) {
    // ======================= TMA producers ======================================
    // Warp 0 streams the K tiles, warps 2 and 3 the V tiles of even and odd
    // tiles: one warp alone cannot issue the 2 KB page boxes fast enough to
    // keep HBM busy. Within a warp the lanes issue a tile's boxes in parallel.
    const bool is_k = warp == 0;
    const int nprod = is_k ? 1 : C::kVProducers;
    const int prod = is_k ? 0 : warp - 2;
    const int nslots = is_k ? C::kKSlots : C::kVSlots;
    const int bar_full = is_k ? kBarFullK : kBarFullV;
    const int bar_empty = is_k ? kBarEmptyK : kBarEmptyV;
    const uint32_t ring = sbase + (is_k ? 0u : (uint32_t)(C::kKSlots * C::kTensorBytes));
    const void* tmap = is_k ? (const void*)&tm_k : (const void*)&tm_v;
    volatile int* ring_tile = slot_tile + (is_k ? 0 : kMaxSlots);
    constexpr int kBoxes = kPagesPerTile * C::kChunks;  // boxes per tile
    static_assert(kBoxes <= 32, "one box per lane");
    const uint64_t kv_policy = l2_evict_first_policy();  // K and V are read once
    int it = 0;
    int j = j_first;
    long long ts = ts_first;
    Piece pc;
    bool ok = true;
    while (ok && next_piece(p, t0, t1, j, ts, pc, seqs)) {
      const int npages = (pc.S + kPageSize - 1) / kPageSize;
      // pages wholly before the window are never loaded (a sliding-window
      // page table need not map them); the softmax zeroes their V rows
      const int pg_first = VAR ? first_key(p, pc.S, pc.L) / kPageSize : 0;
      const int* bt_row = p.block_table + (int64_t)pc.b * p.bt_s0;
      int win = -1;       // first page index cached in the lanes
      int my_page = -1;   // page id of page (win + lane)
      for (int lt = pc.lt0; lt < pc.lt1 && ok; ++lt, ++it) {
        if (it % nprod != prod) continue;
        const int s = it % nslots;
        // page ids first (a block-table load every 32 pages), so that their
        // latency overlaps the wait for the ring slot
        const int pg0 = lt * kPagesPerTile;
        if (win < 0 || pg0 + kPagesPerTile > win + 32) {
          win = pg0;
          const int pg = win + lane;
          my_page = pg < npages ? bt_row[(int64_t)pg * p.bt_s1] : -1;
          if (lane == 0 && win + 32 < npages)  // the next window's entries
            asm volatile("prefetch.global.L2 [%0];" ::"l"(bt_row + (int64_t)(win + 32) * p.bt_s1));
        }
        uint32_t nvalid = 0;
        int ids[kPagesPerTile];
#pragma unroll
        for (int i = 0; i < kPagesPerTile; ++i) {
          ids[i] = __shfl_sync(0xffffffffu, my_page, pg0 + i - win);
          const bool v = (pg0 + i) < npages && (pg0 + i) >= pg_first &&
                         (unsigned)ids[i] < (unsigned)p.num_blocks;
          ids[i] = v ? ids[i] : -1;
          nvalid += v ? 1u : 0u;
        }
        const bool got = __all_sync(
            0xffffffffu, mbar_wait(bar(bar_empty + s), ((it / nslots) & 1) ^ 1, abort_flag, p.wait_limit_ns));
        if (!got) {  // warp-uniform
          if (lane == 0) fail(p, abort_flag, 1);
          ok = false;
          break;
        }
        const uint32_t dst = ring + s * C::kTensorBytes;
        if (lane == 0) {
          ring_tile[s] = it;
          mbar_arrive_expect_tx(bar(bar_full + s), nvalid * (uint32_t)C::kPageBytes);
        }
        __syncwarp();
        if (lane < kBoxes) {  // lane -> (page, 128-byte d chunk)
          const int i = lane / C::kChunks, ch = lane % C::kChunks;
          int id = ids[0];
#pragma unroll
          for (int u = 1; u < kPagesPerTile; ++u)
            if (i == u) id = ids[u];
          if (id >= 0)
            tma_load_4d_hint(dst + ch * C::kRegion + i * 2048, tmap, ch * (128 / C::kEsize), pc.kvh, 0, id,
                             bar(bar_full + s), kv_policy);
        }
        __syncwarp();
      }
    }
    // Copies still in flight land before the CTA goes away, also when another
    // role gave up (then nobody consumes them). This producer's tiles that may
    // be in flight are among the last nslots + nprod - 1 tiles it walked: its
    // last issued tile z is at most nprod tiles back, and a tile is issued
    // only once the tile nslots before it in the ring was consumed.
    if (lane == 0) {
      for (int k = (it > nslots + nprod - 1 ? it - nslots - nprod + 1 : 0); k < it; ++k) {
        if (k % nprod != prod) continue;
        drain_ring_tile(bar(bar_full + k % nslots), k, nslots, ring_tile + k % nslots, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 12) {
    // ======================= MMA issuers ==========================================
    // Warp 1 issues Q K^T into the S buffers, warp 12 issues P V into O: the
    // two write different TMEM columns, and splitting them halves the
    // per-tile issue work of one thread (waits, descriptors, commits).
    if (lane == 0) {
      const bool is_qk = warp == 1;
      const uint32_t qbase = sbase + C::kOffQ;
      int it = 0, piece_idx = 0;
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
      while (ok && next_piece(p, t0, t1, j, ts, pc, seqs)) {
        const int first = it;
        const int ntile = pc.lt1 - pc.lt0;
        if (is_qk) {
          if (!wait_or_fail(kBarQFull, piece_idx & 1, 2)) break;
          tc_fence_after();
          for (int i = 0; i < ntile && ok; ++i) {
            const int cur = first + i;
            const int s = cur % C::kKSlots;
            const int b = cur & (kSBufs - 1);
            if (!wait_or_fail(kBarFullK + s, (cur / C::kKSlots) & 1, 32)) break;
            // S buffer b is free once the softmax has read S(cur - kSBufs) or,
            // with P written over it, once P V(cur - kSBufs) has read that P
            if (cur >= kSBufs &&
                !wait_or_fail(C::kPOverS ? kBarPFree + b : kBarSFree + b, ((cur - kSBufs) / kSBufs) & 1, 64))
              break;
            tc_fence_after();
            const uint32_t kst = sbase + s * C::kTensorBytes;
#pragma unroll
            for (int k = 0; k < C::kQkSteps; ++k) {
              const uint32_t koff = (uint32_t)((k >> 2) * C::kRegion + (k & 3) * 32);
              const uint64_t bdesc = smem_desc(kst + koff, 16, 1024, kLayoutSw128);
              if constexpr (C::kQInTmem) {
                // Q's d bytes [32 k, +32) are columns [8 k, +8) of its TMEM rows
                mma_f8f6f4_ta(tmem + kColS + b * kT, tmem + kColQ + 8 * k, bdesc, C::kIdQK, k ? 1u : 0u);
              } else {
                const uint32_t qoff = (uint32_t)((k >> 2) * C::kQRegion + (k & 3) * 32);
                const uint64_t a = smem_desc(qbase + qoff, 16, 1024, kLayoutSw128);
                mma<FP8>(tmem + kColS + b * kT, a, bdesc, C::kIdQK, k ? 1u : 0u);
              }
            }
            mma_commit(bar(kBarSFull + b));
            mma_commit(bar(kBarEmptyK + s));
            if (i == ntile - 1) mma_commit(bar(kBarQFree));
          }
        } else {
          for (int i = 0; i < ntile && ok; ++i) {
            const int x = first + i;
            const int pb = x & (kPBufs - 1);
            const int s = x % C::kVSlots;
            if (!wait_or_fail(kBarPFull + pb, (x / kPBufs) & 1, 4)) break;
            if (!wait_or_fail(kBarFullV + s, (x / C::kVSlots) & 1, 8)) break;
            if (i == 0 && piece_idx > 0 && !wait_or_fail(kBarOFree, (piece_idx - 1) & 1, 16)) break;
            tc_fence_after();
            const uint32_t vst = sbase + (C::kKSlots + s) * C::kTensorBytes;
            const uint32_t pbuf = sbase + C::kOffP + pb * C::kPBuf;
#pragma unroll
            for (int kk = 0; kk < C::kPvSteps; ++kk) {
              const uint64_t bdesc = smem_desc(vst + kk * (C::kKeysPerPvStep / 8) * 1024, C::kRegion,
                                               1024, kLayoutSw128);
              const uint32_t acc = (i == 0 && kk == 0) ? 0u : 1u;
              if constexpr (C::kPInTmem) {
                // P(x) sits in P tile pb (or over S buffer pb), 8 columns per K-step
                const uint32_t pcol = C::kPOverS ? kColS + pb * kT : kColP + pb * (kT / 4);
                mma_f8f6f4_ta(tmem + kColO, tmem + pcol + 8 * kk, bdesc, C::kIdPV, acc);
              } else {
                const uint64_t a = smem_desc(pbuf + kk * 256, 128, C::kPSbo, kLayoutNone);
                mma<FP8>(tmem + kColO, a, bdesc, C::kIdPV, acc);
              }
            }
            mma_commit(bar(kBarPFree + pb));
            mma_commit(bar(kBarEmptyV + s));
            if (i == ntile - 1) mma_commit(bar(kBarOFull));
          }
        }
        it = first + ntile;
        ++piece_idx;
      }
      // every tensor-core operation of both issuers has finished before TMEM is freed
      mma_commit(bar(kBarDrain));
      mbar_wait_drain(bar(kBarDrain), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ======================= softmax / epilogue ===================================
    const int q = warp & 3;              // TMEM lane quadrant
    const int kh = (warp - 4) >> 2;      // which half of the keys / O columns
    const int sub = lane >> 4;           // which quarter within that half
    const int rl = lane & 15;
    const int r = 16 * q + rl;           // packed row
    const int qtr = 2 * kh + sub;        // key quarter 0..3 of a tile
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float kd = p.k_descale ? *p.k_descale : 1.0f;
    const float vd = p.v_descale ? *p.v_descale : 1.0f;
    // The logit scale is kept positive (the softmax takes the max of the raw
    // dot products and applies the scale after): a negative scale negates Q
    // as it is staged, and a zero one becomes a tiny positive one (logits
    // ~1e-30 s instead of 0).
    const float cscale_signed = p.scale_log2 * kd;
    const float cscale = fmaxf(fabsf(cscale_signed), 1e-30f);
    const bool q_neg = cscale_signed < 0.f;
    const int G = p.group;
    unsigned char* qs = sm + C::kOffQ;
    int it = 0, piece_idx = 0;
    int j = j_first;
    long long ts = ts_first;
    Piece pc;
    bool ok = true;
    // Every lane waits; the outcome is made warp-uniform so that a timeout can
    // never split the warp in front of a .sync.aligned tcgen05 instruction.
    // After a failure the warp keeps walking the same pieces and tiles with
    // all waits and work skipped ("dry"), so both warps of a quadrant still
    // meet at every exchange barrier.
    auto wait_or_fail = [&](int b, uint32_t par, int code) {
      if (!ok) return false;
      const bool got = __all_sync(0xffffffffu, mbar_wait(bar(b), par, abort_flag, p.wait_limit_ns));
      if (!got) {
        if (lane == 0) fail(p, abort_flag, code);
        ok = false;
      }
      return ok;
    };
    // Row-wide combine of a per-thread value: lanes t and t^16 share a row in
    // this warp, the partner warp of the quadrant holds the other half. Values
    // go through shared memory (double-buffered by round parity) around the
    // quadrant's named barrier (ids 1..4, 64 threads). Both warps call this the
    // same number of times, failed or not, so the barrier never strands one.
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
    // Q tile of piece pq (the qidx-th piece of this CTA) into the swizzled
    // K-major A operand, after Q K^T of the previous piece has read the old
    // one; this thread: d [64 qtr, +64). Returns the row's logit scale.
    auto stage_q = [&](const Piece& pq, int qidx) -> float {
      if (qidx > 0) wait_or_fail(kBarQFree, (qidx - 1) & 1, 128);
      const bool row_ok = r < pq.R;
      const int tq = row_ok ? r / G : 0;
      const int gq = row_ok ? r - tq * G : 0;
      float rs = 0.f;
      {
        uint4 raw[8];  // 64 bf16
        const uint16_t* src = p.q + (int64_t)(pq.q0 + tq) * p.q_s0 + (int64_t)(pq.kvh * G + gq) * p.q_s1 + 64 * qtr;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          raw[i] = (ok && row_ok) ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0, 0, 0, 0);
        if constexpr (FP8) {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              amax = fmaxf(amax, fabsf(__uint_as_float(w4[k] << 16)));
              amax = fmaxf(amax, fabsf(__uint_as_float(w4[k] & 0xFFFF0000u)));
            }
          }
          amax = exchange(amax, true);
          int e = 0;
          if (amax > 0.f && amax < INFINITY) {
            const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
            e = 7 - E;
            e = e < -120 ? -120 : (e > 120 ? 120 : e);
          }
          const float up = __uint_as_float((uint32_t)(e + 127) << 23) * (q_neg ? -1.f : 1.f);
          const float down = __uint_as_float((uint32_t)(127 - e) << 23);
          rs = cscale * down;  // rows past R stage zeros: their logits are 0
          // d [64 qtr, +64) of row 16q + rl: 16 words of each term, four per
          // 16-byte piece cc (raw[2 cc], raw[2 cc + 1])
          auto split_piece = [&](int cc, uint32_t* hw, uint32_t* lw) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 a = raw[2 * cc + (k >> 1)];
              const uint32_t wa = (k & 1) ? a.z : a.x;
              const uint32_t wb = (k & 1) ? a.w : a.y;
              const float x0 = __uint_as_float(wa << 16) * up, x1 = __uint_as_float(wa & 0xFFFF0000u) * up;
              const float x2 = __uint_as_float(wb << 16) * up, x3 = __uint_as_float(wb & 0xFFFF0000u) * up;
              const uint32_t h01 = pack_fp8x2(x0, x1), h23 = pack_fp8x2(x2, x3);
              const float2 f01 = unpack_fp8x2(h01), f23 = unpack_fp8x2(h23);
              const uint32_t l01 = pack_fp8x2(x0 - f01.x, x1 - f01.y), l23 = pack_fp8x2(x2 - f23.x, x3 - f23.y);
              hw[k] = h01 | (h23 << 16);
              lw[k] = l01 | (l23 << 16);
            }
          };
          if (ok) {
            if constexpr (C::kQInTmem) {
              // the A operand's columns [16 qtr, +16) of lane 32q + rl (hi) and
              // lane 32q + 16 + rl (lo): per half two 16-lane stores, threads
              // 16-31 (sub 1) at +16
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t hw[8], lw[8];
                split_piece(2 * h, hw, lw);
                split_piece(2 * h + 1, hw + 4, lw + 4);
                tmem_st_16x32bx2_x8<16>(tmem + lane_base + kColQ + 32 * kh + 8 * h, hw);
                tmem_st_16x32bx2_x8<16>(tmem + lane_base + (16u << 16) + kColQ + 32 * kh + 8 * h, lw);
              }
              tmem_wait_st();
            } else {
              // region kh, 16-byte pieces 4 sub .. 4 sub + 3 of A rows 32q + rl
              // (hi) and 32q + 16 + rl (lo)
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                uint32_t hw[4], lw[4];
                split_piece(cc, hw, lw);
                const int swz = ((4 * sub + cc) ^ (rl & 7)) << 4;
                const int ahi = 32 * q + rl, alo = ahi + 16;
                *reinterpret_cast<uint4*>(qs + kh * C::kQRegion + ahi * 128 + swz) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(qs + kh * C::kQRegion + alo * 128 + swz) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
              }
            }
          }
        } else {
          rs = cscale;  // rows past R stage zeros: their logits are 0
          // d [64 qtr, +64) = one whole 128-byte region (qtr), eight 16-byte pieces
          if (ok) {
            const uint32_t flip = q_neg ? 0x80008000u : 0u;  // bf16 sign bits
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int off = qtr * C::kQRegion + r * 128 + ((i ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(qs + off) =
                  make_uint4(raw[i].x ^ flip, raw[i].y ^ flip, raw[i].z ^ flip, raw[i].w ^ flip);
            }
          }
        }
      }
      if (ok) {
        if constexpr (C::kQInTmem)
          tc_fence_before();
        else
          fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQFull));
      }
      return rs;
    };
    // The first lines of the next piece's Q rows, pulled into L2 early.
    auto prefetch_q = [&](const Piece& pq) {
      if (r < pq.R) {
        const int tq = r / G, gq = r - tq * G;
        const uint16_t* src = p.q + (int64_t)(pq.q0 + tq) * p.q_s0 + (int64_t)(pq.kvh * G + gq) * p.q_s1 + 64 * qtr;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
      }
    };
    float rs_next = 0.f;
    bool staged_next = false;
    while (next_piece(p, t0, t1, j, ts, pc, seqs)) {
      // The next piece's Q is staged at the start of this piece's last tile,
      // so its first Q K^T overlaps that tile and this piece's epilogue.
      Piece pn;
      int jn = j;
      long long tsn = ts;
      const bool has_next = next_piece(p, t0, t1, jn, tsn, pn, seqs);
      const float rs = staged_next ? rs_next : stage_q(pc, piece_idx);
      staged_next = false;
      if (has_next) prefetch_q(pn);
      const bool row_ok = r < pc.R;
      const int tq = row_ok ? r / G : 0;
      const int gq = row_ok ? r - tq * G : 0;

      // -- key tiles
      float m_ref = -INFINITY;
      float l = 0.f;
      // last visible key of this row: S - L + t, or for a shard of the
      // sequence's keys E - L + t, never past the shard's own keys
      const int vis_end = min(pc.E - pc.L + tq, pc.S - 1);
      const int mask_from = min(pc.E - pc.L, pc.S - 1);  // tiles past this key hold masked keys
      // first visible key of this row (sliding window), and the largest over rows
      const int vis_lo = VAR && p.window_left >= 0 ? pc.S - pc.L + tq - p.window_left : 0;
      const int vis_lo_max = VAR && p.window_left >= 0 ? pc.S - 1 - p.window_left : 0;
      const int first = it;
      for (int lt = pc.lt0; lt < pc.lt1; ++lt, ++it) {
        const int cur = it;
        const int b = cur & (kSBufs - 1);
        const int pb = cur & (kPBufs - 1);
        if (lt == pc.lt1 - 1 && has_next) {
          rs_next = stage_q(pn, piece_idx + 1);
          staged_next = true;
        }
        float x[kKpt];  // logits of keys [kKpt qtr, +kKpt) of this tile, this row
#pragma unroll
        for (int i = 0; i < kKpt; ++i) x[i] = -INFINITY;
        // x[] holds the raw dot products s (the logit in log2 units is
        // xs * x, xs = the row's scale rs), or with a soft cap c (log2 units)
        // tanh(rs s / c) (then xs = c). xs is applied in the ex2 of P as one
        // FMA, and once to the tile's max (xs > 0 keeps the order), so the
        // scale costs nothing per key and the cap one SFU op per key.
        float rx = 0.f;
        float xs = rs;
        if constexpr (VAR) {
          if (p.softcap_log2 > 0.f) {
            xs = p.softcap_log2;
            rx = rs / xs;
          }
        }
        if (wait_or_fail(kBarSFull + b, (cur / kSBufs) & 1, 256)) {
          tc_fence_after();
          if constexpr (FP8) {
            // the hi and lo partials of row 16q + rl, keys [64 kh + 32 sub,
            // +32): two 16-lane loads (hi rows in lanes 32q.., lo rows in
            // lanes 32q + 16..) whose second halves go to threads 16-31, so
            // every thread gets both terms of its own keys. S buffer b is then
            // free for Q K^T of a later tile, or is overwritten by P(cur) and
            // freed by P V's commit.
            uint32_t vh[32], vl[32];
            tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kColS + b * kT + 64 * kh, vh);
            tmem_ld_16x32bx2_x32<32>(tmem + lane_base + (16u << 16) + kColS + b * kT + 64 * kh, vl);
            tmem_wait_ld();
            tc_fence_before();
            if constexpr (!C::kPOverS) {
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(kBarSFree + b));
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(vh[i]) + __uint_as_float(vl[i]);
          } else {
            uint32_t v[16];
            tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kColS + b * kT + 32 * kh, v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree + b));
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(v[i]);
          }
          if constexpr (VAR) {
            if (p.softcap_log2 > 0.f) {
              // soft cap c tanh(logit / c), before masking, kept as the tanh
              // (see xs). tanh.approx's relative error of ~2^-11 moves a
              // logit l by at most |l| 2^-11 log2 units (0.5 % of a key's
              // weight at l = 10).
#pragma unroll
              for (int i = 0; i < kKpt; ++i) x[i] = tanh_approx(x[i] * rx);
            }
          }
          const int key0 = lt * kT + kKpt * qtr;
          if (lt * kT + kT - 1 > mask_from) {  // tail tile: causal mask
#pragma unroll
            for (int i = 0; i < kKpt; ++i)
              if (key0 + i > vis_end) x[i] = -INFINITY;
          }
          if constexpr (VAR) {
            if (lt * kT < vis_lo_max) {  // a window's first tiles: keys before the row's window
#pragma unroll
              for (int i = 0; i < kKpt; ++i)
                if (key0 + i < vis_lo) x[i] = -INFINITY;
            }
          }
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < kKpt; i += 2) tmax = fmax3(tmax, x[i], x[i + 1]);
        tmax = exchange(tmax * xs, true);  // log2 units (xs > 0 keeps the order)
        if (!ok) continue;

        // P buffer pb was last read by PV(cur - kPBufs). (A P over S(cur):
        // Q K^T(cur) already waited for that.)
        if (!C::kPOverS && cur >= kPBufs &&
            !wait_or_fail(kBarPFree + pb, ((cur - kPBufs) / kPBufs) & 1, 512))
          continue;

        const bool need = tmax > m_ref + kOvershoot;
        // A row's first reference takes more headroom: its running max keeps
        // growing over the next tiles (by ~sd * (sqrt(2 ln n) - sqrt(2 ln T))),
        // and every later move waits for P V of the previous tile.
        const float m_new = need ? tmax + (m_ref == -INFINITY ? kHeadroomFirst : kHeadroom) : m_ref;
        const bool rescale = need && (m_ref != -INFINITY) && (cur > first);
        const float alpha = rescale ? ex2(m_ref - m_new) : 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds earlier tiles of this piece: wait for PV(cur - 1), then
          // scale this thread's part of the row in TMEM
          const int xp = cur - 1;
          if (!wait_or_fail(kBarPFree + (xp & (kPBufs - 1)), (xp / kPBufs) & 1, 1024)) continue;
          tc_fence_after();
#pragma unroll 1
          for (int k = 0; k < (FP8 ? 4 : 2); ++k) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kColO + 128 * kh + 32 * k;
            if constexpr (FP8) {
              tmem_ld_32x32b_x32(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_32x32b_x32(ta, o);
            } else {
              tmem_ld_16x32bx2_x32<64>(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_16x32bx2_x32<64>(ta, o);
            }
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_ref = m_new;

        // P = 2^(x - m_ref + kPShift) into the K-major no-swizzle A operand
        // a row with no visible key yet (m_ref = -inf) gets P = ex2(-inf) = 0
        const float mref_s = m_ref != -INFINITY ? m_ref - kPShift : INFINITY;
        float ls0 = 0.f, ls1 = 0.f;
        unsigned char* pbuf = sm + C::kOffP + pb * C::kPBuf;
        if constexpr (FP8) {
          uint32_t ph[8], pl[8];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = ex2(fmaf(x[2 * i], xs, -mref_s));
            const float bb = ex2(fmaf(x[2 * i + 1], xs, -mref_s));
            ls0 += a;
            ls1 += bb;
            uint32_t h2, l2;
            split_p(a, bb, h2, l2);
            if (i & 1) {
              ph[i >> 1] |= h2 << 16;
              pl[i >> 1] |= l2 << 16;
            } else {
              ph[i >> 1] = h2;
              pl[i >> 1] = l2;
            }
          }
          // A operand of P V in TMEM, P tile pb or over S(cur) (pb == b
          // then): lane 32q + rl (hi row) and
          // lane 32q + 16 + rl (lo row) take the e4m3 bytes of keys
          // [64 kh, +64) at columns [16 kh, +16). This thread holds keys
          // [32 qtr, +32) of both: two 16-lane stores, its hi bytes into the
          // hi row and its lo bytes into the lo row, threads 16-31 at +8.
          // Over S, the quadrant's other warp read its S columns before the
          // exchange.
          const uint32_t pcol = C::kPOverS ? kColS + pb * kT : kColP + pb * (kT / 4);
          tc_fence_after();
          tmem_st_16x32bx2_x8<8>(tmem + lane_base + pcol + 16 * kh, ph);
          tmem_st_16x32bx2_x8<8>(tmem + lane_base + (16u << 16) + pcol + 16 * kh, pl);
          tmem_wait_st();
        } else {
          uint32_t pw[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float a = ex2(fmaf(x[2 * i], xs, -mref_s));
            const float bb = ex2(fmaf(x[2 * i + 1], xs, -mref_s));
            ls0 += a;
            ls1 += bb;
            pw[i] = pack_bf16x2(a, bb);
          }
          // keys [16 qtr, +16) = 32 bytes = core-matrix columns 2 qtr, 2 qtr + 1 of row r
          unsigned char* base = pbuf + (r >> 3) * C::kPSbo + (2 * qtr) * 128 + (r & 7) * 16;
          *reinterpret_cast<uint4*>(base) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(base + 128) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
        }
        l += ls0 + ls1;
        // V rows no row may see and whose pages may hold anything are zeroed,
        // so that 0 * garbage cannot reach O: past S in the item's last tile
        // (partial page, pages never loaded), and in its first tile the pages
        // wholly before a sliding window (never loaded)
        const int zt0 = (lt == pc.nt - 1 && (pc.S % kT) != 0) ? pc.S - lt * kT : kT;
        int zh1 = 0;
        if constexpr (VAR) {
          const int k_first = first_key(p, pc.S, pc.L);
          if (lt == pc.tb && k_first >= kPageSize) zh1 = (k_first / kPageSize) * kPageSize - lt * kT;
        }
        if (zt0 < kT || zh1 > 0) {
          const int vs = cur % C::kVSlots;
          // FullV(vs) alternates between the tiles that share slot vs, so its
          // parity names tile cur only once the slot's previous tile
          // (cur - kVSlots) has been consumed by P V. The softmax at tile cur
          // only knows P V(cur - kPBufs) done (its P buffer's wait above, or
          // for a P over S the S buffer Q K^T waited for); if that is not
          // enough, wait.
          if constexpr (kPBufs > C::kVSlots) {
            const int xv = cur - C::kVSlots;
            if (xv >= 0 && !wait_or_fail(kBarPFree + (xv & (kPBufs - 1)), (xv / kPBufs) & 1, 2049)) continue;
          }
          if (!wait_or_fail(kBarFullV + vs, (cur / C::kVSlots) & 1, 2048)) continue;
          const int nz = zh1 + (kT - zt0);  // rows [0, zh1) and [zt0, kT)
          unsigned char* vst = sm + (C::kKSlots + vs) * C::kTensorBytes;
          for (int idx = tid - 128; idx < nz * 8 * C::kChunks; idx += kSoftmaxThreads) {
            const int k = idx / (8 * C::kChunks);
            const int row = k < zh1 ? k : zt0 + (k - zh1);
            const int rem = idx % (8 * C::kChunks);
            const int ch = rem >> 3;
            const int piece16 = rem & 7;
            *reinterpret_cast<uint4*>(vst + ch * C::kRegion + row * 128 + piece16 * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        if constexpr (C::kPInTmem) tc_fence_before();  // the P store, before the arrive
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + pb));
      }

      // -- epilogue: the row sum first (it does not depend on O, so the
      // exchange with the quadrant's other warp overlaps the last P V), then O
      float lrow = exchange(l, false);
      wait_or_fail(kBarOFull, piece_idx & 1, 4096);
      tc_fence_after();
      ++piece_idx;
      if (!ok) continue;
      // an attention sink joins the normaliser once per row: here for rows
      // written directly, in the merge for split ones
      if constexpr (VAR) {
        if (p.sinks && pc.direct && row_ok && m_ref != -INFINITY)
          lrow += exp2f(p.sinks[pc.kvh * G + gq] * kLog2e - (m_ref - kPShift));
      }
      const float inv = lrow > 0.f ? vd / lrow : 0.f;
      const int64_t piece = (int64_t)pc.j + c;
      // this row's n (16 or 32) values of O from column col (col % 16 == 0)
      auto emit = [&](const uint32_t* o, int col, auto n_c) {
        constexpr int n = decltype(n_c)::value;
        if (!row_ok) return;
        if (pc.direct) {
          uint16_t* dst = p.out + (int64_t)(pc.q0 + tq) * p.o_s0 + (int64_t)(pc.kvh * G + gq) * p.o_s1 + col;
          uint32_t w[n / 2];
#pragma unroll
          for (int e2 = 0; e2 < n / 2; ++e2)
            w[e2] = pack_bf16x2(__uint_as_float(o[2 * e2]) * inv, __uint_as_float(o[2 * e2 + 1]) * inv);
          if (p.out_v8) {  // whole sectors, as for the partials
#pragma unroll
            for (int v = 0; v < n / 16; ++v) st_global_v8(dst + 16 * v, w + 8 * v);
          } else {
#pragma unroll
            for (int v4 = 0; v4 < n / 8; ++v4)
              reinterpret_cast<uint4*>(dst)[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        } else {
          // 32-byte stores: a warp's store writes whole sectors, half the
          // write requests of 16-byte stores (the workspace is 256-byte
          // aligned and col % 16 == 0)
          float* dst = p.ws_acc + (piece * p.max_rows + r) * kHeadDim + col;
#pragma unroll
          for (int v8 = 0; v8 < n / 8; ++v8) st_global_v8(dst + 8 * v8, o + 8 * v8);
        }
      };
      if constexpr (FP8) {
        // O's hi and lo rows sit 16 lanes apart, as S's do. Per 32-column
        // chunk two 16-lane loads (hi lanes, lo lanes; second halves to
        // threads 16-31) give thread i + 16 sub both terms of row 16q + i at
        // columns [16 sub, 16 sub + 16), which it sums and writes.
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          uint32_t oh[16], ol[16];
          tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kColO + 128 * kh + 32 * k, oh);
          tmem_ld_16x32bx2_x16<16>(tmem + lane_base + (16u << 16) + kColO + 128 * kh + 32 * k, ol);
          tmem_wait_ld();
          uint32_t sum[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) sum[i] = __float_as_uint(__uint_as_float(oh[i]) + __uint_as_float(ol[i]));
          emit(sum, 128 * kh + 32 * k + 16 * sub, std::integral_constant<int, 16>{});
        }
      } else {
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
          uint32_t o[32];
          tmem_ld_16x32bx2_x32<64>(tmem + lane_base + kColO + 128 * kh + 32 * k, o);
          tmem_wait_ld();
          emit(o, 128 * kh + 64 * sub + 32 * k, std::integral_constant<int, 32>{});
        }
      }
      if (row_ok && !pc.direct && kh == 0 && sub == 0) {
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

template <bool FP8, bool VAR, bool QTM>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(va_main_tc_kernel<FP8, VAR, QTM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<FP8, VAR, QTM>::kSmemBytes);
}

cudaError_t prepare_main_tc() {
  cudaError_t e = set_smem<true, false, true>();
  if (e == cudaSuccess) e = set_smem<true, false, false>();
  if (e == cudaSuccess) e = set_smem<false, false, false>();
  if (e == cudaSuccess) e = set_smem<true, true, false>();
  if (e == cudaSuccess) e = set_smem<false, true, false>();
  return e;
}

template <bool FP8, bool VAR, bool QTM>
static cudaError_t launch_one(cudaLaunchConfig_t& cfg, const Params& p, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v) {
  cfg.dynamicSmemBytes = Cfg<FP8, VAR, QTM>::kSmemBytes;
  return cudaLaunchKernelEx(&cfg, va_main_tc_kernel<FP8, VAR, QTM>, p, tm_k, tm_v);
}

cudaError_t launch_main_tc(const Params& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           cudaStream_t stream) {
  const bool var = p.window_left >= 0 || p.softcap_log2 > 0.f || p.sinks != nullptr;
  // a programmatic dependent of the stream's previous kernel: its launch and
  // setup overlap that kernel's tail (it waits before touching memory)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.kv_fp8) {
    if (var) return launch_one<true, true, false>(cfg, p, tm_k, tm_v);
    return p.q_in_tmem ? launch_one<true, false, true>(cfg, p, tm_k, tm_v)
                       : launch_one<true, false, false>(cfg, p, tm_k, tm_v);
  }
  return var ? launch_one<false, true, false>(cfg, p, tm_k, tm_v)
             : launch_one<false, false, false>(cfg, p, tm_k, tm_v);
}

}  // namespace va
