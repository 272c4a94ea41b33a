// Split-KV main kernel on the 5th-generation tensor cores (tcgen05, sm_103a),
// FP8 E4M3 KV cache.
//
// Same decomposition and partial format as the CUDA-core kernel: one CTA per
// SM takes an equal share of the batch's 64-key tiles, and for every
// (sequence, KV head) in its share packs all G query heads x L draft tokens
// (<= 64 rows) into one M=64 tile, so each KV page is read from HBM once per
// KV head (sglang PR 30105 digest, "Implementation breakdown" item 2; sglang
// PR 34517 digest, "Motivation": one KV load shared by the heads of a group).
//
// The FP8 pages stay FP8 all the way into the tensor cores (kind::f8f6f4):
//  * S = Q K^T: Q (bf16) is scaled per row by a power of two 2^e (exact) and
//    split into two e4m3 terms, Qh = e4m3(Q 2^e) and Ql = e4m3(Q 2^e - Qh);
//    both MMAs accumulate into the same fp32 TMEM tile, so the logits carry
//    the product (Qh + Ql) K, about 2^-8 relative to Q, with K exact.
//  * O += P V: P = 2^(s - m_ref + 8) <= 2^8.3 is split the same way into
//    e4m3 hi and lo terms; V is the MN-major B operand read straight from the
//    TMA-staged page.
// The k/v descales fold into the logit scale and the output scale.
//
// Roles (256 threads):
//  warp 0     TMA producer: block-table walk (32 page ids per lane load),
//             two 128-byte-swizzled 2 KB boxes per page for K and for V into
//             a 5-stage ring.
//  warp 1     TMEM owner and MMA issuer (one thread).
//  warps 4-7  softmax: thread (quadrant q, lane t) owns row 16q + (t & 15)
//             and half (t >> 4) of each tile's keys and of O's columns.
// Online softmax in log2 units keeps a per-row reference m_ref; it moves (and
// O, l are rescaled in TMEM) only when a tile's max exceeds it by > 0.3, so
// rescaling is rare. Waits are bounded in time: on a timeout the kernel sets
// the workspace status word, stops issuing work and frees its TMEM.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "va_ptx.cuh"
#include "va_split.cuh"

namespace va {
namespace {

using namespace ptx;

constexpr int kT = kTcTileKeys;  // 64 keys per tile
constexpr int kStages = 5;
constexpr int kThreads = 256;
constexpr int kStageBytes = 32768;  // K: 2 halves x 64 keys x 128 B; V: same
constexpr int kQPart = 16384;       // 2 halves x 64 rows x 128 B
constexpr int kPPart = 4096;        // 64 rows x 64 B, no swizzle
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + 2 * kQPart;
constexpr int kOffBar = kOffP + 4 * kPPart;
constexpr int kSmemBytes = kOffBar + 512 + 1024;

constexpr uint32_t kColO = 0;    // 256 fp32 columns
constexpr uint32_t kColS = 256;  // two 64-column S tiles
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdQK = instr_desc(0, 0, false, kT, 64);     // e4m3 x e4m3, M=64, N=64
constexpr uint32_t kIdPV = instr_desc(0, 0, true, kHeadDim, 64);  // B (V) MN-major, N=256

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Barrier slots (8 bytes each) after kOffBar.
enum : int {
  kBarFullK = 0,
  kBarFullV = kBarFullK + kStages,
  kBarEmpty = kBarFullV + kStages,
  kBarSFull = kBarEmpty + kStages,
  kBarSFree = kBarSFull + 2,
  kBarPFull = kBarSFree + 2,
  kBarPFree = kBarPFull + 2,
  kBarQFull = kBarPFree + 2,
  kBarQFree,
  kBarOFull,
  kBarOFree,
  kBarDrain,
  kNumBars
};

struct Piece {
  int j, b, kvh, S, L, q0, R, nt, lt0, lt1;
  bool direct;
};

// Next (sequence, KV head) item of this CTA's tile range [t0, t1).
__device__ __forceinline__ bool next_piece(const Params& p, long long t0, long long t1, int& j,
                                           long long& ts, Piece& pc) {
  while (j < p.num_work && ts < t1) {
    const int nt = work_tiles(p, j);
    if (nt == 0) {
      ++j;
      continue;
    }
    pc.j = j;
    pc.b = j / p.hkv;
    pc.kvh = j - pc.b * p.hkv;
    pc.S = seq_kv_len(p, pc.b);
    pc.L = seq_q_len(p, pc.b);
    pc.q0 = p.cu_q[pc.b];
    pc.R = p.group * pc.L;
    pc.nt = nt;
    pc.lt0 = (int)((t0 > ts ? t0 : ts) - ts);
    pc.lt1 = (int)((t1 < ts + nt ? t1 : ts + nt) - ts);
    pc.direct = (pc.lt0 == 0 && pc.lt1 == nt);
    ts += nt;
    ++j;
    return true;
  }
  return false;
}

__device__ __forceinline__ void fail(const Params& p, volatile int* abort_flag, int code) {
  *abort_flag = 1;
  if (p.ws_status) atomicOr(p.ws_status, code);
}

__device__ __forceinline__ uint32_t pack_fp8x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float2 unpack_fp8x2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(__half2(h));
}

// p (two fp32 values, p.x first) -> e4m3 hi and lo bytes, via f16x2.
__device__ __forceinline__ void split_p(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const __nv_fp8x2_storage_t h8 = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(h), __NV_SATFINITE, __NV_E4M3);
  const __half2 hh = __half2(__nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3));
  const __half2 r = __hsub2(h, hh);
  const __nv_fp8x2_storage_t l8 = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(r), __NV_SATFINITE, __NV_E4M3);
  hi = (uint32_t)h8;
  lo = (uint32_t)l8;
}

__global__ void __launch_bounds__(kThreads, 1)
    va_main_tc_fp8_kernel(const Params p, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffBar + 8 * kNumBars + 4);
  long long* scratch = reinterpret_cast<long long*>(sm + kOffBar + 8 * kNumBars + 16);  // 32 slots
  long long* s_ts = scratch + 32;
  int* s_j = reinterpret_cast<int*>(scratch + 33);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  const uint32_t sbase = smem_addr(sm);
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  // ---- work range (all threads) -------------------------------------------------
  const long long N = scan_work<kThreads>(p, scratch, c == 0);
  const long long t0 = split_begin(N, c, p.num_splits);
  const long long t1 = split_begin(N, c + 1, p.num_splits);
  if (t0 >= t1) return;
  int j_first;
  long long ts_first;
  find_work<kThreads>(p, t0, scratch, s_j, s_ts, &j_first, &ts_first);

  // ---- setup --------------------------------------------------------------------
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFullK + s), 1);
      mbar_init(bar(kBarFullV + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), 4);
      mbar_init(bar(kBarPFull + i), 4);
      mbar_init(bar(kBarPFree + i), 1);
    }
    mbar_init(bar(kBarQFull), 4);
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), 4);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ======================= TMA producer =======================================
    int it = 0;
    int j = j_first;
    long long ts = ts_first;
    Piece pc;
    bool ok = true;
    while (ok && next_piece(p, t0, t1, j, ts, pc)) {
      const int npages = (pc.S + kPageSize - 1) / kPageSize;
      const int* bt_row = p.block_table + (int64_t)pc.b * p.bt_s0;
      int win = -1;       // first page index cached in the lanes
      int my_page = -1;   // page id of page (win + lane)
      for (int lt = pc.lt0; lt < pc.lt1 && ok; ++lt, ++it) {
        const int s = it % kStages;
        const bool got = __all_sync(
            0xffffffffu, mbar_wait(bar(kBarEmpty + s), ((it / kStages) & 1) ^ 1, abort_flag, kWaitLimitNs));
        if (!got) {  // warp-uniform
          if (lane == 0) fail(p, abort_flag, 1);
          ok = false;
          break;
        }
        const int pg0 = lt * (kT / kPageSize);
        if (win < 0 || pg0 + 3 >= win + 32) {
          win = pg0;
          const int pg = win + lane;
          my_page = pg < npages ? bt_row[(int64_t)pg * p.bt_s1] : -1;
        }
        uint32_t nvalid = 0;
        int ids[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ids[i] = __shfl_sync(0xffffffffu, my_page, pg0 + i - win);
          const bool v = (pg0 + i) < npages && (unsigned)ids[i] < (unsigned)p.num_blocks;
          ids[i] = v ? ids[i] : -1;
          nvalid += v ? 1u : 0u;
        }
        if (lane == 0) {
          const uint32_t kst = sbase + s * kStageBytes;
          const uint32_t vst = kst + kStageBytes / 2;
          mbar_arrive_expect_tx(bar(kBarFullK + s), nvalid * 4096u);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ids[i] < 0) continue;
            tma_load_4d(kst + i * 2048, &tm_k, 0, pc.kvh, 0, ids[i], bar(kBarFullK + s));
            tma_load_4d(kst + 8192 + i * 2048, &tm_k, 128, pc.kvh, 0, ids[i], bar(kBarFullK + s));
          }
          mbar_arrive_expect_tx(bar(kBarFullV + s), nvalid * 4096u);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ids[i] < 0) continue;
            tma_load_4d(vst + i * 2048, &tm_v, 0, pc.kvh, 0, ids[i], bar(kBarFullV + s));
            tma_load_4d(vst + 8192 + i * 2048, &tm_v, 128, pc.kvh, 0, ids[i], bar(kBarFullV + s));
          }
        }
        __syncwarp();
      }
    }
    if (!ok) {
      // let copies already in flight land before the CTA goes away
      for (int k = (it > kStages ? it - kStages : 0); k < it; ++k) {
        const int s = k % kStages;
        mbar_wait(bar(kBarFullK + s), (k / kStages) & 1, abort_flag, 10000000ull);
        mbar_wait(bar(kBarFullV + s), (k / kStages) & 1, abort_flag, 10000000ull);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer ===========================================
    if (lane == 0) {
      const uint32_t qh = sbase + kOffQ, ql = qh + kQPart;
      int it = 0, piece_idx = 0;
      int j = j_first;
      long long ts = ts_first;
      Piece pc;
      bool ok = true;
      auto wait_or_fail = [&](int b, uint32_t par, int code) {
        if (!ok) return false;
        if (!mbar_wait(bar(b), par, abort_flag, kWaitLimitNs)) {
          fail(p, abort_flag, code);
          ok = false;
        }
        return ok;
      };
      while (ok && next_piece(p, t0, t1, j, ts, pc)) {
        const int first = it;
        const int ntile = pc.lt1 - pc.lt0;
        if (!wait_or_fail(kBarQFull, piece_idx & 1, 2)) break;
        tc_fence_after();
        auto issue_pv = [&](int x) {
          const int pb = x & 1;
          const int s = x % kStages;
          if (!wait_or_fail(kBarPFull + pb, (x >> 1) & 1, 4)) return;
          if (!wait_or_fail(kBarFullV + s, (x / kStages) & 1, 8)) return;
          if (x == first && piece_idx > 0 && !wait_or_fail(kBarOFree, (piece_idx - 1) & 1, 16)) return;
          tc_fence_after();
          const uint32_t vst = sbase + s * kStageBytes + kStageBytes / 2;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t pbuf = sbase + kOffP + (pb * 2 + part) * kPPart;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint64_t a = smem_desc(pbuf + kk * 256, 128, 512, kLayoutNone);
              const uint64_t bdesc = smem_desc(vst + kk * 4096, 8192, 1024, kLayoutSw128);
              mma_f8f6f4(tmem + kColO, a, bdesc, kIdPV, (x == first && part == 0 && kk == 0) ? 0u : 1u);
            }
          }
          mma_commit(bar(kBarPFree + pb));
          mma_commit(bar(kBarEmpty + s));
          if (x == first + ntile - 1) mma_commit(bar(kBarOFull));
        };
        for (int i = 0; i < ntile && ok; ++i) {
          const int cur = first + i;
          const int s = cur % kStages;
          const int b = cur & 1;
          if (!wait_or_fail(kBarFullK + s, (cur / kStages) & 1, 32)) break;
          if (cur >= 2 && !wait_or_fail(kBarSFree + b, ((cur - 2) >> 1) & 1, 64)) break;
          tc_fence_after();
          const uint32_t kst = sbase + s * kStageBytes;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t qb = part ? ql : qh;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t off = (uint32_t)((k >> 2) * 8192 + (k & 3) * 32);
              const uint64_t a = smem_desc(qb + off, 16, 1024, kLayoutSw128);
              const uint64_t bdesc = smem_desc(kst + off, 16, 1024, kLayoutSw128);
              mma_f8f6f4(tmem + kColS + b * kT, a, bdesc, kIdQK, (part | k) ? 1u : 0u);
            }
          }
          mma_commit(bar(kBarSFull + b));
          if (i == ntile - 1) mma_commit(bar(kBarQFree));
          if (i > 0) issue_pv(cur - 1);
        }
        if (ok) issue_pv(first + ntile - 1);
        it = first + ntile;
        ++piece_idx;
      }
      // make sure every tensor-core operation has finished before TMEM is freed
      mma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, abort_flag, 100000000ull);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ======================= softmax / epilogue ===================================
    const int q = warp & 3;
    const int hf = lane >> 4;
    const int r = 16 * q + (lane & 15);
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float kd = p.k_descale ? *p.k_descale : 1.0f;
    const float vd = p.v_descale ? *p.v_descale : 1.0f;
    const float cscale = p.scale_log2 * kd;
    const int G = p.group;
    unsigned char* qhi = sm + kOffQ;
    unsigned char* qlo = qhi + kQPart;
    int it = 0, piece_idx = 0;
    int j = j_first;
    long long ts = ts_first;
    Piece pc;
    bool ok = true;
    // Every lane waits; the outcome is made warp-uniform so that a timeout can
    // never split the warp in front of a .sync.aligned tcgen05 instruction.
    auto wait_or_fail = [&](int b, uint32_t par, int code) {
      if (!ok) return false;
      const bool got = __all_sync(0xffffffffu, mbar_wait(bar(b), par, abort_flag, kWaitLimitNs));
      if (!got) {
        if (lane == 0) fail(p, abort_flag, code);
        ok = false;
      }
      return ok;
    };
    while (ok && next_piece(p, t0, t1, j, ts, pc)) {
      // -- Q tile: per-row power-of-two scale, e4m3 hi/lo split, swizzled store
      if (piece_idx > 0 && !wait_or_fail(kBarQFree, (piece_idx - 1) & 1, 128)) break;
      const bool row_ok = r < pc.R;
      const int tq = row_ok ? r / G : 0;
      const int gq = row_ok ? r - tq * G : 0;
      float rs = 0.f;
      {
        uint4 raw[16];
        const uint16_t* src = p.q + (int64_t)(pc.q0 + tq) * p.q_s0 + (int64_t)(pc.kvh * G + gq) * p.q_s1 + 128 * hf;
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          raw[i] = row_ok ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0, 0, 0, 0);
          const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[k] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[k] & 0xFFFF0000u)));
          }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
        int e = 0;
        if (amax > 0.f && amax < INFINITY) {
          const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
          e = 7 - E;
          e = e < -120 ? -120 : (e > 120 ? 120 : e);
        }
        const float up = __uint_as_float((uint32_t)(e + 127) << 23);
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);
        rs = row_ok ? cscale * down : 0.f;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {  // 16 d values -> 16 bytes hi, 16 bytes lo
          uint32_t hw[4], lw[4];
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
          const int off = hf * 8192 + r * 128 + ((cc ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(qhi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(qlo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQFull));

      // -- key tiles
      float m_ref = -INFINITY;
      float l = 0.f;
      const int vis_end = pc.S - pc.L + tq;  // last visible key of this row
      const int first = it;
      for (int lt = pc.lt0; lt < pc.lt1; ++lt, ++it) {
        const int cur = it;
        const int b = cur & 1;
        const int s = cur % kStages;
        if (!wait_or_fail(kBarSFull + b, (cur >> 1) & 1, 256)) break;
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kColS + b * kT, sr);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSFree + b));

        float x[32];
        const int key0 = lt * kT + 32 * hf;
        const bool tail = lt * kT + kT - 1 > pc.S - pc.L;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(sr[i]) * rs;
          if (tail && key0 + i > vis_end) x[i] = -INFINITY;
        }
        float tmax = x[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) tmax = fmaxf(tmax, x[i]);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));

        // P buffer b was last read by PV(cur - 2)
        if (cur >= 2 && !wait_or_fail(kBarPFree + b, ((cur - 2) >> 1) & 1, 512)) break;

        const bool need = tmax > m_ref + 0.3f;
        const float m_new = need ? tmax + 0.5f : m_ref;
        const bool rescale = need && (m_ref != -INFINITY) && (cur > first);
        const float alpha = rescale ? exp2f(m_ref - m_new) : 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds earlier tiles of this piece: wait for PV(cur - 1), scale rows in TMEM
          if (!wait_or_fail(kBarPFree + ((cur - 1) & 1), ((cur - 1) >> 1) & 1, 1024)) break;
          tc_fence_after();
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kColO + 32 * k;
            tmem_ld_16x32bx2_x32<128>(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_16x32bx2_x32<128>(ta, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_ref = m_new;

        // P = 2^(x - m_ref + 8), split into e4m3 hi/lo, K-major no-swizzle layout
        const float mref8 = m_ref - 8.f;
        const bool live = m_ref != -INFINITY;
        uint32_t ph[8], pl[8];
        float lsum = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = live ? exp2f(x[2 * i] - mref8) : 0.f;
          const float bb = live ? exp2f(x[2 * i + 1] - mref8) : 0.f;
          lsum += a + bb;
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
        l += lsum;
        {
          unsigned char* pbh = sm + kOffP + (b * 2 + 0) * kPPart;
          unsigned char* pbl = sm + kOffP + (b * 2 + 1) * kPPart;
          const int off0 = (r >> 3) * 512 + (2 * hf) * 128 + (r & 7) * 16;
          *reinterpret_cast<uint4*>(pbh + off0) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(pbh + off0 + 128) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
          *reinterpret_cast<uint4*>(pbl + off0) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          *reinterpret_cast<uint4*>(pbl + off0 + 128) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
        }
        // last tile of the item: V rows past S (partial page, pages never loaded)
        // are zeroed so that 0 * garbage cannot reach O
        if (lt == pc.nt - 1 && (pc.S % kT) != 0) {
          if (!wait_or_fail(kBarFullV + s, (cur / kStages) & 1, 2048)) break;
          const int z0 = pc.S - lt * kT;
          const int nz = kT - z0;
          unsigned char* vst = sm + s * kStageBytes + kStageBytes / 2;
          for (int idx = tid - 128; idx < nz * 16; idx += 128) {
            const int row = z0 + (idx >> 4);
            const int h = (idx >> 3) & 1;
            const int ch = idx & 7;
            *reinterpret_cast<uint4*>(vst + h * 8192 + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + b));
      }
      if (!ok) break;

      // -- epilogue
      if (!wait_or_fail(kBarOFull, piece_idx & 1, 4096)) break;
      tc_fence_after();
      const float lrow = l + __shfl_xor_sync(0xffffffffu, l, 16);
      const float inv = lrow > 0.f ? vd / lrow : 0.f;
      const int64_t piece = (int64_t)pc.j + c;
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        uint32_t o[32];
        tmem_ld_16x32bx2_x32<128>(tmem + lane_base + kColO + 32 * k, o);
        tmem_wait_ld();
        const int col = 128 * hf + 32 * k;
        if (row_ok) {
          if (pc.direct) {
            uint16_t* dst = p.out + (int64_t)(pc.q0 + tq) * p.o_s0 + (int64_t)(pc.kvh * G + gq) * p.o_s1 + col;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint32_t w[4];
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const float y0 = __uint_as_float(o[v4 * 8 + 2 * e2]) * inv;
                const float y1 = __uint_as_float(o[v4 * 8 + 2 * e2 + 1]) * inv;
                w[e2] = (uint32_t)float_to_bf16_bits(y0) | ((uint32_t)float_to_bf16_bits(y1) << 16);
              }
              reinterpret_cast<uint4*>(dst)[v4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float* dst = p.ws_acc + (piece * p.max_rows + r) * kHeadDim + col;
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              reinterpret_cast<float4*>(dst)[v4] =
                  make_float4(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1]),
                              __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
          }
        }
      }
      if (row_ok && !pc.direct && hf == 0) {
        p.ws_ml[(piece * p.max_rows + r) * 2 + 0] = (m_ref == -INFINITY) ? -INFINITY : m_ref - 8.f;
        p.ws_ml[(piece * p.max_rows + r) * 2 + 1] = lrow;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree));
      ++piece_idx;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t prepare_main_tc() {
  return cudaFuncSetAttribute(va_main_tc_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
}

cudaError_t launch_main_tc_fp8(const Params& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                               cudaStream_t stream) {
  va_main_tc_fp8_kernel<<<p.num_splits, kThreads, kSmemBytes, stream>>>(p, tm_k, tm_v);
  return cudaGetLastError();
}

}  // namespace va
