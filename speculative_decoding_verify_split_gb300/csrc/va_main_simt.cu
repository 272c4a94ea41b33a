// Split-KV main kernel, CUDA-core version (plain fp32 FMAs, no tensor cores).
//
// The general path: any KV dtype, any packed row count up to 64. One CTA
// takes an equal share of the batch's key tiles (the split-KV segments of
// sglang PR 36330 digest, "Implementation breakdown" item 1) and, for every
// (sequence, KV head) its share touches, packs all G query heads x L draft
// tokens of that sequence into one tile of rows, so each K/V element is read
// from HBM once per KV head (sglang PR 30105 digest, "Implementation
// breakdown" item 2: one KV load serves the whole GQA group).
//
// Per row r = t * G + g (draft token t, query head kvh * G + g) it keeps an
// online softmax in log2 units: m = running max of scale*log2(e)*q.k, l = sum
// of 2^(s - m), O = sum of 2^(s - m) v. A work item wholly inside the CTA's
// share is normalised and written to `out`; otherwise (m, l, O) go to the
// workspace for the merge kernel.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "va_split.cuh"

namespace va {
namespace {

constexpr int kNT = 256;           // threads; thread d owns output column d
constexpr int kT = kSimtTileKeys;  // keys per tile
constexpr int kKStride = kHeadDim + 1;

struct SimtSmem {
  float q[kMaxRows][kHeadDim];
  float k[kT][kKStride];
  float v[kT][kHeadDim];
  float s[kMaxRows][kT + 1];
  float m[kMaxRows];
  float l[kMaxRows];
  float alpha[kMaxRows];
  long long scratch[32];
  long long ts;
  int j;
};

__device__ __forceinline__ float load_kv(const void* base, int64_t off, bool fp8) {
  if (fp8) {
    const __nv_fp8_storage_t x = reinterpret_cast<const uint8_t*>(base)[off];
    const __half_raw h = __nv_cvt_fp8_to_halfraw(x, __NV_E4M3);
    return __half2float(__half(h));
  }
  return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(base)[off]);
}

__global__ void __launch_bounds__(kNT, 1) va_main_simt_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const bool fp8 = p.kv_fp8 != 0;

  const long long N = scan_work<kNT>(p, sm.scratch, c == 0);
  const long long t0 = split_begin(N, c, p.num_splits);
  const long long t1 = split_begin(N, c + 1, p.num_splits);
  if (t0 >= t1) return;

  int j;
  long long ts;
  find_work<kNT>(p, t0, sm.scratch, &sm.j, &sm.ts, &j, &ts);

  const float kd = p.k_descale ? *p.k_descale : 1.0f;
  const float vd = p.v_descale ? *p.v_descale : 1.0f;
  const float cscale = p.scale_log2 * kd;
  const int G = p.group;

  while (j < p.num_work && ts < t1) {
    const int nt = work_tiles(p, j);
    if (nt == 0) {  // an item with no tiles occupies no range
      ++j;
      continue;
    }
    const int b = j / p.hkv;
    const int kvh = j - b * p.hkv;
    const int S = seq_kv_len(p, b);
    const int L = seq_q_len(p, b);
    const int q0 = p.cu_q[b];
    const int R = G * L;
    const long long lt0 = (t0 > ts ? t0 : ts) - ts;
    const long long lt1 = (t1 < ts + nt ? t1 : ts + nt) - ts;
    const bool direct = (lt0 == 0 && lt1 == nt);

    for (int idx = tid; idx < kMaxRows * kHeadDim; idx += kNT) {
      const int r = idx / kHeadDim, d = idx % kHeadDim;
      float val = 0.f;
      if (r < R) {
        const int t = r / G, g = r - t * G;
        val = bf16_bits_to_float(p.q[(int64_t)(q0 + t) * p.q_s0 + (int64_t)(kvh * G + g) * p.q_s1 + d]);
      }
      sm.q[r][d] = val;
    }
    if (tid < kMaxRows) {
      sm.m[tid] = -INFINITY;
      sm.l[tid] = 0.f;
    }
    float o[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) o[r] = 0.f;
    __syncthreads();

    for (long long lt = lt0; lt < lt1; ++lt) {
      const int key0 = (int)lt * kT;
      for (int idx = tid; idx < kT * kHeadDim; idx += kNT) {
        const int kk = idx / kHeadDim, d = idx % kHeadDim;
        const int key = key0 + kk;
        float kx = 0.f, vx = 0.f;
        if (key < S) {
          const int page = p.block_table[(int64_t)b * p.bt_s0 + (int64_t)(key / kPageSize) * p.bt_s1];
          if ((unsigned)page < (unsigned)p.num_blocks) {
            const int slot = key % kPageSize;
            kx = load_kv(p.k, (int64_t)page * p.k_s0 + (int64_t)slot * p.k_s1 + (int64_t)kvh * p.k_s2 + d, fp8);
            vx = load_kv(p.v, (int64_t)page * p.v_s0 + (int64_t)slot * p.v_s1 + (int64_t)kvh * p.v_s2 + d, fp8);
          }
        }
        sm.k[kk][d] = kx;
        sm.v[kk][d] = vx;
      }
      __syncthreads();

      {  // logits: warp w handles rows w, w+8, ...; lane = key within the tile
        const int kk = tid & 31;
        const int key = key0 + kk;
        for (int r = tid >> 5; r < R; r += kNT / 32) {
          float acc = 0.f;
#pragma unroll 8
          for (int d = 0; d < kHeadDim; ++d) acc = fmaf(sm.q[r][d], sm.k[kk][d], acc);
          const int t = r / G;
          const bool vis = key < S && key <= S - L + t;
          sm.s[r][kk] = vis ? acc * cscale : -INFINITY;
        }
      }
      __syncthreads();

      if (tid < R) {  // online softmax, one thread per row
        const int r = tid;
        float mx = -INFINITY;
        for (int kk = 0; kk < kT; ++kk) mx = fmaxf(mx, sm.s[r][kk]);
        const float mold = sm.m[r];
        const float mnew = fmaxf(mold, mx);
        const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(mold - mnew);
        float sum = 0.f;
        for (int kk = 0; kk < kT; ++kk) {
          const float sv = sm.s[r][kk];
          const float pv = (sv == -INFINITY) ? 0.f : exp2f(sv - mnew);
          sm.s[r][kk] = pv;
          sum += pv;
        }
        sm.l[r] = sm.l[r] * alpha + sum;
        sm.m[r] = mnew;
        sm.alpha[r] = alpha;
      }
      __syncthreads();

      {  // O[r][d] = alpha * O[r][d] + sum_k P[r][k] V[k][d]
        const int d = tid;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          if (r < R) {
            float acc = o[r] * sm.alpha[r];
#pragma unroll 8
            for (int kk = 0; kk < kT; ++kk) acc = fmaf(sm.s[r][kk], sm.v[kk][d], acc);
            o[r] = acc;
          }
        }
      }
      __syncthreads();
    }

    const int d = tid;
    if (direct) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < R) {
          const int t = r / G, g = r - t * G;
          const float lr = sm.l[r];
          const float y = lr > 0.f ? o[r] * (vd / lr) : 0.f;
          p.out[(int64_t)(q0 + t) * p.o_s0 + (int64_t)(kvh * G + g) * p.o_s1 + d] = float_to_bf16_bits(y);
        }
      }
    } else {
      const int64_t piece = (int64_t)j + c;
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < R) p.ws_acc[(piece * p.max_rows + r) * kHeadDim + d] = o[r];
      }
      if (tid < R) {
        p.ws_ml[(piece * p.max_rows + tid) * 2 + 0] = sm.m[tid];
        p.ws_ml[(piece * p.max_rows + tid) * 2 + 1] = sm.l[tid];
      }
    }
    __syncthreads();
    ts += nt;
    ++j;
  }
}

constexpr int kSmemBytes = (int)sizeof(SimtSmem);

}  // namespace

cudaError_t prepare_main_simt() {
  return cudaFuncSetAttribute(va_main_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
}

cudaError_t launch_main_simt(const Params& p, cudaStream_t stream) {
  va_main_simt_kernel<<<p.num_splits, kNT, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace va
