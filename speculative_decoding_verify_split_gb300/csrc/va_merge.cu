// Segment-merge kernel: combines the per-segment partials (m, l, O) of every
// (sequence, KV head) whose key tiles were split over several CTAs, with
// log-sum-exp rescaling (the "reduce segments" pass of sglang PR 36330 digest,
// "Implementation breakdown" item 1):
//
//   M = max_s m_s,  out = v_descale * (sum_s 2^(m_s - M) O_s) / (sum_s 2^(m_s - M) l_s)
//
// Segments that saw no visible key (m = -inf, l = 0) weigh 0, and so do CTAs
// whose tile range is empty. The sums run in a fixed order (CTA order), so
// the result does not depend on timing or on physical page ids. Work items
// held by one CTA were written by the main kernel; items with no key tiles
// get zero rows here.
//
// One warp per packed row: the lanes read the segments' (m, l) in parallel,
// reduce, then each lane accumulates 8 of the 256 output columns. Launched as
// a programmatic dependent of the main kernel; it waits for the main kernel's
// memory before touching the workspace.
#include "va_split.cuh"

namespace va {
namespace {

constexpr int kRowsPerCta = 8;

__global__ void __launch_bounds__(32 * kRowsPerCta) va_merge_kernel(const Params p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int j = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.y * kRowsPerCta + warp;
  const int b = j / p.hkv;
  const int kvh = j - b * p.hkv;
  const int L = seq_q_len(p, b);
  const int G = p.group;
  if (r >= G * L) return;
  const int t = r / G, g = r - t * G;
  const int q0 = p.cu_q[b];
  uint16_t* dst = p.out + (int64_t)(q0 + t) * p.o_s0 + (int64_t)(kvh * G + g) * p.o_s1 + 8 * lane;

  const int nt = work_tiles(p, j);
  if (nt == 0) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    return;
  }
  const long long N = p.ws_meta[p.num_work];
  const long long ts = p.ws_meta[j];
  const int c0 = split_of(ts, N, p.num_splits);
  const int c1 = split_of(ts + nt - 1, N, p.num_splits);
  if (c0 == c1) return;  // one CTA held the whole item and wrote it
  const int ns = c1 - c0 + 1;

  // (m, l) of every segment, lanes in parallel
  auto seg_m = [&](int k, float& m, float& l) {
    const int c = c0 + k;
    m = -INFINITY;
    l = 0.f;
    if (split_begin(N, c, p.num_splits) == split_begin(N, c + 1, p.num_splits)) return;  // empty CTA
    const int64_t piece = (int64_t)j + c;
    const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + (piece * p.max_rows + r) * 2);
    m = ml.x;
    l = ml.y;
  };
  float M = -INFINITY;
  for (int k = lane; k < ns; k += 32) {
    float m, l;
    seg_m(k, m, l);
    M = fmaxf(M, m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M == -INFINITY) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    return;
  }

  float den = 0.f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int base = 0; base < ns; base += 32) {
    float m, l, w = 0.f;
    if (base + lane < ns) {
      seg_m(base + lane, m, l);
      w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      den = fmaf(w, l, den);
    }
    const int cnt = ns - base < 32 ? ns - base : 32;
#pragma unroll 4
    for (int k = 0; k < cnt; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      if (wk == 0.f) continue;
      const int64_t piece = (int64_t)j + c0 + base + k;
      const float4* src = reinterpret_cast<const float4*>(p.ws_acc + (piece * p.max_rows + r) * kHeadDim) + 2 * lane;
      const float4 a = src[0], bq = src[1];
      acc[0] = fmaf(wk, a.x, acc[0]);
      acc[1] = fmaf(wk, a.y, acc[1]);
      acc[2] = fmaf(wk, a.z, acc[2]);
      acc[3] = fmaf(wk, a.w, acc[3]);
      acc[4] = fmaf(wk, bq.x, acc[4]);
      acc[5] = fmaf(wk, bq.y, acc[5]);
      acc[6] = fmaf(wk, bq.z, acc[6]);
      acc[7] = fmaf(wk, bq.w, acc[7]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float vd = p.v_descale ? *p.v_descale : 1.0f;
  const float inv = vd / den;
  uint32_t w4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w4[i] = (uint32_t)float_to_bf16_bits(acc[2 * i] * inv) |
            ((uint32_t)float_to_bf16_bits(acc[2 * i + 1] * inv) << 16);
  *reinterpret_cast<uint4*>(dst) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
}

}  // namespace

cudaError_t launch_merge(const Params& p, cudaStream_t stream) {
  if (p.num_work == 0 || p.max_rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_work, (unsigned)((p.max_rows + kRowsPerCta - 1) / kRowsPerCta));
  cfg.blockDim = dim3(32 * kRowsPerCta);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, va_merge_kernel, p);
}

}  // namespace va
