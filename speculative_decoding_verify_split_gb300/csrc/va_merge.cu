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
// One thread per float4 of a packed row's output columns (64 threads for the
// 256 columns of a head, 128 for the 512 of a latent), so a row's segments
// are read as coalesced lines. Segments are taken eight
// at a time with all their loads in flight together, and folded into a
// running (max, denominator, accumulator) triple: the latency of a merge is
// one L2 round trip per eight segments. Launched as a programmatic dependent
// of the main kernel; it waits for the main kernel's memory before touching
// the workspace.
#include "va_split.cuh"

namespace va {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kSegChunk = 8;

// SINKS: compiled with the attention-sink term. DV: output columns per row.
template <bool SINKS, int DV>
__global__ void __launch_bounds__(kMergeThreads, 4) va_merge_kernel(const Params p) {
  constexpr int kThreadsPerRow = DV / 4;
  constexpr int kRowsPerCta = kMergeThreads / kThreadsPerRow;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int j = blockIdx.x;
  const int r = blockIdx.y * kRowsPerCta + (int)(threadIdx.x / kThreadsPerRow);
  const int col4 = (int)(threadIdx.x % kThreadsPerRow);
  const int b = j / p.hkv;
  const int kvh = j - b * p.hkv;
  const int L = seq_q_len(p, b);
  const int G = p.group;
  if (r >= G * L) return;
  const int t = r / G, g = r - t * G;
  const int q0 = p.cu_q[b];
  uint16_t* dst = p.out + (int64_t)(q0 + t) * p.o_s0 + (int64_t)(kvh * G + g) * p.o_s1 + 4 * col4;

  const int nt = work_tiles(p, j);
  if (nt == 0) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
    return;
  }
  const long long N = p.ws_meta[p.num_work];
  const long long ts = p.ws_meta[j];
  const int c0 = split_of(ts, N, p.num_splits);
  const int c1 = split_of(ts + nt - 1, N, p.num_splits);
  if (c0 == c1) return;  // one CTA held the whole item and wrote it
  const int ns = c1 - c0 + 1;
  // A CTA range can only be empty when there are fewer split units than CTAs;
  // otherwise skip the two 64-bit divisions per segment.
  const bool may_be_empty = N < (long long)p.num_splits;

  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < ns; base += kSegChunk) {
    float m[kSegChunk], l[kSegChunk];
    float4 a[kSegChunk];
#pragma unroll
    for (int k = 0; k < kSegChunk; ++k) {
      m[k] = -INFINITY;
      l[k] = 0.f;
      a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int c = c0 + base + k;
      if (base + k < ns &&
          (!may_be_empty || split_begin(N, c, p.num_splits) != split_begin(N, c + 1, p.num_splits))) {
        const int64_t row = ((int64_t)j + c) * p.max_rows + r;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + row * 2));
        m[k] = ml.x;
        l[k] = ml.y;
        a[k] = __ldcg(reinterpret_cast<const float4*>(p.ws_acc + row * DV) + col4);
      }
    }
    float mc = M;
#pragma unroll
    for (int k = 0; k < kSegChunk; ++k) mc = fmaxf(mc, m[k]);
    if (mc == -INFINITY) continue;  // nothing visible yet
    const float sc = (M == -INFINITY) ? 0.f : exp2f(M - mc);
    den *= sc;
    acc.x *= sc;
    acc.y *= sc;
    acc.z *= sc;
    acc.w *= sc;
#pragma unroll
    for (int k = 0; k < kSegChunk; ++k) {
      if (m[k] == -INFINITY) continue;  // weight 0; its partial is never read
      const float w = exp2f(m[k] - mc);
      den = fmaf(w, l[k], den);
      acc.x = fmaf(w, a[k].x, acc.x);
      acc.y = fmaf(w, a[k].y, acc.y);
      acc.z = fmaf(w, a[k].z, acc.z);
      acc.w = fmaf(w, a[k].w, acc.w);
    }
    M = mc;
  }
  if (M == -INFINITY) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
    return;
  }
  if constexpr (SINKS)  // the attention sink's share of the normaliser, once per row
    den += exp2f(p.sinks[kvh * G + g] * 1.4426950408889634f - M);
  const float vd = p.v_descale ? *p.v_descale : 1.0f;
  const float inv = vd / den;
  const uint32_t w0 = (uint32_t)float_to_bf16_bits(acc.x * inv) | ((uint32_t)float_to_bf16_bits(acc.y * inv) << 16);
  const uint32_t w1 = (uint32_t)float_to_bf16_bits(acc.z * inv) | ((uint32_t)float_to_bf16_bits(acc.w * inv) << 16);
  *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
}

}  // namespace

cudaError_t launch_merge(const Params& p, cudaStream_t stream) {
  if (p.num_work == 0 || p.max_rows == 0) return cudaSuccess;
  if (p.dv != kHeadDim && p.dv != kMlaNope) return cudaErrorInvalidValue;
  const int rows_per_cta = kMergeThreads / (p.dv / 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_work, (unsigned)((p.max_rows + rows_per_cta - 1) / rows_per_cta));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.dv == kMlaNope) return cudaLaunchKernelEx(&cfg, va_merge_kernel<false, kMlaNope>, p);
  return p.sinks ? cudaLaunchKernelEx(&cfg, va_merge_kernel<true, kHeadDim>, p)
                 : cudaLaunchKernelEx(&cfg, va_merge_kernel<false, kHeadDim>, p);
}

}  // namespace va
