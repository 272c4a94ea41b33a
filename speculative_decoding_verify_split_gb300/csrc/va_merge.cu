// Segment-merge kernel: combines the per-segment partials (m, l, O) of every
// (sequence, KV head) whose key tiles were split over several CTAs, with
// log-sum-exp rescaling (the "reduce segments" pass of sglang PR 36330 digest,
// "Implementation breakdown" item 1):
//
//   M = max_s m_s,  out = v_descale * (sum_s 2^(m_s - M) O_s) / (sum_s 2^(m_s - M) l_s)
//
// Segments that saw no visible key (m = -inf, l = 0) weigh 0. The segment
// order is fixed (CTA order), so the result does not depend on timing or on
// physical page ids. Work items held by one CTA were written by the main
// kernel; items with no key tiles get zero rows here.
//
// Grid: (work item j, packed row r); 256 threads, thread d owns column d.
#include "va_split.cuh"

namespace va {
namespace {

__global__ void __launch_bounds__(kHeadDim) va_merge_kernel(const Params p) {
  const int j = blockIdx.x;
  const int r = blockIdx.y;
  const int d = threadIdx.x;
  const int b = j / p.hkv;
  const int kvh = j - b * p.hkv;
  const int L = seq_q_len(p, b);
  const int G = p.group;
  if (r >= G * L) return;
  const int t = r / G, g = r - t * G;
  const int q0 = p.cu_q[b];
  uint16_t* dst = p.out + (int64_t)(q0 + t) * p.o_s0 + (int64_t)(kvh * G + g) * p.o_s1 + d;

  const int nt = work_tiles(p, j);
  if (nt == 0) {
    *dst = 0;
    return;
  }
  const long long N = p.ws_meta[p.num_work];
  const long long ts = p.ws_meta[j];
  const int c0 = split_of(ts, N, p.num_splits);
  const int c1 = split_of(ts + nt - 1, N, p.num_splits);
  if (c0 == c1) return;  // one CTA held the whole item and wrote it

  // CTAs with an empty range (possible when there are more CTAs than tiles)
  // wrote no partial and are skipped.
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c) {
    if (split_begin(N, c, p.num_splits) == split_begin(N, c + 1, p.num_splits)) continue;
    const int64_t piece = (int64_t)j + c;
    M = fmaxf(M, p.ws_ml[(piece * p.max_rows + r) * 2]);
  }
  if (M == -INFINITY) {
    *dst = 0;
    return;
  }
  float num = 0.f, den = 0.f;
  for (int c = c0; c <= c1; ++c) {
    if (split_begin(N, c, p.num_splits) == split_begin(N, c + 1, p.num_splits)) continue;
    const int64_t piece = (int64_t)j + c;
    const float m = p.ws_ml[(piece * p.max_rows + r) * 2];
    const float l = p.ws_ml[(piece * p.max_rows + r) * 2 + 1];
    const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
    den = fmaf(w, l, den);
    num = fmaf(w, p.ws_acc[(piece * p.max_rows + r) * kHeadDim + d], num);
  }
  const float vd = p.v_descale ? *p.v_descale : 1.0f;
  *dst = float_to_bf16_bits(num * (vd / den));
}

}  // namespace

cudaError_t launch_merge(const Params& p, cudaStream_t stream) {
  if (p.num_work == 0 || p.max_rows == 0) return cudaSuccess;
  dim3 grid((unsigned)p.num_work, (unsigned)p.max_rows);
  va_merge_kernel<<<grid, kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace va
