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
// PARTIAL: a shard's result (verify_attn_partial): every item is merged here,
// also one held by a single CTA, and the row is written as fp32 o and its
// natural-log lse instead of bf16 out.
template <bool SINKS, int DV, bool PARTIAL>
__global__ void __launch_bounds__(kMergeThreads, 4) va_merge_kernel(const Params p) {
  constexpr int kThreadsPerRow = DV / 4;
  constexpr int kRowsPerCta = kMergeThreads / kThreadsPerRow;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next call's main kernel may be scheduled now (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int j = blockIdx.x;
  const int r = blockIdx.y * kRowsPerCta + (int)(threadIdx.x / kThreadsPerRow);
  const int col4 = (int)(threadIdx.x % kThreadsPerRow);
  const int b = j / p.hkv;
  const int kvh = j - b * p.hkv;
  // the split metadata (written for every item) is read with the lengths,
  // not after them: one round trip instead of two before the partials
  const long long N = p.ws_meta[p.num_work];
  const long long ts = p.ws_meta[j];
  const int L = seq_q_len(p, b);
  const int G = p.group;
  if (r >= G * L) return;
  const int t = r / G, g = r - t * G;
  const int q0 = p.cu_q[b];
  uint16_t* dst = p.out + (int64_t)(q0 + t) * p.o_s0 + (int64_t)(kvh * G + g) * p.o_s1 + 4 * col4;
  // a shard's row: o (fp32) and, from the row's first thread, lse
  auto put_partial = [&](float4 o, float lse) {
    *reinterpret_cast<float4*>(p.o_part + (int64_t)(q0 + t) * p.op_s0 + (int64_t)(kvh * G + g) * p.op_s1 + 4 * col4) = o;
    if (col4 == 0) p.lse_part[(int64_t)(q0 + t) * p.lse_s0 + (int64_t)(kvh * G + g) * p.lse_s1] = lse;
  };

  const int nt = work_tiles(p, j);
  if (nt == 0) {
    if constexpr (PARTIAL)
      put_partial(make_float4(0.f, 0.f, 0.f, 0.f), -INFINITY);
    else
      *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
    return;
  }
  const int c0 = split_of(ts, N, p.num_splits);
  const int c1 = split_of(ts + nt - 1, N, p.num_splits);
  if (!PARTIAL && c0 == c1) return;  // one CTA held the whole item and wrote it
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
    if constexpr (PARTIAL)
      put_partial(make_float4(0.f, 0.f, 0.f, 0.f), -INFINITY);
    else
      *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
    return;
  }
  if constexpr (SINKS)  // the attention sink's share of the normaliser, once per row
    den += exp2f(p.sinks[kvh * G + g] * 1.4426950408889634f - M);
  const float vd = p.v_descale ? *p.v_descale : 1.0f;
  const float inv = vd / den;
  if constexpr (PARTIAL) {
    // the rows' logits are in log2 units: sum 2^x = 2^M den
    put_partial(make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv),
                (M + log2f(den)) * 0.6931471805599453f);
    return;
  }
  const uint32_t w0 = (uint32_t)float_to_bf16_bits(acc.x * inv) | ((uint32_t)float_to_bf16_bits(acc.y * inv) << 16);
  const uint32_t w1 = (uint32_t)float_to_bf16_bits(acc.z * inv) | ((uint32_t)float_to_bf16_bits(acc.w * inv) << 16);
  *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
}

// The latent-cache path's merge. Its partials come in groups of four rows,
// partial[piece][row / 4][column][row % 4] (mla_acc_index), and every piece
// has one, also when a single CTA held the whole item. One thread per output
// column (512), GROUPS groups of four packed rows per CTA: a thread reads one
// 16-byte group per segment and group, a warp's loads are 512 contiguous
// bytes, and two CTAs fit on an SM. Segments go SEGS at a time: every thread
// issues all its partial loads at once (one L2 round trip per chunk), while
// warp 0, one lane per (segment, row), reads the chunk's (m, l), moves each
// row's running max and publishes the chunk's weights 2^(m_s - M) and the
// rescale of the earlier sum in shared memory. Each output row is written as
// one coalesced 1 KB line. (GROUPS, SEGS) is (1, 8) while the four-row CTAs
// fit in one wave, else (2, 4): half the CTAs, two row groups of four
// segments per thread.
template <int GROUPS, int SEGS>
__global__ void __launch_bounds__(kMlaNope, 2) va_merge_mla_kernel(const Params p) {
  constexpr int kRows = 4 * GROUPS;  // rows per CTA
  static_assert(SEGS * kRows == 32, "warp 0: one lane per (segment, row)");
  __shared__ float s_w[SEGS][kRows];
  __shared__ float s_sc[kRows];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int j = blockIdx.x;  // one KV head: item j is sequence j
  const int r0 = blockIdx.y * kRows;
  const int d = threadIdx.x;
  const int L = seq_q_len(p, j);
  const int G = p.group;
  const int R = G * L;
  if (r0 >= R) return;  // CTA-uniform
  const int nrow = R - r0 < kRows ? R - r0 : kRows;
  const int q0 = p.cu_q[j];
  auto dst = [&](int rr) {
    const int t = (r0 + rr) / G, g = (r0 + rr) - t * G;
    return p.out + (int64_t)(q0 + t) * p.o_s0 + (int64_t)g * p.o_s1 + d;
  };
  const int nt = work_tiles(p, j);
  if (nt == 0) {
    for (int rr = 0; rr < nrow; ++rr) *dst(rr) = 0;
    return;
  }
  const long long N = p.ws_meta[p.num_work];
  const long long ts = p.ws_meta[j];
  const int c0 = split_of(ts, N, p.num_splits);
  const int c1 = split_of(ts + nt - 1, N, p.num_splits);
  const int ns = c1 - c0 + 1;
  const bool may_be_empty = N < (long long)p.num_splits;
  const int ldr = mla_row_stride(p.max_rows);
  // a CTA range can be empty only with fewer split units than CTAs; such a
  // segment wrote nothing and is never read
  auto exists = [&](int k) {
    const int c = c0 + k;
    return k < ns && (!may_be_empty || split_begin(N, c, p.num_splits) != split_begin(N, c + 1, p.num_splits));
  };

  float acc[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) acc[i] = 0.f;
  float M = -INFINITY, den = 0.f;  // row (d % kRows)'s, in warp 0
  for (int base = 0; base < ns; base += SEGS) {
    float4 a[SEGS][GROUPS];
#pragma unroll
    for (int k = 0; k < SEGS; ++k) {
      const int64_t piece = (int64_t)j + c0 + base + k;
#pragma unroll
      for (int gg = 0; gg < GROUPS; ++gg)  // groups past the piece's rows do not exist
        a[k][gg] = (exists(base + k) && r0 + 4 * gg < ldr)
                       ? __ldcg(reinterpret_cast<const float4*>(p.ws_acc + mla_acc_index(piece, r0 + 4 * gg, d, ldr)))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (d < 32) {
      // warp 0: lane kRows k + i holds segment base + k, row r0 + i; rows
      // reduce over the lanes with the same i
      const int k = d / kRows, i = d % kRows;
      float2 ml = make_float2(-INFINITY, 0.f);
      if (i < nrow && exists(base + k))
        ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + (((int64_t)j + c0 + base + k) * p.max_rows + r0 + i) * 2));
      float mc = ml.x;
#pragma unroll
      for (int o = kRows; o < 32; o <<= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
      mc = fmaxf(mc, M);
      const float sc = (M == -INFINITY || mc == -INFINITY) ? 0.f : exp2f(M - mc);
      const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mc);
      float wl = w * ml.y;
#pragma unroll
      for (int o = kRows; o < 32; o <<= 1) wl += __shfl_xor_sync(0xffffffffu, wl, o);
      den = den * sc + wl;  // each lane keeps its row's (M, den)
      if (mc != -INFINITY) M = mc;
      s_w[k][i] = w;
      if (k == 0) s_sc[i] = sc;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      float x = acc[i] * s_sc[i];
#pragma unroll
      for (int k = 0; k < SEGS; ++k) {
        const float4 v = a[k][i / 4];
        const int e = i % 4;
        x = fmaf(s_w[k][i], e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w)), x);
      }
      acc[i] = x;
    }
    __syncthreads();  // s_w and s_sc are rewritten by the next group
  }
  const float vd = p.v_descale ? *p.v_descale : 1.0f;
  if (d < kRows) s_sc[d] = (M == -INFINITY || !(den > 0.f)) ? 0.f : vd / den;  // lanes 0..kRows-1
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kRows; ++i)
    if (i < nrow) *dst(i) = float_to_bf16_bits(acc[i] * s_sc[i]);
}

// Log-sum-exp merge of shard results (verify_attn_merge_partials):
// out = sum_i exp(lse_i - LSE) o_i, LSE = ln sum_i exp(lse_i), as bf16; rows
// whose lse are all -inf are 0. 64 threads per row, one float4 of the 256
// columns each; the shards' loads go out together.
__global__ void __launch_bounds__(kMergeThreads) va_merge_shards_kernel(const ShardMergeParams m) {
  constexpr int kThreadsPerRow = kHeadDim / 4;
  constexpr int kRowsPerCta = kMergeThreads / kThreadsPerRow;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + threadIdx.x / kThreadsPerRow;
  const int col4 = threadIdx.x % kThreadsPerRow;
  if (row >= (int64_t)m.total_q * m.hq) return;
  const int t = (int)(row / m.hq), h = (int)(row - (int64_t)t * m.hq);
  float lse[kMaxShards];
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxShards; ++i) {
    lse[i] = i < m.n ? m.lse[i][(int64_t)t * m.lse_s0[i] + (int64_t)h * m.lse_s1[i]] : -INFINITY;
    M = fmaxf(M, lse[i]);
  }
  uint16_t* dst = m.out + (int64_t)t * m.out_s0 + (int64_t)h * m.out_s1 + 4 * col4;
  if (M == -INFINITY) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
    return;
  }
  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxShards; ++i) {
    if (i >= m.n || lse[i] == -INFINITY) continue;  // a shard with no visible key is never read
    const float w = __expf(lse[i] - M);
    const float4 o = *reinterpret_cast<const float4*>(m.o[i] + (int64_t)t * m.o_s0[i] + (int64_t)h * m.o_s1[i] + 4 * col4);
    den += w;
    acc.x = fmaf(w, o.x, acc.x);
    acc.y = fmaf(w, o.y, acc.y);
    acc.z = fmaf(w, o.z, acc.z);
    acc.w = fmaf(w, o.w, acc.w);
  }
  const float inv = 1.f / den;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2((uint32_t)float_to_bf16_bits(acc.x * inv) | ((uint32_t)float_to_bf16_bits(acc.y * inv) << 16),
                 (uint32_t)float_to_bf16_bits(acc.z * inv) | ((uint32_t)float_to_bf16_bits(acc.w * inv) << 16));
}

}  // namespace

cudaError_t launch_merge(const Params& p, cudaStream_t stream) {
  if (p.num_work == 0 || p.max_rows == 0) return cudaSuccess;
  if (p.dv != kHeadDim && p.dv != kMlaNope) return cudaErrorInvalidValue;
  if (p.dv == kMlaNope) {
    // four-row CTAs while they fit in one wave (two per SM, one split per
    // SM), else eight-row CTAs: mla_mid_context_fp8 (768 four-row CTAs)
    const int64_t ctas4 = (int64_t)p.num_work * ((p.max_rows + 3) / 4);
    const bool wide = ctas4 > 2 * (int64_t)p.num_splits;
    const int rows = wide ? 8 : 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.num_work, (unsigned)((p.max_rows + rows - 1) / rows));
    cfg.blockDim = dim3(kMlaNope);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return wide ? cudaLaunchKernelEx(&cfg, va_merge_mla_kernel<2, 4>, p)
                : cudaLaunchKernelEx(&cfg, va_merge_mla_kernel<1, 8>, p);
  }
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
  if (p.partial) return cudaLaunchKernelEx(&cfg, va_merge_kernel<false, kHeadDim, true>, p);
  return p.sinks ? cudaLaunchKernelEx(&cfg, va_merge_kernel<true, kHeadDim, false>, p)
                 : cudaLaunchKernelEx(&cfg, va_merge_kernel<false, kHeadDim, false>, p);
}

}  // namespace va

namespace va {

cudaError_t launch_merge_shards(const ShardMergeParams& m, cudaStream_t stream) {
  const int64_t rows = (int64_t)m.total_q * m.hq;
  if (rows == 0) return cudaSuccess;
  constexpr int kRowsPerCta = kMergeThreads / (kHeadDim / 4);
  va_merge_shards_kernel<<<(unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta), kMergeThreads, 0, stream>>>(m);
  return cudaGetLastError();
}

}  // namespace va
