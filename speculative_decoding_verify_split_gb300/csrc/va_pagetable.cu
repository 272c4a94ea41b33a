// Block table and KV lengths from the flat token-slot form of a batch
// (sglang PR 30105 digest, "Fix 2: draft_extend_v2 re-routed to
// unified_attention"): the draft-extend pass builds a 2D page table from its
// flat metadata and takes each sequence's KV length as the difference of
// consecutive kv_indptr entries, then runs the same split-KV attention.
//
// kv_indices holds the cache token slot of every token (slot = page * 16 +
// position in the page), sequence b's tokens at [kv_indptr[b], kv_indptr[b+1]).
// Entry p of row b is the page of tokens [16p, 16p + 16): the page of its
// first slot. One thread per entry checks that the page's slots are one
// aligned page in order; problems are ORed into an optional status word.
#include "va_internal.h"

namespace va {
namespace {

constexpr int kBtThreads = 256;

__global__ void __launch_bounds__(kBtThreads)
    va_block_table_kernel(const int32_t* __restrict__ indptr, const int32_t* __restrict__ indices,
                          int64_t nnz, int32_t width, int32_t* __restrict__ bt, int64_t bt_s0,
                          int64_t bt_s1, int32_t* __restrict__ seqused, int64_t sk_s0, int32_t pad,
                          int32_t* status) {
  const int b = blockIdx.y;
  const int64_t p = (int64_t)blockIdx.x * kBtThreads + threadIdx.x;
  int64_t a = indptr[b], e = indptr[b + 1];
  int flags = 0;
  if (a < 0 || e < a || e > nnz) {  // unusable range: empty row, length 0
    if (p == 0) flags |= kBtBadIndptr;
    a = e = 0;
  }
  const int64_t n = e - a;
  const int64_t npg = (n + kPageSize - 1) / kPageSize;
  if (p == 0) {
    seqused[(int64_t)b * sk_s0] = (int32_t)(n < INT32_MAX ? n : INT32_MAX);
    if (npg > width) flags |= kBtTruncated;
  }
  if (p < width) {
    int32_t v = pad;
    if (p < npg) {
      const int64_t t0 = a + (int64_t)kPageSize * p;
      const int64_t left = n - (int64_t)kPageSize * p;
      const int cnt = left < kPageSize ? (int)left : kPageSize;
      const int32_t s0 = indices[t0];
      bool in_order = s0 >= 0 && (s0 % kPageSize) == 0;
      for (int i = 1; i < cnt; ++i) in_order &= indices[t0 + i] == s0 + i;
      if (!in_order) flags |= kBtBadPage;
      v = s0 >= 0 ? s0 / kPageSize : pad;
    }
    bt[(int64_t)b * bt_s0 + p * bt_s1] = v;
  }
  if (flags && status) atomicOr(status, flags);
}

}  // namespace

cudaError_t launch_block_table(const int32_t* indptr, const int32_t* indices, int64_t nnz,
                               int32_t num_seqs, int32_t width, int32_t* bt, int64_t bt_s0,
                               int64_t bt_s1, int32_t* seqused, int64_t sk_s0, int32_t pad,
                               int32_t* status, cudaStream_t stream) {
  if (num_seqs == 0) return cudaSuccess;
  const int64_t cols = width > 0 ? width : 1;  // column 0 also writes the length
  const dim3 grid((unsigned)((cols + kBtThreads - 1) / kBtThreads), (unsigned)num_seqs);
  va_block_table_kernel<<<grid, kBtThreads, 0, stream>>>(indptr, indices, nnz, width, bt, bt_s0, bt_s1,
                                                         seqused, sk_s0, pad, status);
  return cudaGetLastError();
}

}  // namespace va
