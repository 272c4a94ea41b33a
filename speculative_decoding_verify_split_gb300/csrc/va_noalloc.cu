// verify_attn_noalloc: the same computation as verify_attn, for callers that
// must not allocate device memory.
//
// Some callers cannot call cudaMalloc at the moment they run attention: a
// serving runtime that sized its memory pool at start-up and forbids later
// device allocations (cudaMalloc synchronises the device and fragments the
// pool), an allocator or memory-manager callback that must not re-enter the
// allocator, or embedded hosts that own all GPU memory themselves. They can
// still pass their inputs and outputs; the split-KV partials the main kernel
// hands to the merge kernel then live in a fixed array compiled into this
// library instead of a workspace.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes bytes.
// Every GPU that loads the library keeps it until the process exits. Host
// code cannot use the array's name as a device address, so the address is
// looked up with cudaGetSymbolAddress once per device (with that device
// current) on the first call, and passed to the kernels.
#include <mutex>

#include "va_host_impl.h"

namespace {

constexpr size_t kNoAllocScratchBytes = VERIFY_ATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

namespace va_host_impl {

// Device address of the scratch array on the current device (looked up once,
// with that device current).
va_status noalloc_scratch(void** out, bool lookup) {
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return VA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] && lookup) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return VA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return VA_OK;
}

}  // namespace va_host_impl

using namespace va_host_impl;

VA_EXPORT va_status verify_attn_noalloc(const va_tensor* q, const va_tensor* k_cache,
                                        const va_tensor* v_cache, const va_tensor* block_table,
                                        const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                                        int32_t max_seqlen_q, int32_t max_seqlen_k,
                                        float softmax_scale, const va_tensor* k_descale,
                                        const va_tensor* v_descale, va_tensor* out, void* stream) {
  Shapes sh;
  va_status s = validate(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                         max_seqlen_k, k_descale, v_descale, out, &sh);
  if (s != VA_OK) return s;
  int sms = 0;
  s = current_device_sms(&sms);
  if (s != VA_OK) return s;
  va_plan plan;
  s = make_plan(sh.num_seqs, sh.hkv, sh.hq, max_seqlen_q, max_seqlen_k, sh.kv_dtype, sms, 0, &plan);
  if (s != VA_OK) return s;
  if ((size_t)plan.workspace_bytes > kNoAllocScratchBytes) return VA_ERR_WORKSPACE;
  if (sh.total_q == 0 || sh.num_seqs == 0) return VA_OK;
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch, true);
  if (s != VA_OK) return s;
  // Nothing in the scratch has to start at zero: every byte the merge kernel
  // reads is written earlier in the same call by the main kernel. Its first
  // word is the status word of bounded waits that ran out (sticky, as in a
  // workspace); verify_attn_last_device_error(NULL, ...) reads and clears it.
  return launch(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                max_seqlen_k, softmax_scale, k_descale, v_descale, out, sh, plan, scratch,
                kNoAllocScratchBytes, nullptr, static_cast<cudaStream_t>(stream));
}
