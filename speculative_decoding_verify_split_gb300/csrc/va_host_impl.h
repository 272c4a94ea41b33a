// Host helpers shared by the translation units that implement the C ABI.
#pragma once

#include <cuda_runtime.h>

#include "verify_attn.h"
#include "va_internal.h"

#define VA_EXPORT extern "C" __attribute__((visibility("default")))

namespace va_host_impl {

struct Shapes {
  int64_t total_q, hq, hkv, num_blocks, num_seqs, width;
  int32_t kv_dtype;
};

// Argument checks shared by every entry point (pure host code).
va_status validate(const va_tensor* q, const va_tensor* k, const va_tensor* v,
                   const va_tensor* bt, const va_tensor* cu, const va_tensor* su,
                   int32_t max_seqlen_q, int32_t max_seqlen_k, const va_tensor* kd,
                   const va_tensor* vd, const va_tensor* out, Shapes* sh);

// The split heuristic (pure host code). With a sliding window (window_left
// >= 0) an item's tiles are bounded by the window.
va_status make_plan(int64_t B, int64_t hkv, int64_t hq, int32_t max_q, int32_t max_k,
                    int32_t kv_dtype, int32_t num_sms, int32_t force, va_plan* plan,
                    int32_t window_left = -1);

// Checks the variant options against the shapes (NULL = all off).
va_status validate_options(const va_options* opts, const Shapes& sh);

// A shard's outputs (verify_attn_partial): fp32 o, natural-log lse, and the
// optional per-sequence causal extent.
struct PartialOut {
  const va_tensor* kv_extent;  // nullable
  va_tensor* o;
  va_tensor* lse;
};

// Launches the main and merge kernels with the given workspace and options
// (NULL = all off); with `part`, the merge writes the shard's o and lse.
va_status launch(const va_tensor* q, const va_tensor* k, const va_tensor* v, const va_tensor* bt,
                 const va_tensor* cu, const va_tensor* su, int32_t max_q, int32_t max_k,
                 float scale, const va_tensor* kd, const va_tensor* vd, va_tensor* out,
                 const Shapes& sh, const va_plan& plan, void* ws, size_t ws_bytes,
                 cudaEvent_t ev_mid, cudaStream_t stream, const va_options* opts = nullptr,
                 const PartialOut* part = nullptr);

// SM count of the current device (initialises the per-device state once).
va_status current_device_sms(int* sms);

// Limit of the main kernels' bounded waits for launches made now, in ns.
uint64_t wait_limit_ns();

// Device address of verify_attn_noalloc's built-in scratch on the current
// device. With lookup, looks it up on first use; without, *out is NULL until
// a verify_attn_noalloc call on this device has looked it up.
va_status noalloc_scratch(void** out, bool lookup);

}  // namespace va_host_impl
