// Host side of the C ABI (include/verify_attn.h): argument validation, the
// split heuristic, the library-owned workspace and the kernel launches.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "va_host_impl.h"

namespace va_host_impl {

using namespace va;

constexpr int kMaxDevices = 64;

int64_t numel(const va_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int32_t dt) {
  switch (dt) {
    case VA_BF16: return 2;
    case VA_FP8_E4M3: return 1;
    case VA_INT32: return 4;
    case VA_FP32: return 4;
    default: return 0;
  }
}

bool dims_ok(const va_tensor* t, int ndim) {
  if (t->ndim != ndim) return false;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0 || t->stride[i] < 0) return false;
  return true;
}

// Strides of all but the innermost dimension, in bytes, are multiples of 16
// and the innermost stride is 1.
bool rows_16b(const va_tensor* t) {
  const int es = elem_size(t->dtype);
  if (t->stride[t->ndim - 1] != 1) return false;
  for (int i = 0; i < t->ndim - 1; ++i)
    if ((t->stride[i] * es) % 16 != 0) return false;
  return true;
}

va_status check_descale(const va_tensor* t) {
  if (!t) return VA_OK;
  if (t->ndim < 0 || t->ndim > 4) return VA_ERR_SHAPE;
  if (t->dtype != VA_FP32) return VA_ERR_DTYPE;
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] < 0) return VA_ERR_SHAPE;
  if (numel(t) != 1) return VA_ERR_SHAPE;
  if (!t->data) return VA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(t->data) & 3u) != 0) return VA_ERR_LAYOUT;
  return VA_OK;
}

va_status validate(const va_tensor* q, const va_tensor* k, const va_tensor* v,
                   const va_tensor* bt, const va_tensor* cu, const va_tensor* su,
                   int32_t max_seqlen_q, int32_t max_seqlen_k, const va_tensor* kd,
                   const va_tensor* vd, const va_tensor* out, Shapes* sh) {
  if (!q || !k || !v || !bt || !cu || !su || !out) return VA_ERR_NULL;
  if (!dims_ok(q, 3) || !dims_ok(k, 4) || !dims_ok(v, 4) || !dims_ok(bt, 2) || !dims_ok(cu, 1) ||
      !dims_ok(su, 1) || !dims_ok(out, 3))
    return VA_ERR_SHAPE;
  if (q->dtype != VA_BF16 || out->dtype != VA_BF16) return VA_ERR_DTYPE;
  if (k->dtype != VA_FP8_E4M3 && k->dtype != VA_BF16) return VA_ERR_DTYPE;
  if (v->dtype != k->dtype) return VA_ERR_DTYPE;
  if (bt->dtype != VA_INT32 || cu->dtype != VA_INT32 || su->dtype != VA_INT32) return VA_ERR_DTYPE;

  // Shape gate (sglang PR 36330 digest, aiter_backend.py excerpt): head size
  // 256, page size 16, Hk == Hv; Hq % Hkv == 0 (same digest, review notes).
  if (q->shape[2] != kHeadDim || k->shape[3] != kHeadDim) return VA_ERR_UNSUPPORTED;
  if (k->shape[1] != kPageSize) return VA_ERR_UNSUPPORTED;
  for (int i = 0; i < 4; ++i)
    if (v->shape[i] != k->shape[i]) return VA_ERR_SHAPE;
  for (int i = 0; i < 3; ++i)
    if (out->shape[i] != q->shape[i]) return VA_ERR_SHAPE;
  const int64_t hq = q->shape[1], hkv = k->shape[2];
  if (hq < 1 || hkv < 1) return VA_ERR_SHAPE;
  if (hq % hkv != 0) return VA_ERR_SHAPE;
  const int64_t B = su->shape[0];
  if (cu->shape[0] != B + 1 || bt->shape[0] != B) return VA_ERR_SHAPE;
  if (max_seqlen_q < 1 || max_seqlen_k < 0) return VA_ERR_UNSUPPORTED;
  if ((hq / hkv) * (int64_t)max_seqlen_q > kMaxRows) return VA_ERR_UNSUPPORTED;
  if (B > 0 && bt->shape[1] * kPageSize < (int64_t)max_seqlen_k) return VA_ERR_SHAPE;
  if (q->shape[0] > INT32_MAX || k->shape[0] > INT32_MAX || B * hkv > INT32_MAX / 2 ||
      bt->shape[1] > INT32_MAX / kPageSize)
    return VA_ERR_UNSUPPORTED;

  // Layout: innermost stride 1, 16-byte rows (what 16-byte vector and bulk
  // copies need), contiguous index vectors.
  if (!rows_16b(q) || !rows_16b(out) || !rows_16b(k) || !rows_16b(v)) return VA_ERR_LAYOUT;
  if (cu->stride[0] != 1 || su->stride[0] != 1) return VA_ERR_LAYOUT;

  const bool has_q = numel(q) > 0;
  if (has_q && (!q->data || !out->data)) return VA_ERR_NULL;
  if (numel(k) > 0 && (!k->data || !v->data)) return VA_ERR_NULL;
  if (!cu->data) return VA_ERR_NULL;
  if (B > 0 && !su->data) return VA_ERR_NULL;
  if (numel(bt) > 0 && !bt->data) return VA_ERR_NULL;
  if ((q->data && !aligned16(q->data)) || (out->data && !aligned16(out->data)) ||
      (k->data && !aligned16(k->data)) || (v->data && !aligned16(v->data)))
    return VA_ERR_LAYOUT;
  va_status s = check_descale(kd);
  if (s != VA_OK) return s;
  s = check_descale(vd);
  if (s != VA_OK) return s;

  sh->total_q = q->shape[0];
  sh->hq = hq;
  sh->hkv = hkv;
  sh->num_blocks = k->shape[0];
  sh->num_seqs = B;
  sh->width = bt->shape[1];
  sh->kv_dtype = k->dtype;
  return VA_OK;
}

// Upper bound on the key tiles of a batch (B sequences x hkv KV heads of at
// most max_k keys, or of a window of max_q + window_left keys).
static int64_t tiles_upper_bound(int64_t B, int64_t hkv, int32_t max_q, int32_t max_k, int tile,
                                 int32_t window_left) {
  int64_t item_tiles = (max_k + tile - 1) / tile;
  if (window_left >= 0) {  // a window of max_q + window_left keys spans at most this many tiles
    const int64_t w_tiles = ((int64_t)max_q + window_left + tile - 1) / tile + 1;
    if (w_tiles < item_tiles) item_tiles = w_tiles;
  }
  return B * hkv * item_tiles;
}

// The split cost of starting an item (see kPieceCostTiles) for a plan: the
// full cost when CTAs hold many tiles, 1 when the tile bound per CTA is
// small (every CTA then pays a start-up anyway).
static int32_t piece_cost_for(const va_plan& plan, int64_t tiles_bound) {
  return tiles_bound < kSmallSplitTiles * (int64_t)plan.num_splits ? kPieceCostTilesSmall
                                                                    : kPieceCostTiles;
}

va_status make_plan(int64_t B, int64_t hkv, int64_t hq, int32_t max_q, int32_t max_k, int32_t kv_dtype,
                    int32_t num_sms, int32_t force, va_plan* plan, int32_t window_left) {
  if (!plan) return VA_ERR_NULL;
  if (B < 0 || hkv < 1 || hq < 1 || hq % hkv != 0 || max_q < 1 || max_k < 0 || num_sms < 1)
    return VA_ERR_UNSUPPORTED;
  if (kv_dtype != VA_FP8_E4M3 && kv_dtype != VA_BF16) return VA_ERR_UNSUPPORTED;
  const int64_t G = hq / hkv;
  if (G * max_q > kMaxRows) return VA_ERR_UNSUPPORTED;
  const int tile = kv_dtype == VA_FP8_E4M3 ? kTcTileKeysFp8 : kTcTileKeysBf16;
  const int64_t J = B * hkv;
  const int64_t tiles_bound = tiles_upper_bound(B, hkv, max_q, max_k, tile, window_left);
  if (tiles_bound + J * kPieceCostTiles > INT32_MAX / 2) return VA_ERR_UNSUPPORTED;
  // Heuristic: one CTA per SM (the main kernel keeps one CTA per SM), fewer
  // only when the upper-bound workload has fewer tiles than SMs. A CTA's
  // time is its start-up and drain plus its tiles, so spreading a small batch
  // thinly is the lowest-latency choice; the merge that it needs costs a few
  // microseconds.
  constexpr int64_t kMinTiles = 1;
  int64_t splits;
  if (force > 0) {
    splits = force;
    if (splits > tiles_bound) splits = tiles_bound;
  } else {
    splits = (tiles_bound + kMinTiles - 1) / kMinTiles;
    if (splits > num_sms) splits = num_sms;
  }
  if (splits < 1) splits = 1;
  std::memset(plan, 0, sizeof(*plan));
  plan->tile_keys = tile;
  plan->num_splits = (int32_t)splits;
  plan->max_rows = (int32_t)(G * max_q);
  plan->num_work = (int32_t)J;
  // Q in TMEM and the deeper K ring pay off when CTAs stream many tiles; a
  // small batch's CTAs hold a few tiles each, whose latency the single S tile
  // lengthens (gqa_32q2kv: 27.3 against 26.3 us per call)
  plan->kernel = kv_dtype == VA_FP8_E4M3 && window_left < 0 && tiles_bound >= kSmallSplitTiles * splits
                     ? kKernelTcQTmem
                     : kKernelTc;
  plan->workspace_bytes = (int64_t)workspace_layout(J, splits, G * max_q).total;
  return VA_OK;
}

// cuTensorMapEncodeTiled, fetched through the runtime so that the library
// does not link the driver library (it must load on machines without one).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 4-D map over a cache [num_blocks, 16, Hkv, 256]: box = one page of one KV
// head, 128 bytes of the head dim (16 tokens x 128 bytes), 128-byte swizzle,
// so each box lands as two 1 KB swizzle atoms.
static bool make_kv_map(CUtensorMap* m, const va_tensor* t, int64_t nb, int64_t hkv) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const int64_t es_bytes = elem_size(t->dtype);
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv, (cuuint64_t)kPageSize, (cuuint64_t)nb};
  cuuint64_t strides[3] = {(cuuint64_t)(t->stride[2] * es_bytes), (cuuint64_t)(t->stride[1] * es_bytes),
                           (cuuint64_t)(t->stride[0] * es_bytes)};
  cuuint32_t box[4] = {(cuuint32_t)(128 / es_bytes), 1, (cuuint32_t)kPageSize, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      es_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  return fn(m, dt, 4, t->data, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Limit of the main kernels' bounded waits for the next launches; 0 means
// kDefaultWaitLimitNs (see verify_attn_set_wait_limit).
static std::atomic<uint64_t> g_wait_limit_ns{0};

uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : kDefaultWaitLimitNs;
}

struct DeviceState {
  bool ready = false;
  int sms = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

static std::mutex g_mu;
static DeviceState g_dev[kMaxDevices];

// Current device's state, initialised once (SM count, kernel attributes).
// Caller holds g_mu.
static va_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return VA_ERR_UNSUPPORTED;
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return VA_ERR_CUDA;
    if (prepare_main_tc() != cudaSuccess || prepare_mla_tc() != cudaSuccess ||
        prepare_mla_bf16_tc() != cudaSuccess)
      return VA_ERR_CUDA;
    st.ready = true;
  }
  *out = &st;
  return VA_OK;
}

va_status validate_options(const va_options* opts, const Shapes& sh) {
  if (!opts) return VA_OK;
  if (opts->window_left < -1) return VA_ERR_UNSUPPORTED;
  if (!(opts->softcap >= 0.f) || !std::isfinite(opts->softcap)) return VA_ERR_UNSUPPORTED;
  const va_tensor* t = opts->sinks;
  if (t) {
    if (t->dtype != VA_FP32) return VA_ERR_DTYPE;
    if (!dims_ok(t, 1) || t->shape[0] != sh.hq) return VA_ERR_SHAPE;
    if (sh.hq > 1 && t->stride[0] != 1) return VA_ERR_LAYOUT;
    if (!t->data) return VA_ERR_NULL;
  }
  return VA_OK;
}

va_status launch(const va_tensor* q, const va_tensor* k, const va_tensor* v, const va_tensor* bt,
                 const va_tensor* cu, const va_tensor* su, int32_t max_q, int32_t max_k,
                 float scale, const va_tensor* kd, const va_tensor* vd, va_tensor* out,
                 const Shapes& sh, const va_plan& plan, void* ws, size_t ws_bytes,
                 cudaEvent_t ev_mid, cudaStream_t stream, const va_options* opts,
                 const PartialOut* part) {
  if (sh.total_q == 0 || sh.num_seqs == 0) return VA_OK;  // no output rows
  if ((size_t)plan.workspace_bytes > ws_bytes || !ws) return VA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return VA_ERR_WORKSPACE;
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q->data);
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.k = k->data;
  p.k_s0 = k->stride[0];
  p.k_s1 = k->stride[1];
  p.k_s2 = k->stride[2];
  p.v = v->data;
  p.v_s0 = v->stride[0];
  p.v_s1 = v->stride[1];
  p.v_s2 = v->stride[2];
  p.block_table = static_cast<const int32_t*>(bt->data);
  p.bt_s0 = bt->stride[0];
  p.bt_s1 = bt->stride[1];
  p.bt_width = (int32_t)sh.width;
  p.cu_q = static_cast<const int32_t*>(cu->data);
  p.seqused_k = static_cast<const int32_t*>(su->data);
  p.k_descale = kd ? static_cast<const float*>(kd->data) : nullptr;
  p.v_descale = vd ? static_cast<const float*>(vd->data) : nullptr;
  p.out = static_cast<uint16_t*>(out->data);
  p.o_s0 = out->stride[0];
  p.o_s1 = out->stride[1];
  p.out_v8 = (reinterpret_cast<uintptr_t>(out->data) & 31u) == 0 && (p.o_s0 * 2) % 32 == 0 &&
             (p.o_s1 * 2) % 32 == 0;
  p.num_seqs = (int32_t)sh.num_seqs;
  p.hq = (int32_t)sh.hq;
  p.hkv = (int32_t)sh.hkv;
  p.group = (int32_t)(sh.hq / sh.hkv);
  p.num_blocks = (int32_t)sh.num_blocks;
  p.total_q = (int32_t)sh.total_q;
  p.max_seqlen_q = max_q;
  p.max_seqlen_k = max_k;
  p.kv_fp8 = sh.kv_dtype == VA_FP8_E4M3 ? 1 : 0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.window_left = opts ? opts->window_left : -1;
  p.softcap_log2 = opts ? (float)((double)opts->softcap * 1.4426950408889634) : 0.f;
  p.sinks = (opts && opts->sinks) ? static_cast<const float*>(opts->sinks->data) : nullptr;
  p.tile_keys = plan.tile_keys;
  p.num_splits = plan.num_splits;
  p.max_rows = plan.max_rows;
  p.num_work = plan.num_work;
  p.piece_cost = piece_cost_for(
      plan, tiles_upper_bound(sh.num_seqs, sh.hkv, max_q, max_k, plan.tile_keys, p.window_left));
  p.q_in_tmem = plan.kernel == kKernelTcQTmem ? 1 : 0;
  p.dv = kHeadDim;
  p.wait_limit_ns = wait_limit_ns();
  if (part) {
    p.partial = 1;
    p.kv_extent = part->kv_extent ? static_cast<const int32_t*>(part->kv_extent->data) : nullptr;
    p.o_part = static_cast<float*>(part->o->data);
    p.op_s0 = part->o->stride[0];
    p.op_s1 = part->o->stride[1];
    p.lse_part = static_cast<float*>(part->lse->data);
    p.lse_s0 = part->lse->stride[0];
    p.lse_s1 = part->lse->stride[1];
  }
  const WorkspaceLayout lay = workspace_layout(plan.num_work, plan.num_splits, plan.max_rows);
  char* base = static_cast<char*>(ws);
  p.ws_meta = reinterpret_cast<int32_t*>(base + lay.meta_off);
  p.ws_ml = reinterpret_cast<float*>(base + lay.ml_off);
  p.ws_acc = reinterpret_cast<float*>(base + lay.acc_off);
  p.ws_status = reinterpret_cast<int32_t*>(base + lay.status_off);
  CUtensorMap tm_k, tm_v;
  std::memset(&tm_k, 0, sizeof(tm_k));
  std::memset(&tm_v, 0, sizeof(tm_v));
  if (sh.num_blocks > 0) {  // an empty cache has no page to load
    if (!make_kv_map(&tm_k, k, sh.num_blocks, sh.hkv) || !make_kv_map(&tm_v, v, sh.num_blocks, sh.hkv))
      return VA_ERR_LAYOUT;
  }
  if (launch_main_tc(p, tm_k, tm_v, stream) != cudaSuccess) return VA_ERR_CUDA;
  if (ev_mid && cudaEventRecord(ev_mid, stream) != cudaSuccess) return VA_ERR_CUDA;
  if (launch_merge(p, stream) != cudaSuccess) return VA_ERR_CUDA;
  return VA_OK;
}

// ---- absorbed-MLA latent cache ------------------------------------------------

va_status validate_mla(const va_tensor* q, const va_tensor* kv, const va_tensor* bt,
                       const va_tensor* cu, const va_tensor* su, int32_t max_seqlen_q,
                       int32_t max_seqlen_k, const va_tensor* kd, const va_tensor* vd,
                       const va_tensor* out, Shapes* sh) {
  if (!q || !kv || !bt || !cu || !su || !out) return VA_ERR_NULL;
  if (!dims_ok(q, 3) || !dims_ok(kv, 4) || !dims_ok(bt, 2) || !dims_ok(cu, 1) || !dims_ok(su, 1) ||
      !dims_ok(out, 3))
    return VA_ERR_SHAPE;
  if (q->dtype != VA_BF16 || out->dtype != VA_BF16) return VA_ERR_DTYPE;
  if (kv->dtype != VA_FP8_E4M3 && kv->dtype != VA_BF16) return VA_ERR_DTYPE;
  if (bt->dtype != VA_INT32 || cu->dtype != VA_INT32 || su->dtype != VA_INT32) return VA_ERR_DTYPE;
  // one latent KV head (the digest's k_extend.shape[1] != 1 rejection), rows
  // [latent | rope]; FP8 E4M3 or BF16
  if (kv->shape[1] != kPageSize || kv->shape[2] != 1 || kv->shape[3] != kMlaRow) return VA_ERR_UNSUPPORTED;
  if (q->shape[2] != kMlaRow || out->shape[2] != kMlaNope) return VA_ERR_UNSUPPORTED;
  if (out->shape[0] != q->shape[0] || out->shape[1] != q->shape[1]) return VA_ERR_SHAPE;
  const int64_t hq = q->shape[1];
  if (hq < 1) return VA_ERR_SHAPE;
  const int64_t B = su->shape[0];
  if (cu->shape[0] != B + 1 || bt->shape[0] != B) return VA_ERR_SHAPE;
  if (max_seqlen_q < 1 || max_seqlen_k < 0) return VA_ERR_UNSUPPORTED;
  if (hq * (int64_t)max_seqlen_q > kMaxRows) return VA_ERR_UNSUPPORTED;
  if (B > 0 && bt->shape[1] * kPageSize < (int64_t)max_seqlen_k) return VA_ERR_SHAPE;
  if (q->shape[0] > INT32_MAX || kv->shape[0] > INT32_MAX || B > INT32_MAX / 2 ||
      bt->shape[1] > INT32_MAX / kPageSize)
    return VA_ERR_UNSUPPORTED;
  if (!rows_16b(q) || !rows_16b(out) || !rows_16b(kv)) return VA_ERR_LAYOUT;
  if (cu->stride[0] != 1 || su->stride[0] != 1) return VA_ERR_LAYOUT;
  if (numel(q) > 0 && (!q->data || !out->data)) return VA_ERR_NULL;
  if (numel(kv) > 0 && !kv->data) return VA_ERR_NULL;
  if (!cu->data) return VA_ERR_NULL;
  if (B > 0 && !su->data) return VA_ERR_NULL;
  if (numel(bt) > 0 && !bt->data) return VA_ERR_NULL;
  if ((q->data && !aligned16(q->data)) || (out->data && !aligned16(out->data)) ||
      (kv->data && !aligned16(kv->data)))
    return VA_ERR_LAYOUT;
  va_status s = check_descale(kd);
  if (s != VA_OK) return s;
  s = check_descale(vd);
  if (s != VA_OK) return s;
  sh->total_q = q->shape[0];
  sh->hq = hq;
  sh->hkv = 1;
  sh->num_blocks = kv->shape[0];
  sh->num_seqs = B;
  sh->width = bt->shape[1];
  sh->kv_dtype = kv->dtype;
  return VA_OK;
}

// The split heuristic of make_plan on latent tiles (64 keys for an FP8 cache,
// 32 for BF16), value width 512.
va_status make_mla_plan(int64_t B, int64_t hq, int32_t max_q, int32_t max_k, int32_t num_sms,
                        int32_t force, va_plan* plan, int32_t kv_dtype) {
  if (!plan) return VA_ERR_NULL;
  if (B < 0 || hq < 1 || max_q < 1 || max_k < 0 || num_sms < 1) return VA_ERR_UNSUPPORTED;
  if (kv_dtype != VA_FP8_E4M3 && kv_dtype != VA_BF16) return VA_ERR_UNSUPPORTED;
  if (hq * max_q > kMaxRows) return VA_ERR_UNSUPPORTED;
  const int tile = kv_dtype == VA_FP8_E4M3 ? kMlaTileKeys : kMlaTileKeysBf16;
  const int cost = kv_dtype == VA_FP8_E4M3 ? kMlaPieceCostTiles : kMlaPieceCostTilesBf16;
  const int64_t item_tiles = ((int64_t)max_k + tile - 1) / tile;
  const int64_t tiles_bound = B * item_tiles;
  if (tiles_bound + B * cost > INT32_MAX / 2) return VA_ERR_UNSUPPORTED;
  int64_t splits = force > 0 ? force : num_sms;
  if (splits > tiles_bound) splits = tiles_bound;
  if (splits < 1) splits = 1;
  std::memset(plan, 0, sizeof(*plan));
  plan->tile_keys = tile;
  plan->num_splits = (int32_t)splits;
  plan->max_rows = (int32_t)(hq * max_q);
  plan->num_work = (int32_t)B;
  plan->kernel = kKernelTc;
  // the partials' rows are padded to mla_row_stride; the layout is sized with
  // that row count (launch_mla takes the same offsets)
  plan->workspace_bytes =
      (int64_t)workspace_layout(B, splits, mla_row_stride((int)(hq * max_q)), kMlaNope).total;
  return VA_OK;
}

// 4-D map over a latent cache [num_blocks, 16, 1, 576]: box = one page, 128
// bytes of the row, 128-byte swizzle. For e4m3 the box at column 512 holds the
// 64 rope bytes, its other 64 lie past the row end and are zero-filled; a
// bf16 row is nine whole boxes of 64 elements.
// Box: 128 bytes of one row (a latent chunk, 128-byte swizzle), or with
// `rope` the row's 64 rope bytes (64-byte swizzle), x 16 page rows.
static bool make_mla_map(CUtensorMap* m, const va_tensor* t, int64_t nb, bool rope = false) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t es_bytes = (cuuint64_t)elem_size(t->dtype);
  cuuint64_t dims[4] = {(cuuint64_t)kMlaRow, 1, (cuuint64_t)kPageSize, (cuuint64_t)nb};
  cuuint64_t strides[3] = {(cuuint64_t)t->stride[2] * es_bytes, (cuuint64_t)t->stride[1] * es_bytes,
                           (cuuint64_t)t->stride[0] * es_bytes};
  if (strides[0] == 0 || strides[0] % 16 != 0) strides[0] = (cuuint64_t)kMlaRow * es_bytes;  // one head: unused
  cuuint32_t box[4] = {(cuuint32_t)((rope ? 64 : 128) / es_bytes), 1, (cuuint32_t)kPageSize, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = es_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  return fn(m, dt, 4, t->data, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            rope ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

va_status launch_mla(const va_tensor* q, const va_tensor* kv, const va_tensor* bt, const va_tensor* cu,
                     const va_tensor* su, int32_t max_q, int32_t max_k, float scale,
                     const va_tensor* kd, const va_tensor* vd, va_tensor* out, const Shapes& sh,
                     const va_plan& plan, void* ws, size_t ws_bytes, cudaEvent_t ev_mid,
                     cudaStream_t stream) {
  if (sh.total_q == 0 || sh.num_seqs == 0) return VA_OK;
  if ((size_t)plan.workspace_bytes > ws_bytes || !ws) return VA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return VA_ERR_WORKSPACE;
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q->data);
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.k = p.v = kv->data;
  p.k_s0 = p.v_s0 = kv->stride[0];
  p.k_s1 = p.v_s1 = kv->stride[1];
  p.k_s2 = p.v_s2 = kv->stride[2];
  p.block_table = static_cast<const int32_t*>(bt->data);
  p.bt_s0 = bt->stride[0];
  p.bt_s1 = bt->stride[1];
  p.bt_width = (int32_t)sh.width;
  p.cu_q = static_cast<const int32_t*>(cu->data);
  p.seqused_k = static_cast<const int32_t*>(su->data);
  p.k_descale = kd ? static_cast<const float*>(kd->data) : nullptr;
  p.v_descale = vd ? static_cast<const float*>(vd->data) : nullptr;
  p.out = static_cast<uint16_t*>(out->data);
  p.o_s0 = out->stride[0];
  p.o_s1 = out->stride[1];
  p.num_seqs = (int32_t)sh.num_seqs;
  p.hq = (int32_t)sh.hq;
  p.hkv = 1;
  p.group = (int32_t)sh.hq;
  p.num_blocks = (int32_t)sh.num_blocks;
  p.total_q = (int32_t)sh.total_q;
  p.max_seqlen_q = max_q;
  p.max_seqlen_k = max_k;
  p.kv_fp8 = sh.kv_dtype == VA_FP8_E4M3 ? 1 : 0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.window_left = -1;
  p.tile_keys = plan.tile_keys;
  p.num_splits = plan.num_splits;
  p.max_rows = plan.max_rows;
  p.num_work = plan.num_work;
  p.piece_cost = p.kv_fp8 ? kMlaPieceCostTiles : kMlaPieceCostTilesBf16;
  p.dv = kMlaNope;
  p.wait_limit_ns = wait_limit_ns();
  const WorkspaceLayout lay =
      workspace_layout(plan.num_work, plan.num_splits, mla_row_stride(plan.max_rows), kMlaNope);
  char* base = static_cast<char*>(ws);
  p.ws_status = reinterpret_cast<int32_t*>(base + lay.status_off);
  p.ws_meta = reinterpret_cast<int32_t*>(base + lay.meta_off);
  p.ws_ml = reinterpret_cast<float*>(base + lay.ml_off);
  p.ws_acc = reinterpret_cast<float*>(base + lay.acc_off);
  CUtensorMap tm, tm_pe;
  std::memset(&tm, 0, sizeof(tm));
  std::memset(&tm_pe, 0, sizeof(tm_pe));
  if (sh.num_blocks > 0 && !make_mla_map(&tm, kv, sh.num_blocks)) return VA_ERR_LAYOUT;
  if (sh.num_blocks > 0 && p.kv_fp8 && !make_mla_map(&tm_pe, kv, sh.num_blocks, true)) return VA_ERR_LAYOUT;
  if ((p.kv_fp8 ? launch_mla_tc(p, tm, tm_pe, stream) : launch_mla_bf16_tc(p, tm, stream)) != cudaSuccess)
    return VA_ERR_CUDA;
  if (ev_mid && cudaEventRecord(ev_mid, stream) != cudaSuccess) return VA_ERR_CUDA;
  if (launch_merge(p, stream) != cudaSuccess) return VA_ERR_CUDA;
  return VA_OK;
}

// The library's per-device workspace, grown to `bytes` if smaller. Grow only:
// cudaFree waits for work already queued on the old buffer. A new buffer's
// status word is zeroed on the caller's stream (the rest needs no clearing).
// Caller holds g_mu.
static va_status library_workspace(DeviceState* st, size_t bytes, cudaStream_t stream) {
  if (bytes <= st->ws_bytes) return VA_OK;
  if (st->ws) cudaFree(st->ws);
  st->ws = nullptr;
  st->ws_bytes = 0;
  if (cudaMalloc(&st->ws, bytes) != cudaSuccess) {
    st->ws = nullptr;
    return VA_ERR_CUDA;
  }
  if (cudaMemsetAsync(st->ws, 0, 256, stream) != cudaSuccess) return VA_ERR_CUDA;
  st->ws_bytes = bytes;
  return VA_OK;
}

va_status current_device_sms(int* sms) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  const va_status s = device_state(&st);
  if (s == VA_OK) *sms = st->sms;
  return s;
}

}  // namespace va_host_impl

using namespace va_host_impl;

VA_EXPORT va_status verify_attn_check(const va_tensor* q, const va_tensor* k_cache,
                                      const va_tensor* v_cache, const va_tensor* block_table,
                                      const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                                      int32_t max_seqlen_q, int32_t max_seqlen_k,
                                      const va_tensor* k_descale, const va_tensor* v_descale,
                                      const va_tensor* out) {
  Shapes sh;
  return validate(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                  max_seqlen_k, k_descale, v_descale, out, &sh);
}

VA_EXPORT va_status verify_attn_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t kv_dtype,
                                     int32_t num_sms, int32_t force_splits, va_plan* plan) {
  return make_plan(num_seqs, num_kv_heads, num_q_heads, max_seqlen_q, max_seqlen_k, kv_dtype,
                   num_sms, force_splits, plan);
}

VA_EXPORT size_t verify_attn_workspace_size(int32_t num_seqs, int32_t num_kv_heads,
                                            int32_t num_q_heads, int32_t max_seqlen_q,
                                            int32_t max_seqlen_k, int32_t kv_dtype,
                                            int32_t num_splits) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  if (device_state(&st) != VA_OK) return 0;
  va_plan plan;
  if (make_plan(num_seqs, num_kv_heads, num_q_heads, max_seqlen_q, max_seqlen_k, kv_dtype, st->sms,
                num_splits, &plan) != VA_OK)
    return 0;
  return (size_t)plan.workspace_bytes;
}

// Shared body of verify_attn, verify_attn_ex and verify_attn_opt. A NULL
// workspace with own_ws uses (and grows) the library's per-device workspace.
static va_status run_call(const va_tensor* q, const va_tensor* k_cache, const va_tensor* v_cache,
                          const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                          const va_tensor* seqused_k, int32_t max_seqlen_q, int32_t max_seqlen_k,
                          float softmax_scale, const va_tensor* k_descale,
                          const va_tensor* v_descale, va_tensor* out, const va_options* opts,
                          void* workspace, size_t workspace_bytes, bool own_ws, int32_t num_splits,
                          cudaEvent_t ev_mid, cudaStream_t stream) {
  Shapes sh;
  va_status s = validate(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                         max_seqlen_k, k_descale, v_descale, out, &sh);
  if (s != VA_OK) return s;
  s = validate_options(opts, sh);
  if (s != VA_OK) return s;
  if (num_splits < 0) return VA_ERR_UNSUPPORTED;
  std::unique_lock<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != VA_OK) return s;
  va_plan plan;
  s = make_plan(sh.num_seqs, sh.hkv, sh.hq, max_seqlen_q, max_seqlen_k, sh.kv_dtype, st->sms,
                num_splits, &plan, opts ? opts->window_left : -1);
  if (s != VA_OK) return s;
  if (own_ws) {
    if (sh.total_q == 0 || sh.num_seqs == 0) return VA_OK;
    s = library_workspace(st, (size_t)plan.workspace_bytes, stream);
    if (s != VA_OK) return s;
    workspace = st->ws;
    workspace_bytes = st->ws_bytes;
  } else {
    lk.unlock();
  }
  return launch(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                max_seqlen_k, softmax_scale, k_descale, v_descale, out, sh, plan, workspace,
                workspace_bytes, ev_mid, stream, opts);
}

VA_EXPORT va_status verify_attn_ex(const va_tensor* q, const va_tensor* k_cache,
                                   const va_tensor* v_cache, const va_tensor* block_table,
                                   const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                                   int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                                   const va_tensor* k_descale, const va_tensor* v_descale,
                                   va_tensor* out, void* workspace, size_t workspace_bytes,
                                   int32_t num_splits, void* event_after_main, void* stream) {
  return run_call(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                  max_seqlen_k, softmax_scale, k_descale, v_descale, out, nullptr, workspace,
                  workspace_bytes, false, num_splits, static_cast<cudaEvent_t>(event_after_main),
                  static_cast<cudaStream_t>(stream));
}

VA_EXPORT va_status verify_attn(const va_tensor* q, const va_tensor* k_cache,
                                const va_tensor* v_cache, const va_tensor* block_table,
                                const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                                int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                                const va_tensor* k_descale, const va_tensor* v_descale,
                                va_tensor* out, void* stream) {
  return run_call(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                  max_seqlen_k, softmax_scale, k_descale, v_descale, out, nullptr, nullptr, 0, true,
                  0, nullptr, static_cast<cudaStream_t>(stream));
}

VA_EXPORT va_status verify_attn_opt(const va_tensor* q, const va_tensor* k_cache,
                                    const va_tensor* v_cache, const va_tensor* block_table,
                                    const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                                    const va_tensor* k_descale, const va_tensor* v_descale,
                                    va_tensor* out, const va_options* opts, void* workspace,
                                    size_t workspace_bytes, int32_t num_splits, void* stream) {
  return run_call(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                  max_seqlen_k, softmax_scale, k_descale, v_descale, out, opts, workspace,
                  workspace_bytes, workspace == nullptr, num_splits, nullptr,
                  static_cast<cudaStream_t>(stream));
}

// Descriptor checks of verify_attn_block_table_from_indptr (host only).
static va_status validate_block_table_args(const va_tensor* indptr, const va_tensor* indices,
                                           const va_tensor* bt, const va_tensor* seqused) {
  if (!indptr || !indices || !bt || !seqused) return VA_ERR_NULL;
  if (indptr->dtype != VA_INT32 || indices->dtype != VA_INT32 || bt->dtype != VA_INT32 ||
      seqused->dtype != VA_INT32)
    return VA_ERR_DTYPE;
  if (!dims_ok(indptr, 1) || !dims_ok(indices, 1) || !dims_ok(bt, 2) || !dims_ok(seqused, 1))
    return VA_ERR_SHAPE;
  const int64_t B = indptr->shape[0] - 1;
  if (B < 0 || bt->shape[0] != B || seqused->shape[0] != B) return VA_ERR_SHAPE;
  if (B > 65535 || bt->shape[1] > INT32_MAX || indices->shape[0] > INT32_MAX)
    return VA_ERR_UNSUPPORTED;
  if ((B + 1 > 1 && indptr->stride[0] != 1) || (indices->shape[0] > 1 && indices->stride[0] != 1))
    return VA_ERR_LAYOUT;
  if (!indptr->data) return VA_ERR_NULL;
  if (B > 0 && (!seqused->data || (bt->shape[1] > 0 && !bt->data))) return VA_ERR_NULL;
  if (indices->shape[0] > 0 && !indices->data) return VA_ERR_NULL;
  return VA_OK;
}

VA_EXPORT va_status verify_attn_block_table_from_indptr(const va_tensor* kv_indptr,
                                                        const va_tensor* kv_indices,
                                                        va_tensor* block_table, va_tensor* seqused_k,
                                                        int32_t pad_page, int32_t* status,
                                                        void* stream) {
  const va_status v = validate_block_table_args(kv_indptr, kv_indices, block_table, seqused_k);
  if (v != VA_OK) return v;
  const cudaError_t e = va::launch_block_table(
      static_cast<const int32_t*>(kv_indptr->data), static_cast<const int32_t*>(kv_indices->data),
      kv_indices->shape[0], (int32_t)(kv_indptr->shape[0] - 1), (int32_t)block_table->shape[1],
      static_cast<int32_t*>(block_table->data), block_table->stride[0], block_table->stride[1],
      static_cast<int32_t*>(seqused_k->data), seqused_k->stride[0], pad_page, status,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VA_OK : VA_ERR_CUDA;
}

VA_EXPORT va_status verify_attn_mla(const va_tensor* q, const va_tensor* kv_cache,
                                    const va_tensor* block_table, const va_tensor* cu_seqlens_q,
                                    const va_tensor* seqused_k, int32_t max_seqlen_q,
                                    int32_t max_seqlen_k, float softmax_scale,
                                    const va_tensor* k_descale, const va_tensor* v_descale,
                                    va_tensor* out, void* workspace, size_t workspace_bytes,
                                    int32_t num_splits, void* event_after_main, void* stream) {
  Shapes sh;
  va_status s = validate_mla(q, kv_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                             max_seqlen_k, k_descale, v_descale, out, &sh);
  if (s != VA_OK) return s;
  if (num_splits < 0) return VA_ERR_UNSUPPORTED;
  std::unique_lock<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != VA_OK) return s;
  va_plan plan;
  s = make_mla_plan(sh.num_seqs, sh.hq, max_seqlen_q, max_seqlen_k, st->sms, num_splits, &plan, sh.kv_dtype);
  if (s != VA_OK) return s;
  if (!workspace) {
    if (sh.total_q == 0 || sh.num_seqs == 0) return VA_OK;
    s = library_workspace(st, (size_t)plan.workspace_bytes, static_cast<cudaStream_t>(stream));
    if (s != VA_OK) return s;
    workspace = st->ws;
    workspace_bytes = st->ws_bytes;
  } else {
    lk.unlock();
  }
  return launch_mla(q, kv_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q, max_seqlen_k,
                    softmax_scale, k_descale, v_descale, out, sh, plan, workspace, workspace_bytes,
                    static_cast<cudaEvent_t>(event_after_main), static_cast<cudaStream_t>(stream));
}

VA_EXPORT size_t verify_attn_mla_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                int32_t max_seqlen_q, int32_t max_seqlen_k,
                                                int32_t num_splits) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  if (device_state(&st) != VA_OK) return 0;
  // enough for either cache dtype (their tiles, and so their splits, differ)
  size_t bytes = 0;
  for (int32_t dt : {(int32_t)VA_FP8_E4M3, (int32_t)VA_BF16}) {
    va_plan plan;
    if (make_mla_plan(num_seqs, num_q_heads, max_seqlen_q, max_seqlen_k, st->sms, num_splits, &plan, dt) !=
        VA_OK)
      return 0;
    if ((size_t)plan.workspace_bytes > bytes) bytes = (size_t)plan.workspace_bytes;
  }
  return bytes;
}

// ---- one shard of each sequence's keys, and the merge of shards ---------------

// Checks of verify_attn_partial's own arguments (the rest as verify_attn).
static va_status validate_partial_outputs(const va_tensor* ext, const va_tensor* o,
                                          const va_tensor* lse, const Shapes& sh) {
  if (!o || !lse) return VA_ERR_NULL;
  if (o->dtype != VA_FP32 || lse->dtype != VA_FP32) return VA_ERR_DTYPE;
  if (!dims_ok(o, 3) || !dims_ok(lse, 2)) return VA_ERR_SHAPE;
  if (o->shape[0] != sh.total_q || o->shape[1] != sh.hq || o->shape[2] != kHeadDim) return VA_ERR_SHAPE;
  if (lse->shape[0] != sh.total_q || lse->shape[1] != sh.hq) return VA_ERR_SHAPE;
  if (!rows_16b(o)) return VA_ERR_LAYOUT;
  if (sh.total_q > 0 && (!o->data || !lse->data)) return VA_ERR_NULL;
  if ((o->data && !aligned16(o->data)) || (lse->data && (reinterpret_cast<uintptr_t>(lse->data) & 3u)))
    return VA_ERR_LAYOUT;
  if (ext) {
    if (ext->dtype != VA_INT32) return VA_ERR_DTYPE;
    if (!dims_ok(ext, 1) || ext->shape[0] != sh.num_seqs) return VA_ERR_SHAPE;
    if (sh.num_seqs > 1 && ext->stride[0] != 1) return VA_ERR_LAYOUT;
    if (sh.num_seqs > 0 && !ext->data) return VA_ERR_NULL;
  }
  return VA_OK;
}

VA_EXPORT va_status verify_attn_partial(const va_tensor* q, const va_tensor* k_cache,
                                        const va_tensor* v_cache, const va_tensor* block_table,
                                        const va_tensor* cu_seqlens_q, const va_tensor* seqused_k,
                                        const va_tensor* kv_extent, int32_t max_seqlen_q,
                                        int32_t max_seqlen_k, float softmax_scale,
                                        const va_tensor* k_descale, const va_tensor* v_descale,
                                        va_tensor* o, va_tensor* lse, void* workspace,
                                        size_t workspace_bytes, int32_t num_splits, void* stream) {
  // q stands in for the bf16 out that validate() checks: the shard writes o and lse
  Shapes sh;
  va_status s = validate(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                         max_seqlen_k, k_descale, v_descale, q, &sh);
  if (s != VA_OK) return s;
  s = validate_partial_outputs(kv_extent, o, lse, sh);
  if (s != VA_OK) return s;
  if (num_splits < 0) return VA_ERR_UNSUPPORTED;
  std::unique_lock<std::mutex> lk(g_mu);
  DeviceState* st = nullptr;
  s = device_state(&st);
  if (s != VA_OK) return s;
  va_plan plan;
  s = make_plan(sh.num_seqs, sh.hkv, sh.hq, max_seqlen_q, max_seqlen_k, sh.kv_dtype, st->sms,
                num_splits, &plan);
  if (s != VA_OK) return s;
  if (!workspace) {
    if (sh.total_q == 0 || sh.num_seqs == 0) return VA_OK;
    s = library_workspace(st, (size_t)plan.workspace_bytes, static_cast<cudaStream_t>(stream));
    if (s != VA_OK) return s;
    workspace = st->ws;
    workspace_bytes = st->ws_bytes;
  } else {
    lk.unlock();
  }
  const PartialOut part{kv_extent, o, lse};
  va_tensor unused_out = *q;  // no piece writes bf16 rows in partial mode
  return launch(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q,
                max_seqlen_k, softmax_scale, k_descale, v_descale, &unused_out, sh, plan, workspace,
                workspace_bytes, nullptr, static_cast<cudaStream_t>(stream), nullptr, &part);
}

VA_EXPORT va_status verify_attn_merge_partials(int32_t n, const va_tensor* o_parts,
                                               const va_tensor* lse_parts, va_tensor* out,
                                               void* stream) {
  if (!o_parts || !lse_parts || !out) return VA_ERR_NULL;
  if (n < 1 || n > kMaxShards) return VA_ERR_UNSUPPORTED;
  if (out->dtype != VA_BF16) return VA_ERR_DTYPE;
  if (!dims_ok(out, 3) || out->shape[2] != kHeadDim) return VA_ERR_SHAPE;
  if (!rows_16b(out)) return VA_ERR_LAYOUT;
  if (out->shape[0] > INT32_MAX || out->shape[1] > INT32_MAX) return VA_ERR_UNSUPPORTED;
  ShardMergeParams m;
  std::memset(&m, 0, sizeof(m));
  m.n = n;
  m.total_q = (int32_t)out->shape[0];
  m.hq = (int32_t)out->shape[1];
  const bool any = m.total_q > 0 && m.hq > 0;
  if (any && (!out->data || !aligned16(out->data))) return out->data ? VA_ERR_LAYOUT : VA_ERR_NULL;
  m.out = static_cast<uint16_t*>(out->data);
  m.out_s0 = out->stride[0];
  m.out_s1 = out->stride[1];
  for (int i = 0; i < n; ++i) {
    const va_tensor* o = &o_parts[i];
    const va_tensor* l = &lse_parts[i];
    if (o->dtype != VA_FP32 || l->dtype != VA_FP32) return VA_ERR_DTYPE;
    if (!dims_ok(o, 3) || !dims_ok(l, 2)) return VA_ERR_SHAPE;
    for (int d = 0; d < 3; ++d)
      if (o->shape[d] != out->shape[d]) return VA_ERR_SHAPE;
    if (l->shape[0] != out->shape[0] || l->shape[1] != out->shape[1]) return VA_ERR_SHAPE;
    if (!rows_16b(o)) return VA_ERR_LAYOUT;
    if (any && (!o->data || !l->data)) return VA_ERR_NULL;
    if (any && (!aligned16(o->data) || (reinterpret_cast<uintptr_t>(l->data) & 3u))) return VA_ERR_LAYOUT;
    m.o[i] = static_cast<const float*>(o->data);
    m.o_s0[i] = o->stride[0];
    m.o_s1[i] = o->stride[1];
    m.lse[i] = static_cast<const float*>(l->data);
    m.lse_s0[i] = l->stride[0];
    m.lse_s1[i] = l->stride[1];
  }
  return launch_merge_shards(m, static_cast<cudaStream_t>(stream)) == cudaSuccess ? VA_OK : VA_ERR_CUDA;
}

VA_EXPORT va_status verify_attn_set_wait_limit(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  return VA_OK;
}

// Reads the status word at `word` after the work queued on `stream`, ORs it
// into *bits and queues its clearing.
static va_status take_status(void* word, int32_t* bits, cudaStream_t stream) {
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return VA_ERR_CUDA;
  *bits |= v;
  if (v != 0 && cudaMemsetAsync(word, 0, sizeof(v), stream) != cudaSuccess) return VA_ERR_CUDA;
  return VA_OK;
}

VA_EXPORT va_status verify_attn_last_device_error(const void* workspace, int32_t* bits, void* stream) {
  if (!bits) return VA_ERR_NULL;
  *bits = 0;
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return VA_ERR_WORKSPACE;
    return take_status(const_cast<void*>(workspace), bits, st_);
  }
  void* lib_ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = nullptr;
    const va_status s = device_state(&st);
    if (s != VA_OK) return s;
    lib_ws = st->ws;
  }
  if (lib_ws) {
    const va_status s = take_status(lib_ws, bits, st_);
    if (s != VA_OK) return s;
  }
  void* scratch = nullptr;
  va_status s = noalloc_scratch(&scratch, false);
  if (s != VA_OK) return s;
  if (scratch) s = take_status(scratch, bits, st_);
  return s;
}

VA_EXPORT const char* verify_attn_status_string(int32_t status) {
  switch (status) {
    case VA_OK: return "VA_OK";
    case VA_ERR_NULL: return "VA_ERR_NULL: a required pointer or descriptor is NULL";
    case VA_ERR_SHAPE: return "VA_ERR_SHAPE: tensor shapes disagree";
    case VA_ERR_DTYPE: return "VA_ERR_DTYPE: wrong element type";
    case VA_ERR_UNSUPPORTED: return "VA_ERR_UNSUPPORTED: outside what the kernels cover";
    case VA_ERR_WORKSPACE: return "VA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case VA_ERR_CUDA: return "VA_ERR_CUDA: a CUDA call or launch failed";
    case VA_ERR_LAYOUT: return "VA_ERR_LAYOUT: unsupported stride or alignment";
    default: return "unknown va_status";
  }
}
