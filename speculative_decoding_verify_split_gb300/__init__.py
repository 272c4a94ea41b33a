"""Python binding of the verify-attention C-ABI library (``include/verify_attn.h``).

Argument marshalling only: torch tensors become ``va_tensor`` descriptors
(device pointer, dtype code, shape, strides) and the call goes to the native
library, which runs every step in its own CUDA kernels. There is no Python or
CPU fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libverify_attn.so")

VA_BF16, VA_FP8_E4M3, VA_INT32, VA_FP32 = 0, 1, 2, 3
VA_OK = 0
STATUS_NAMES = {0: "VA_OK", 1: "VA_ERR_NULL", 2: "VA_ERR_SHAPE", 3: "VA_ERR_DTYPE",
                4: "VA_ERR_UNSUPPORTED", 5: "VA_ERR_WORKSPACE", 6: "VA_ERR_CUDA",
                7: "VA_ERR_LAYOUT"}

_DTYPES = {torch.bfloat16: VA_BF16, torch.float8_e4m3fn: VA_FP8_E4M3,
           torch.int32: VA_INT32, torch.float32: VA_FP32}

# Every symbol include/verify_attn.h declares.
EXPORTS = ("verify_attn", "verify_attn_ex", "verify_attn_check", "verify_attn_plan",
           "verify_attn_workspace_size", "verify_attn_status_string", "verify_attn_noalloc",
           "verify_attn_block_table_from_indptr", "verify_attn_opt", "verify_attn_mla",
           "verify_attn_mla_workspace_size", "verify_attn_partial", "verify_attn_merge_partials",
           "verify_attn_last_device_error", "verify_attn_set_wait_limit")

# Absorbed-MLA latent cache: row = [latent (MLA_NOPE) | rope key (MLA_PE)].
MLA_NOPE, MLA_PE = 512, 64

# Status bits of verify_attn_block_table_from_indptr.
BT_BAD_PAGE, BT_TRUNCATED, BT_BAD_INDPTR = 1, 2, 4

# Size of the library's built-in partials array used by verify_attn_noalloc.
NOALLOC_SCRATCH_BYTES = 16 << 20


class VaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class VaPlan(ctypes.Structure):
    _fields_ = [("tile_keys", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("max_rows", ctypes.c_int32), ("num_work", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64)]


class VaOptions(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int32), ("softcap", ctypes.c_float),
                ("sinks", ctypes.POINTER(VaTensor))]


class VerifyAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({_lib().verify_attn_status_string(status).decode()})")


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"native library not built: {LIB_PATH} is missing "
                               "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(VaTensor)
        tens = [P] * 6 + [ctypes.c_int32, ctypes.c_int32]
        lib.verify_attn.argtypes = tens + [ctypes.c_float, P, P, P, ctypes.c_void_p]
        lib.verify_attn.restype = ctypes.c_int32
        lib.verify_attn_ex.argtypes = tens + [ctypes.c_float, P, P, P, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_void_p]
        lib.verify_attn_ex.restype = ctypes.c_int32
        lib.verify_attn_check.argtypes = tens + [P, P, P]
        lib.verify_attn_check.restype = ctypes.c_int32
        lib.verify_attn_plan.argtypes = [ctypes.c_int32] * 8 + [ctypes.POINTER(VaPlan)]
        lib.verify_attn_plan.restype = ctypes.c_int32
        lib.verify_attn_workspace_size.argtypes = [ctypes.c_int32] * 7
        lib.verify_attn_workspace_size.restype = ctypes.c_size_t
        lib.verify_attn_noalloc.argtypes = tens + [ctypes.c_float, P, P, P, ctypes.c_void_p]
        lib.verify_attn_noalloc.restype = ctypes.c_int32
        lib.verify_attn_block_table_from_indptr.argtypes = [P, P, P, P, ctypes.c_int32,
                                                            ctypes.c_void_p, ctypes.c_void_p]
        lib.verify_attn_block_table_from_indptr.restype = ctypes.c_int32
        lib.verify_attn_opt.argtypes = tens + [ctypes.c_float, P, P, P, ctypes.POINTER(VaOptions),
                                               ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                               ctypes.c_void_p]
        lib.verify_attn_opt.restype = ctypes.c_int32
        lib.verify_attn_mla.argtypes = [P] * 5 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                  P, P, P, ctypes.c_void_p, ctypes.c_size_t,
                                                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.verify_attn_mla.restype = ctypes.c_int32
        lib.verify_attn_mla_workspace_size.argtypes = [ctypes.c_int32] * 5
        lib.verify_attn_mla_workspace_size.restype = ctypes.c_size_t
        lib.verify_attn_partial.argtypes = [P] * 7 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                                      P, P, P, P, ctypes.c_void_p, ctypes.c_size_t,
                                                      ctypes.c_int32, ctypes.c_void_p]
        lib.verify_attn_partial.restype = ctypes.c_int32
        lib.verify_attn_merge_partials.argtypes = [ctypes.c_int32, P, P, P, ctypes.c_void_p]
        lib.verify_attn_merge_partials.restype = ctypes.c_int32
        lib.verify_attn_last_device_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                                      ctypes.c_void_p]
        lib.verify_attn_last_device_error.restype = ctypes.c_int32
        lib.verify_attn_set_wait_limit.argtypes = [ctypes.c_uint64]
        lib.verify_attn_set_wait_limit.restype = ctypes.c_int32
        lib.verify_attn_status_string.argtypes = [ctypes.c_int32]
        lib.verify_attn_status_string.restype = ctypes.c_char_p
        _LIB = lib
    return _LIB


def library():
    """The loaded ctypes library (raises if it was not built)."""
    return _lib()


def desc(t: Optional[torch.Tensor]):
    """va_tensor descriptor of a torch tensor (None -> NULL)."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("at most 4 dimensions")
    d = VaTensor()
    d.data = t.data_ptr() if t.numel() > 0 else 0
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _event_handle(ev) -> int:
    if ev is None:
        return 0
    if ev.cuda_event == 0:      # torch creates the CUDA event lazily
        ev.record()
    return int(ev.cuda_event)


def _args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, k_descale, v_descale, out):
    ds = [desc(x) for x in (q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                            k_descale, v_descale, out)]
    return ds, [_ref(d) for d in ds]


def verify_attn(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q: int,
                max_seqlen_k: int, softmax_scale: float, k_descale=None, v_descale=None,
                out=None, stream=None):
    """Target-verify attention (see include/verify_attn.h). Returns ``out``."""
    if out is None:
        out = torch.empty_like(q)
    ds, r = _args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, k_descale,
                  v_descale, out)
    with torch.cuda.device(q.device):
        s = _lib().verify_attn(r[0], r[1], r[2], r[3], r[4], r[5], int(max_seqlen_q),
                               int(max_seqlen_k), float(softmax_scale), r[6], r[7], r[8],
                               ctypes.c_void_p(_stream_handle(stream, q.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn")
    return out


def verify_attn_ex(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q: int,
                   max_seqlen_k: int, softmax_scale: float, k_descale=None, v_descale=None,
                   out=None, workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                   stream=None, event_after_main=None):
    """verify_attn with a caller workspace (a uint8 device tensor) and a forced
    split count (0 = heuristic). Allocates the workspace with torch if None.
    ``event_after_main`` (a torch.cuda.Event) is recorded between the two
    kernels when given."""
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = workspace_size(q, k_cache, seqused_k, max_seqlen_q, max_seqlen_k, num_splits)
        workspace = torch.zeros(n + 256, dtype=torch.uint8, device=q.device)
    addr = workspace.data_ptr()
    off = (-addr) % 256
    ds, r = _args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, k_descale,
                  v_descale, out)
    with torch.cuda.device(q.device):
        s = _lib().verify_attn_ex(r[0], r[1], r[2], r[3], r[4], r[5], int(max_seqlen_q),
                                  int(max_seqlen_k), float(softmax_scale), r[6], r[7], r[8],
                                  ctypes.c_void_p(addr + off), workspace.numel() - off,
                                  int(num_splits), ctypes.c_void_p(_event_handle(event_after_main)),
                                  ctypes.c_void_p(_stream_handle(stream, q.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_ex")
    return out


def verify_attn_noalloc(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                        max_seqlen_q: int, max_seqlen_k: int, softmax_scale: float,
                        k_descale=None, v_descale=None, out=None, stream=None):
    """verify_attn for callers that cannot allocate device memory: the
    split-KV partials live in an array built into the library
    (NOALLOC_SCRATCH_BYTES per GPU), so the call itself allocates nothing.
    ``out`` must be given by such callers (here it is created with torch only
    when omitted). Calls that overlap on the GPU share that array and race."""
    if out is None:
        out = torch.empty_like(q)
    ds, r = _args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, k_descale,
                  v_descale, out)
    with torch.cuda.device(q.device):
        s = _lib().verify_attn_noalloc(r[0], r[1], r[2], r[3], r[4], r[5], int(max_seqlen_q),
                                       int(max_seqlen_k), float(softmax_scale), r[6], r[7], r[8],
                                       ctypes.c_void_p(_stream_handle(stream, q.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_noalloc")
    return out


def _workspace_addr(workspace: Optional[torch.Tensor]) -> int:
    """The 256-byte-aligned address the wrappers pass for a workspace tensor."""
    if workspace is None:
        return 0
    a = workspace.data_ptr()
    return a + (-a) % 256


def last_device_error(workspace: Optional[torch.Tensor] = None, stream=None, device=None) -> int:
    """Reads and clears the status word of bounded waits that ran out (0 =
    none): of ``workspace`` as the wrappers passed it, or with None, of the
    library's own scratch on the device (its workspace and the no-alloc
    array). Synchronises ``stream`` (see include/verify_attn.h)."""
    if workspace is not None:
        dev = workspace.device
    else:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    bits = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        s = _lib().verify_attn_last_device_error(ctypes.c_void_p(_workspace_addr(workspace)),
                                                 ctypes.byref(bits),
                                                 ctypes.c_void_p(_stream_handle(stream, dev)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_last_device_error")
    return int(bits.value)


def set_wait_limit(limit_ns: int) -> None:
    """Time limit of the kernels' bounded waits for later launches (0 = the
    default 2 s). A test hook for the timeout path."""
    _lib().verify_attn_set_wait_limit(int(limit_ns))


def workspace_status(workspace: torch.Tensor) -> int:
    """Sticky error bits the kernels set in a caller workspace (0 = no bounded
    wait ever timed out). Reads device memory, so it synchronises."""
    off = (-workspace.data_ptr()) % 256
    return int(workspace[off:off + 4].view(torch.int32).item())


def check(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q: int,
          max_seqlen_k: int, k_descale=None, v_descale=None, out=None) -> int:
    """Host-only validation; returns the va_status code (no CUDA call)."""
    ds, r = _args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, k_descale,
                  v_descale, out)
    return int(_lib().verify_attn_check(r[0], r[1], r[2], r[3], r[4], r[5], int(max_seqlen_q),
                                        int(max_seqlen_k), r[6], r[7], r[8]))


def plan(num_seqs, num_kv_heads, num_q_heads, max_seqlen_q, max_seqlen_k, kv_dtype, num_sms,
         force_splits=0) -> dict:
    """The host launch heuristic (pure function). Raises on an error status."""
    p = VaPlan()
    code = VA_FP8_E4M3 if kv_dtype in ("fp8_e4m3", VA_FP8_E4M3, torch.float8_e4m3fn) else VA_BF16
    s = _lib().verify_attn_plan(int(num_seqs), int(num_kv_heads), int(num_q_heads),
                                int(max_seqlen_q), int(max_seqlen_k), code, int(num_sms),
                                int(force_splits), ctypes.byref(p))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_plan")
    return {f: getattr(p, f) for f, _ in VaPlan._fields_ if f != "reserved"}


def workspace_size(q, k_cache, seqused_k, max_seqlen_q, max_seqlen_k, num_splits=0) -> int:
    code = _DTYPES[k_cache.dtype]
    with torch.cuda.device(q.device):
        n = _lib().verify_attn_workspace_size(int(seqused_k.shape[0]), int(k_cache.shape[2]),
                                              int(q.shape[1]), int(max_seqlen_q),
                                              int(max_seqlen_k), code, int(num_splits))
    if n == 0:
        raise VerifyAttnError(4, "verify_attn_workspace_size")
    return int(n)


def run_workload(w, out=None, stream=None, **kw):
    """verify_attn on a ``workloads.Workload`` whose tensors are on the GPU."""
    return verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                       w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale,
                       w.v_descale, out=out, stream=stream, **kw)


def run_workload_ex(w, out=None, workspace=None, num_splits=0, stream=None,
                    event_after_main=None):
    return verify_attn_ex(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                          w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale,
                          w.v_descale, out=out, workspace=workspace, num_splits=num_splits,
                          stream=stream, event_after_main=event_after_main)


def block_table_from_indptr(kv_indptr, kv_indices, width: int, pad_page: int = 0,
                            block_table=None, seqused_k=None, status=None, stream=None):
    """Block table [B, width] and KV lengths [B] of a batch in flat token-slot
    form (see include/verify_attn.h). ``status``, if given, is a one-element
    int32 device tensor the kernel ORs BT_* bits into. Returns
    (block_table, seqused_k)."""
    B = kv_indptr.shape[0] - 1
    dev = kv_indptr.device
    if block_table is None:
        block_table = torch.empty((B, int(width)), dtype=torch.int32, device=dev)
    if seqused_k is None:
        seqused_k = torch.empty((B,), dtype=torch.int32, device=dev)
    st = 0 if status is None else status.data_ptr()
    di, dx, db, ds = desc(kv_indptr), desc(kv_indices), desc(block_table), desc(seqused_k)
    with torch.cuda.device(dev):
        s = _lib().verify_attn_block_table_from_indptr(
            _ref(di), _ref(dx), _ref(db), _ref(ds), int(pad_page), ctypes.c_void_p(st),
            ctypes.c_void_p(_stream_handle(stream, dev)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_block_table_from_indptr")
    return block_table, seqused_k


def verify_attn_opt(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                    max_seqlen_q: int, max_seqlen_k: int, softmax_scale: float, k_descale=None,
                    v_descale=None, out=None, window_left: int = -1, softcap: float = 0.0,
                    sinks=None, workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                    stream=None):
    """verify_attn with the generic attention's variants (see include/verify_attn.h):
    sliding window (keys [i - window_left, i]), logit soft cap, per-head sinks
    ([Hq] fp32). ``workspace`` None uses the library's own."""
    if out is None:
        out = torch.empty_like(q)
    ds, r = _args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, k_descale,
                  v_descale, out)
    dsk = desc(sinks)
    opts = VaOptions(int(window_left), float(softcap),
                     ctypes.pointer(dsk) if dsk is not None else None)
    if workspace is None:
        addr, nbytes = 0, 0
    else:
        a = workspace.data_ptr()
        off = (-a) % 256
        addr, nbytes = a + off, workspace.numel() - off
    with torch.cuda.device(q.device):
        s = _lib().verify_attn_opt(r[0], r[1], r[2], r[3], r[4], r[5], int(max_seqlen_q),
                                   int(max_seqlen_k), float(softmax_scale), r[6], r[7], r[8],
                                   ctypes.byref(opts), ctypes.c_void_p(addr), nbytes,
                                   int(num_splits), ctypes.c_void_p(_stream_handle(stream, q.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_opt")
    return out


def draft_extend_attn(q, k_cache, v_cache, kv_indptr, kv_indices, cu_seqlens_q,
                      max_seqlen_q: int, width: int, softmax_scale: float, k_descale=None,
                      v_descale=None, out=None, pad_page: int = 0, status=None, stream=None,
                      window_left: int = -1, softcap: float = 0.0, sinks=None):
    """The draft-extend pass: block table and lengths from the flat token-slot
    form, then the same attention as target verify with
    max_seqlen_k = width * 16 (and the pages' window / softcap / sinks
    pass-through). Two C-ABI calls on ``stream``."""
    bt, sk = block_table_from_indptr(kv_indptr, kv_indices, width, pad_page, status=status,
                                     stream=stream)
    if window_left < 0 and not softcap and sinks is None:
        return verify_attn(q, k_cache, v_cache, bt, cu_seqlens_q, sk, max_seqlen_q,
                           int(width) * 16, softmax_scale, k_descale, v_descale, out=out,
                           stream=stream)
    return verify_attn_opt(q, k_cache, v_cache, bt, cu_seqlens_q, sk, max_seqlen_q,
                           int(width) * 16, softmax_scale, k_descale, v_descale, out=out,
                           window_left=window_left, softcap=softcap, sinks=sinks, stream=stream)


def verify_attn_mla(q, kv_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q: int,
                    max_seqlen_k: int, softmax_scale: float, k_descale=None, v_descale=None,
                    out=None, workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                    stream=None, event_after_main=None):
    """Target-verify attention over an absorbed-MLA latent cache (see
    include/verify_attn.h): q [total_q, Hq, 576] bf16, kv_cache
    [num_blocks, 16, 1, 576] e4m3, out [total_q, Hq, 512] bf16. ``workspace``
    None uses the library's own; ``event_after_main`` (a torch.cuda.Event) is
    recorded between the two kernels when given."""
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], MLA_NOPE, dtype=torch.bfloat16, device=q.device)
    ds = [desc(x) for x in (q, kv_cache, block_table, cu_seqlens_q, seqused_k, k_descale,
                            v_descale, out)]
    r = [_ref(d) for d in ds]
    if workspace is None:
        addr, nbytes = 0, 0
    else:
        a = workspace.data_ptr()
        off = (-a) % 256
        addr, nbytes = a + off, workspace.numel() - off
    with torch.cuda.device(q.device):
        s = _lib().verify_attn_mla(r[0], r[1], r[2], r[3], r[4], int(max_seqlen_q),
                                   int(max_seqlen_k), float(softmax_scale), r[5], r[6], r[7],
                                   ctypes.c_void_p(addr), nbytes, int(num_splits),
                                   ctypes.c_void_p(_event_handle(event_after_main)),
                                   ctypes.c_void_p(_stream_handle(stream, q.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_mla")
    return out


def mla_workspace_size(q, seqused_k, max_seqlen_q, max_seqlen_k, num_splits=0) -> int:
    with torch.cuda.device(q.device):
        n = _lib().verify_attn_mla_workspace_size(int(seqused_k.shape[0]), int(q.shape[1]),
                                                  int(max_seqlen_q), int(max_seqlen_k),
                                                  int(num_splits))
    if n == 0:
        raise VerifyAttnError(4, "verify_attn_mla_workspace_size")
    return int(n)


def run_mla_workload(w, out=None, workspace=None, num_splits=0, stream=None,
                     event_after_main=None):
    """verify_attn_mla on a ``workloads.MlaWorkload`` whose tensors are on the GPU."""
    return verify_attn_mla(w.q, w.kv_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                           w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale,
                           w.v_descale, out=out, workspace=workspace, num_splits=num_splits,
                           stream=stream, event_after_main=event_after_main)


def verify_attn_partial(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q: int,
                        max_seqlen_k: int, softmax_scale: float, k_descale=None, v_descale=None,
                        kv_extent=None, o=None, lse=None, workspace: Optional[torch.Tensor] = None,
                        num_splits: int = 0, stream=None):
    """One shard of each sequence's keys (see include/verify_attn.h): returns
    (o [total_q, Hq, 256] fp32, lse [total_q, Hq] fp32). ``kv_extent`` [B]
    int32: the sequence's total keys minus the shard's first key position
    (None: the shard ends the sequence)."""
    if o is None:
        o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ds = [desc(x) for x in (q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, kv_extent,
                            k_descale, v_descale, o, lse)]
    r = [_ref(d) for d in ds]
    if workspace is None:
        addr, nbytes = 0, 0
    else:
        a = workspace.data_ptr()
        off = (-a) % 256
        addr, nbytes = a + off, workspace.numel() - off
    with torch.cuda.device(q.device):
        s = _lib().verify_attn_partial(r[0], r[1], r[2], r[3], r[4], r[5], r[6], int(max_seqlen_q),
                                       int(max_seqlen_k), float(softmax_scale), r[7], r[8], r[9],
                                       r[10], ctypes.c_void_p(addr), nbytes, int(num_splits),
                                       ctypes.c_void_p(_stream_handle(stream, q.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_partial")
    return o, lse


def merge_partials(parts, out=None, stream=None):
    """Log-sum-exp merge of shard results: ``parts`` is a list of (o, lse)
    pairs from verify_attn_partial; returns out [total_q, Hq, 256] bf16."""
    o0 = parts[0][0]
    if out is None:
        out = torch.empty(o0.shape, dtype=torch.bfloat16, device=o0.device)
    n = len(parts)
    oa = (VaTensor * n)(*[desc(o) for o, _ in parts])
    la = (VaTensor * n)(*[desc(l) for _, l in parts])
    d = desc(out)
    with torch.cuda.device(o0.device):
        s = _lib().verify_attn_merge_partials(n, oa, la, _ref(d),
                                              ctypes.c_void_p(_stream_handle(stream, o0.device)))
    if s != VA_OK:
        raise VerifyAttnError(s, "verify_attn_merge_partials")
    return out
