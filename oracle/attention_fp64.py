"""CPU oracle for target-verify attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module. The product
path (the C-ABI library and its Python binding) never calls it, and it shares
no code with that path: it has its own float decoders and its own gather.

What it computes (plain definition, fp64 throughout):

    for every sequence b with L = q_len, S = seqused_k[b]:
        K, V = dequantised keys/values of the first S token slots reached
               through block_table[b] (page size 16), times k/v descale
        for every query head h (KV head kvh = h // G, G = Hq / Hkv)
            for every draft token t in [0, L):
                keys visible to t: [0, S - L + t]              (causal, bottom-right)
                out[t, h] = softmax(softmax_scale * q[t, h] . K[vis, kvh]^T) @ V[vis, kvh]

Sources:
* sglang PR 36330 digest, "Motivation": the verify shape (max_seqlen_q <= 4,
  16 query heads per KV head, head size 256, page size 16, FP8 KV cache).
* sglang PR 36330 digest, "Key code excerpts" (aiter_backend.py): the call
  passes ``seqused_k = seq_lens + max_q_len``, so ``seqused_k`` counts the
  draft tokens too; the reference it is compared against (the generic
  unified attention, same excerpt, unit test) runs with ``causal=True``, so
  query token t of a sequence sees keys up to ``S - L + t``.
* sglang PR 30105 digest, "Implementation breakdown" item 2: dropping the KV
  head ``.expand()`` only changes tiling, not the math, i.e. grouped-query
  attention equals multi-head attention over the KV heads repeated G times.
* sglang PR 34517 digest, "Key code excerpts" (the shared-KV verify kernel):
  logits are multiplied by ``sm_scale * k_scale`` (per-tensor K descale); the
  same per-tensor rule is read for V.
* e4m3 decoding: OCP 8-bit floating point "E4M3" (the "FN" variant torch calls
  float8_e4m3fn): bias 7, no infinities, S.1111.111 is NaN, max 448.

Readings where the pages are silent: a row with no visible key (S < L) gets
output 0; token slots past S in the last page and block-table slots past the
last page are never read.
"""

from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

PAGE_SIZE = 16

# ---------------------------------------------------------------------------
# Decoders (own code, from the format definitions).
# ---------------------------------------------------------------------------


def _e4m3fn_value(byte: int) -> float:
    """Value of one OCP E4M3 ("FN") byte: 1 sign, 4 exponent (bias 7), 3 mantissa."""
    s = -1.0 if (byte >> 7) & 1 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)          # subnormal: 2^(1-7) * m/8
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


_E4M3_TABLE = np.array([_e4m3fn_value(b) for b in range(256)], dtype=np.float64)


def decode_e4m3fn(raw: np.ndarray) -> np.ndarray:
    """uint8 e4m3fn bytes -> float64 (exact)."""
    return _E4M3_TABLE[np.asarray(raw, dtype=np.uint8)]


def decode_bf16(raw: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact): bf16 is the top half of fp32."""
    u32 = np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even), returned as float64.

    Goes through fp32 first (round to nearest even), then rounds the fp32 bit
    pattern to its top 16 bits with ties to even. Used only to state what a
    bf16 output can represent."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    nan = np.isnan(f)
    out = decode_bf16(r.astype(np.uint16))
    out[nan] = np.nan
    return out


DECODERS = {"fp8_e4m3": decode_e4m3fn, "bf16": decode_bf16}

# ---------------------------------------------------------------------------
# Steps of the definition. Kept as small functions so the tests can check each
# one against the pages and plant mistakes in them.
# ---------------------------------------------------------------------------


def kv_head_of(h: int, group: int, num_kv_heads: int) -> int:
    """Query head h reads KV head h // G (contiguous groups of G query heads)."""
    return h // group


def visible_keys(S: int, L: int, t: int) -> int:
    """Number of keys draft token t sees: keys [0, S - L + t], clamped to [0, S]."""
    return max(0, min(S, S - L + t + 1))


def first_visible_key(S: int, L: int, t: int, window_left: int) -> int:
    """First key draft token t sees. Without a window (window_left < 0) that
    is key 0. With window_size = (window_left, 0) the token at position
    i = S - L + t sees keys [i - window_left, i] (sglang PR 30105 digest,
    "Key code excerpts": window_size = (sliding_window_size - 1, 0))."""
    if window_left < 0:
        return 0
    return max(0, S - L + t - window_left)


def gather_kv(cache_raw: np.ndarray, decode, block_table_row: np.ndarray, S: int,
              descale: float, start: int = 0) -> np.ndarray:
    """[S - start, Hkv, D] float64: token slots [start, S) reached through the
    block table. Pages holding only keys before ``start`` are never read (a
    sliding-window page table need not map them)."""
    if S <= start:
        return np.zeros((0,) + cache_raw.shape[2:], dtype=np.float64)
    p0 = start // PAGE_SIZE
    n_pages = (S + PAGE_SIZE - 1) // PAGE_SIZE
    pages = np.asarray(block_table_row[p0:n_pages], dtype=np.int64)
    raw = cache_raw[pages]                                  # [pages, 16, Hkv, D]
    raw = raw.reshape((len(pages) * PAGE_SIZE,) + cache_raw.shape[2:])
    raw = raw[start - p0 * PAGE_SIZE:S - p0 * PAGE_SIZE]
    return decode(raw) * float(descale)


def softcapped(logits: np.ndarray, softcap: float) -> np.ndarray:
    """Logit soft-capping, softcap * tanh(s / softcap); 0 means off (sglang PR
    30105 digest, "Key code excerpts": softcap=layer.logit_cap)."""
    if not softcap:
        return logits
    return softcap * np.tanh(logits / softcap)


def sink_weight(sink: float, m: np.ndarray) -> np.ndarray:
    """Weight of a sink logit in the normaliser, relative to the row max m."""
    return np.exp(sink - m)


def softmax_attend(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray,
                   n_visible: np.ndarray, scale: float, first=None, softcap: float = 0.0,
                   sink: Optional[float] = None) -> np.ndarray:
    """Row i attends to K[first[i]:n_visible[i]] (first defaults to 0); rows
    with no visible key give 0.

    q_rows [R, D], K [S, D], V [S, D] -> [R, D]; softmax in the usual
    max-subtracted form (exact up to fp64 rounding). ``sink`` is an extra
    logit with a zero value vector: it joins the normaliser only."""
    R = q_rows.shape[0]
    out = np.zeros((R, V.shape[1]), dtype=np.float64)
    if K.shape[0] == 0:
        return out
    lo = np.zeros(R, dtype=np.int64) if first is None else np.asarray(first, dtype=np.int64)
    logits = softcapped(scale * (q_rows @ K.T), softcap)     # [R, S]
    cols = np.arange(K.shape[0])[None, :]
    vis = (cols < n_visible[:, None]) & (cols >= lo[:, None])
    logits = np.where(vis, logits, -np.inf)
    has = vis.any(axis=1)
    if not np.any(has):
        return out
    lg = logits[has]
    m = lg.max(axis=1, keepdims=True)
    if sink is not None:
        m = np.maximum(m, sink)
    p = np.exp(lg - m)
    p = np.where(vis[has], p, 0.0)
    den = p.sum(axis=1, keepdims=True)
    if sink is not None:
        den = den + sink_weight(sink, m)
    out[has] = (p @ V) / den
    return out


# ---------------------------------------------------------------------------
# The oracle.
# ---------------------------------------------------------------------------


def verify_attn_oracle(
    q_raw: np.ndarray,            # [total_q, Hq, D] uint16 (bf16 bits)
    k_raw: np.ndarray,            # [num_blocks, 16, Hkv, D] uint8 (e4m3fn) or uint16 (bf16)
    v_raw: np.ndarray,
    kv_dtype: str,                # "fp8_e4m3" or "bf16"
    block_table: np.ndarray,      # [B, W] int
    cu_seqlens_q: np.ndarray,     # [B + 1] int
    seqused_k: np.ndarray,        # [B] int
    softmax_scale: float,
    k_descale: Optional[float] = None,
    v_descale: Optional[float] = None,
    seqs: Optional[Sequence[int]] = None,
    window_left: int = -1,        # sliding window: keys [i - window_left, i]; -1 = none
    softcap: float = 0.0,         # logit soft cap; 0 = none
    sinks: Optional[np.ndarray] = None,  # [Hq] per-head sink logits (natural log); None = none
) -> np.ndarray:
    """Exact (fp64) verify attention. Returns out [total_q, Hq, D] float64.

    ``seqs`` restricts the work to a subset of sequences (the other rows of the
    result stay NaN), so full-size workloads can be checked on a sample.
    ``window_left``, ``softcap`` and ``sinks`` are the generic attention's
    variants the pages pass through (sglang PR 30105 digest, "Key code
    excerpts": window_size, softcap, sinks): the logits are
    softcap * tanh(scale * q.k / softcap), a row sees the keys of its window
    only, and a sink logit joins each head's softmax normaliser."""
    decode = DECODERS[kv_dtype]
    q = decode_bf16(q_raw)
    total_q, Hq, D = q.shape
    Hkv = k_raw.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    kd = 1.0 if k_descale is None else float(k_descale)
    vd = 1.0 if v_descale is None else float(v_descale)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    su = np.asarray(seqused_k, dtype=np.int64)
    B = su.shape[0]
    out = np.full((total_q, Hq, D), np.nan, dtype=np.float64)
    for b in (range(B) if seqs is None else seqs):
        L = int(cu[b + 1] - cu[b])
        S = int(su[b])
        if L <= 0:
            continue
        first = np.array([first_visible_key(S, L, t, window_left) for t in range(L)],
                         dtype=np.int64)
        k0 = int(first.min()) if L else 0                         # keys before k0: never read
        K = gather_kv(k_raw, decode, block_table[b], S, kd, k0)  # [S - k0, Hkv, D]
        V = gather_kv(v_raw, decode, block_table[b], S, vd, k0)
        n_vis = np.array([visible_keys(S, L, t) for t in range(L)], dtype=np.int64) - k0
        for h in range(Hq):
            kvh = kv_head_of(h, G, Hkv)
            rows = q[cu[b]:cu[b] + L, h, :]                       # [L, D]
            sink = None if sinks is None else float(sinks[h])
            out[cu[b]:cu[b] + L, h, :] = softmax_attend(rows, K[:, kvh, :], V[:, kvh, :],
                                                        n_vis, softmax_scale, first - k0,
                                                        softcap, sink)
    return out


def oracle_from_torch(w, seqs=None, window_left=None, softcap=None, sinks=None) -> np.ndarray:
    """Convenience: run the oracle on a workload of CPU torch tensors.

    Only reads the tensors' bytes (``.view`` to integer types, ``.numpy()``).
    The variants default to the workload's own (attributes window_left,
    softcap, sinks when it has them)."""
    import torch
    kv_dtype = "fp8_e4m3" if w.k_cache.dtype == torch.float8_e4m3fn else "bf16"
    def raw(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.float8_e4m3fn:
            return t.view(torch.uint8).numpy()
        return t.view(torch.int16).numpy().view(np.uint16)
    kd = None if w.k_descale is None else float(w.k_descale.cpu()[0])
    vd = None if w.v_descale is None else float(w.v_descale.cpu()[0])
    if window_left is None:
        window_left = int(getattr(w, "window_left", -1))
    if softcap is None:
        softcap = float(getattr(w, "softcap", 0.0))
    if sinks is None and getattr(w, "sinks", None) is not None:
        sinks = w.sinks.detach().cpu().numpy().astype(np.float64)
    return verify_attn_oracle(raw(w.q), raw(w.k_cache), raw(w.v_cache), kv_dtype,
                              w.block_table.cpu().numpy(), w.cu_seqlens_q.cpu().numpy(),
                              w.seqused_k.cpu().numpy(), w.softmax_scale, kd, vd, seqs,
                              window_left, softcap, sinks)
