"""CPU oracle for target-verify attention over an absorbed-MLA latent cache.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.
It shares no code with the C-ABI library.

Source: sglang PR 34517 digest, "Implementation breakdown" item 1 and the
kernel excerpt of verify_mla.py. The grouped-head shared-KV verify kernel
serves two layouts through NOPE_DIM / PE_DIM:
* absorbed MLA (Kimi-K3): the single TP-local KV head is the MLA latent;
  NOPE_DIM is the latent width and PE_DIM = 64 is an extra RoPE part;
* plain GQA: PE_DIM = 0 and NOPE_DIM is the whole head (the path of
  ``attention_fp64``).
Its logits are ``(q_nope . k_nope + q_pe . k_pe) * sm_scale * k_scale``,
masked causally; a width check rejects ``q_head_dim < v_head_dim``.

What it computes (fp64), for every sequence b with L draft tokens and S
cached tokens, every query head h and every draft token t:

    row j of the cache (reached through block_table[b], page size 16),
        decoded, is [c_j (NOPE_DIM latent) | r_j (PE_DIM rope key)]
    logit_j = softmax_scale * k_descale * (q_nope[t, h] . c_j + q_pe[t, h] . r_j)
    out[t, h] = sum_j softmax(logit)_j * c_j * v_descale
    over the keys j in [0, S - L + t]

Readings where the pages are silent (each listed in the design notes):
* the values are the latent part of the same cache rows (absorbed MLA: V is
  the latent the keys' NOPE part is made of, and ``v_head_dim`` =
  NOPE_DIM <= ``q_head_dim``); V takes ``v_descale`` (callers with one cache
  scale pass it as both descales);
* NOPE_DIM = 512 in the tests and benchmarks (the latent width of the
  DeepSeek-V3 / Kimi-K2 MLA family; the pages give no width), PE_DIM = 64;
* the query's columns are [q_nope | q_pe], the cache row's [latent | rope];
* a row with no visible key gets output 0 (as in ``attention_fp64``).
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from oracle.attention_fp64 import DECODERS, decode_bf16, gather_kv, visible_keys

PE_DIM = 64


def latent_and_rope(rows: np.ndarray, nope_dim: int):
    """Split cache rows [S, NOPE_DIM + PE_DIM] into the latent c and the rope key r."""
    return rows[:, :nope_dim], rows[:, nope_dim:]


def query_parts(q_rows: np.ndarray, nope_dim: int):
    """Split query rows [R, NOPE_DIM + PE_DIM] into q_nope and q_pe."""
    return q_rows[:, :nope_dim], q_rows[:, nope_dim:]


def mla_logit_rows(q_rows: np.ndarray, cache_rows: np.ndarray, nope_dim: int) -> np.ndarray:
    """q_nope . c + q_pe . r for every (query row, key): [R, S], unscaled."""
    qn, qp = query_parts(q_rows, nope_dim)
    c, r = latent_and_rope(cache_rows, nope_dim)
    return qn @ c.T + qp @ r.T


def verify_attn_mla_oracle(
    q_raw: np.ndarray,            # [total_q, Hq, NOPE + PE] uint16 (bf16 bits)
    kv_raw: np.ndarray,           # [num_blocks, 16, 1, NOPE + PE] uint8 (e4m3fn) or uint16 (bf16)
    kv_dtype: str,                # "fp8_e4m3" or "bf16"
    block_table: np.ndarray,      # [B, W] int
    cu_seqlens_q: np.ndarray,     # [B + 1] int
    seqused_k: np.ndarray,        # [B] int
    softmax_scale: float,
    k_descale: Optional[float] = None,
    v_descale: Optional[float] = None,
    nope_dim: int = 512,
    seqs: Optional[Sequence[int]] = None,
) -> np.ndarray:
    """Exact (fp64) verify attention over a latent cache. Returns
    out [total_q, Hq, NOPE_DIM] float64; with ``seqs`` only those sequences'
    rows are filled (the rest stay NaN)."""
    decode = DECODERS[kv_dtype]
    q = decode_bf16(q_raw)
    total_q, Hq, Dq = q.shape
    if kv_raw.shape[2] != 1:
        raise ValueError("an MLA latent cache has one KV head")
    if kv_raw.shape[3] != Dq or Dq <= nope_dim:
        raise ValueError("query and cache rows must both be NOPE_DIM + PE_DIM wide")
    kd = 1.0 if k_descale is None else float(k_descale)
    vd = 1.0 if v_descale is None else float(v_descale)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    su = np.asarray(seqused_k, dtype=np.int64)
    out = np.full((total_q, Hq, nope_dim), np.nan, dtype=np.float64)
    for b in (range(su.shape[0]) if seqs is None else seqs):
        L = int(cu[b + 1] - cu[b])
        S = int(su[b])
        if L <= 0:
            continue
        rows = gather_kv(kv_raw, decode, block_table[b], S, 1.0)[:, 0, :]   # [S, NOPE + PE]
        K = rows * kd
        c, _ = latent_and_rope(rows, nope_dim)
        V = c * vd
        n_vis = np.array([visible_keys(S, L, t) for t in range(L)], dtype=np.int64)
        for h in range(Hq):
            qr = q[cu[b]:cu[b] + L, h, :]
            out[cu[b]:cu[b] + L, h, :] = _attend(qr, K, V, n_vis, softmax_scale, nope_dim)
    return out


def _attend(q_rows, K, V, n_vis, scale, nope_dim):
    """Softmax attention with the two-term MLA logit (rows with no visible
    key give 0)."""
    R = q_rows.shape[0]
    out = np.zeros((R, V.shape[1]), dtype=np.float64)
    if K.shape[0] == 0:
        return out
    logits = scale * mla_logit_rows(q_rows, K, nope_dim)
    cols = np.arange(K.shape[0])[None, :]
    vis = cols < n_vis[:, None]
    has = vis.any(axis=1)
    if not has.any():
        return out
    lg = np.where(vis, logits, -np.inf)[has]
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    out[has] = (p @ V) / p.sum(axis=1, keepdims=True)
    return out


def mla_oracle_from_torch(w, seqs=None) -> np.ndarray:
    """Runs the oracle on an MLA workload of CPU torch tensors (reads bytes only)."""
    import torch
    kv_dtype = "fp8_e4m3" if w.kv_cache.dtype == torch.float8_e4m3fn else "bf16"

    def raw(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.float8_e4m3fn:
            return t.view(torch.uint8).numpy()
        return t.view(torch.int16).numpy().view(np.uint16)
    kd = None if w.k_descale is None else float(w.k_descale.cpu()[0])
    vd = None if w.v_descale is None else float(w.v_descale.cpu()[0])
    return verify_attn_mla_oracle(raw(w.q), raw(w.kv_cache), kv_dtype, w.block_table.cpu().numpy(),
                                  w.cu_seqlens_q.cpu().numpy(), w.seqused_k.cpu().numpy(),
                                  w.softmax_scale, kd, vd, w.nope_dim, seqs)

