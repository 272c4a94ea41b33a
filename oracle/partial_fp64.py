"""CPU oracle for verify attention over one shard of each sequence's keys, and
for the log-sum-exp merge of shard results.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.
It shares no code with the C-ABI library.

Source: the segment merge of sglang PR 36330 digest ("Implementation
breakdown" item 1: the main kernel's per-segment partials combined by a
"reduce segments" kernel), applied across shards of a sequence's KV as the
decode-context-parallel degree of sglang PR 34517 digest (``attn_dcp_size``)
implies. The pages show neither the shard layout nor the partials' format, so
these are readings:

* a shard holds the keys of global positions [o_b, o_b + S_b) of sequence b
  (S_b = the shard's ``seqused_k``), through its own block table;
* the shard's ``kv_extent`` E_b = (total keys of the sequence) - o_b: draft
  token t (of L) sits at global position o_b + E_b - L + t, so it sees the
  shard's local keys j <= E_b - L + t (E_b = S_b for the last shard);
* a shard result is o = softmax over the visible shard keys . V (times
  v_descale) and lse = ln(sum over those keys of exp(softmax_scale *
  k_descale * q . k)), natural log; a row with no visible key has o = 0 and
  lse = -inf;
* merging shards: out = sum_i exp(lse_i - LSE) o_i with LSE = ln sum_i
  exp(lse_i); rows whose lse are all -inf give 0.
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from oracle.attention_fp64 import DECODERS, decode_bf16, gather_kv, kv_head_of

PAGE_SIZE = 16


def visible_in_shard(E: int, S: int, L: int, t: int) -> int:
    """Local keys of the shard visible to draft token t: [0, E - L + t], clamped to [0, S]."""
    return max(0, min(S, E - L + t + 1))


def partial_rows(q_rows, K, V, n_vis, scale):
    """(o, lse) of rows attending to K[:n_vis[i]], V[:n_vis[i]] (fp64)."""
    R = q_rows.shape[0]
    o = np.zeros((R, V.shape[1]), dtype=np.float64)
    lse = np.full(R, -np.inf, dtype=np.float64)
    if K.shape[0] == 0:
        return o, lse
    logits = scale * (q_rows @ K.T)
    cols = np.arange(K.shape[0])[None, :]
    vis = cols < n_vis[:, None]
    for i in range(R):
        if not vis[i].any():
            continue
        lg = logits[i, vis[i]]
        m = lg.max()
        p = np.exp(lg - m)
        o[i] = (p @ V[:len(lg)]) / p.sum()
        lse[i] = m + np.log(p.sum())
    return o, lse


def verify_attn_partial_oracle(q_raw, k_raw, v_raw, kv_dtype, block_table, cu_seqlens_q, seqused_k,
                               kv_extent, softmax_scale, k_descale=None, v_descale=None,
                               seqs: Optional[Sequence[int]] = None):
    """Returns (o [total_q, Hq, D] float64, lse [total_q, Hq] float64) of one
    shard; rows of sequences outside ``seqs`` stay NaN."""
    decode = DECODERS[kv_dtype]
    q = decode_bf16(q_raw)
    total_q, Hq, D = q.shape
    Hkv = k_raw.shape[2]
    G = Hq // Hkv
    kd = 1.0 if k_descale is None else float(k_descale)
    vd = 1.0 if v_descale is None else float(v_descale)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    su = np.asarray(seqused_k, dtype=np.int64)
    ext = su if kv_extent is None else np.asarray(kv_extent, dtype=np.int64)
    o = np.full((total_q, Hq, D), np.nan)
    lse = np.full((total_q, Hq), np.nan)
    for b in (range(su.shape[0]) if seqs is None else seqs):
        L = int(cu[b + 1] - cu[b])
        S, E = int(su[b]), max(int(ext[b]), int(su[b]))
        if L <= 0:
            continue
        K = gather_kv(k_raw, decode, block_table[b], S, kd)
        V = gather_kv(v_raw, decode, block_table[b], S, vd)
        n_vis = np.array([visible_in_shard(E, S, L, t) for t in range(L)], dtype=np.int64)
        for h in range(Hq):
            kvh = kv_head_of(h, G, Hkv)
            ob, lb = partial_rows(q[cu[b]:cu[b] + L, h, :], K[:, kvh, :], V[:, kvh, :], n_vis,
                                  softmax_scale)
            o[cu[b]:cu[b] + L, h, :] = ob
            lse[cu[b]:cu[b] + L, h] = lb
    return o, lse


def merge_partials(os_, lses):
    """Log-sum-exp merge of shard results: lists of o [..., D] and lse [...]."""
    lse = np.stack(lses)                                     # [n, ...]
    big = np.max(lse, axis=0)
    safe = np.where(np.isfinite(big), big, 0.0)
    w = np.where(np.isfinite(lse), np.exp(lse - safe), 0.0)  # [n, ...]
    den = w.sum(axis=0)
    num = sum(wi[..., None] * oi for wi, oi in zip(w, os_))
    return np.where(den[..., None] > 0, num / np.where(den > 0, den, 1.0)[..., None], 0.0)


def partial_oracle_from_torch(w, kv_extent=None, seqs=None):
    """(o, lse) on a workload of CPU torch tensors (reads bytes only)."""
    import torch

    def raw(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.float8_e4m3fn:
            return t.view(torch.uint8).numpy()
        return t.view(torch.int16).numpy().view(np.uint16)
    kv_dtype = "fp8_e4m3" if w.k_cache.dtype == torch.float8_e4m3fn else "bf16"
    kd = None if w.k_descale is None else float(w.k_descale.cpu()[0])
    vd = None if w.v_descale is None else float(w.v_descale.cpu()[0])
    ext = None if kv_extent is None else np.asarray(kv_extent.cpu() if hasattr(kv_extent, "cpu") else kv_extent)
    return verify_attn_partial_oracle(raw(w.q), raw(w.k_cache), raw(w.v_cache), kv_dtype,
                                      w.block_table.cpu().numpy(), w.cu_seqlens_q.cpu().numpy(),
                                      w.seqused_k.cpu().numpy(), ext, w.softmax_scale, kd, vd, seqs)
