"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` takes the oracle module and raises AssertionError when the
oracle disagrees with:
* a library routine it does not call (torch's float8/bf16 conversions, torch's
  float64 ``scaled_dot_product_attention`` on dense, expanded K/V);
* a closed form (mean of V over the visible keys when every logit is equal;
  a single dominant key);
* an invariant of the definition (GQA equals MHA over repeated KV heads;
  relabelling physical pages; linearity in the V descale).

The same functions run in ``test_oracle_pins.py`` against the real oracle and
in ``test_oracle_mutations.py`` against copies with planted mistakes, which
shows that each plausible mistake fails at least one pin.
"""

from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from speculative_decoding_verify_split_gb300.workloads import make_workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _raw(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def run(orc, w, seqs=None, **variants):
    kv_dtype = "fp8_e4m3" if w.k_cache.dtype == torch.float8_e4m3fn else "bf16"
    kd = None if w.k_descale is None else float(w.k_descale[0])
    vd = None if w.v_descale is None else float(w.v_descale[0])
    return orc.verify_attn_oracle(_raw(w.q), _raw(w.k_cache), _raw(w.v_cache), kv_dtype,
                                  w.block_table.numpy(), w.cu_seqlens_q.numpy(),
                                  w.seqused_k.numpy(), w.softmax_scale, kd, vd, seqs, **variants)


def dense_kv(w, b):
    """[S, Hkv, D] float64 K and V of sequence b, gathered with torch indexing
    and converted with torch's own float conversion (not the oracle's)."""
    S = int(w.seqused_k[b])
    n = (S + 15) // 16
    pages = w.block_table[b, :n].long()
    k = w.k_cache[pages].to(torch.float64).reshape(n * 16, *w.k_cache.shape[2:])[:S]
    v = w.v_cache[pages].to(torch.float64).reshape(n * 16, *w.v_cache.shape[2:])[:S]
    kd = 1.0 if w.k_descale is None else float(w.k_descale[0])
    vd = 1.0 if w.v_descale is None else float(w.v_descale[0])
    return k * kd, v * vd


def sdpa_reference(w, b, causal=True, window_left=-1):
    """torch SDPA in float64 over the expanded (MHA) K/V of sequence b.
    Returns [L, Hq, D]; rows with no visible key are NaN from SDPA itself.
    With window_left >= 0 the mask also drops keys before i - window_left."""
    L = int(w.cu_seqlens_q[b + 1] - w.cu_seqlens_q[b])
    S = int(w.seqused_k[b])
    q0 = int(w.cu_seqlens_q[b])
    Hq, Hkv = w.q.shape[1], w.k_cache.shape[2]
    G = Hq // Hkv
    k, v = dense_kv(w, b)
    k = k.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]      # [1, Hq, S, D]
    v = v.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    q = w.q[q0:q0 + L].to(torch.float64).permute(1, 0, 2)[None]   # [1, Hq, L, D]
    if causal:
        t = torch.arange(L)[:, None]
        j = torch.arange(S)[None, :]
        mask = j <= (S - L + t)                                   # bottom-right causal
        if window_left >= 0:
            mask = mask & (j >= (S - L + t - window_left))
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=w.softmax_scale)
    else:
        o = F.scaled_dot_product_attention(q, k, v, scale=w.softmax_scale)
    return o[0].permute(1, 0, 2).numpy()                          # [L, Hq, D]


def _close(a, b, tol=1e-11):
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol * max(1.0, float(np.max(np.abs(b))) if b.size else 1.0), f"max err {err}"


# ---------------------------------------------------------------------------


def pin_e4m3_exhaustive(orc):
    bytes_ = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = bytes_.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.decode_e4m3fn(bytes_.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(got)), "NaN encodings differ"
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok]), "e4m3fn decode differs from torch"
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok])), "sign of zero differs"


def pin_e4m3_spec_points(orc):
    """Values printed in the OCP OFP8 specification's E4M3 table."""
    with open(os.path.join(GOLDEN, "e4m3fn_spec_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            byte_s, val_s = line.split()
            got = orc.decode_e4m3fn(np.array([int(byte_s, 16)], dtype=np.uint8))[0]
            if val_s == "nan":
                assert math.isnan(got), byte_s
            else:
                assert got == float(val_s) and math.copysign(1, got) == math.copysign(1, float(val_s)), (byte_s, got)


def pin_bf16_exhaustive(orc):
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = pats.view(torch.bfloat16).to(torch.float64).numpy()
    got = orc.decode_bf16(pats.numpy().view(np.uint16))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok]), "bf16 decode differs from torch"


_BRUTE_CASES = [
    # q_lens, kv_lens, Hq, Hkv, dtype, descales
    ([4, 2], [37, 19], 16, 1, "fp8_e4m3", (None, None)),
    ([3, 1, 4], [16, 33, 5], 8, 2, "fp8_e4m3", (0.75, 1.5)),
    ([2, 2], [48, 17], 4, 4, "bf16", (None, None)),
    ([1, 3], [64, 9], 8, 1, "bf16", (None, None)),
]


def pin_sdpa_bruteforce(orc):
    for i, (ql, kl, hq, hkv, dt, (kd, vd)) in enumerate(_BRUTE_CASES):
        w = make_workload(ql, kl, hq, hkv, dt, seed=100 + i, k_descale=kd, v_descale=vd)
        got = run(orc, w)
        for b in range(len(ql)):
            q0 = int(w.cu_seqlens_q[b])
            ref = sdpa_reference(w, b)
            _close(got[q0:q0 + ql[b]], ref)


def pin_gqa_equals_mha(orc):
    w = make_workload([3, 2], [40, 23], 8, 2, "fp8_e4m3", seed=7)
    G = 4
    m = make_workload([3, 2], [40, 23], 8, 2, "fp8_e4m3", seed=7)
    m.k_cache = w.k_cache.view(torch.uint8).repeat_interleave(G, dim=2).view(torch.float8_e4m3fn)
    m.v_cache = w.v_cache.view(torch.uint8).repeat_interleave(G, dim=2).view(torch.float8_e4m3fn)
    a = run(orc, w)
    b = run(orc, m)
    _close(a, b, 1e-13)


def pin_page_permutation(orc):
    w = make_workload([4, 3], [70, 45], 16, 1, "fp8_e4m3", seed=11)
    a = run(orc, w)
    nb = w.k_cache.shape[0]
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(nb, generator=g)             # old physical page p -> perm[p]
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    w.k_cache = w.k_cache.view(torch.uint8)[inv].view(torch.float8_e4m3fn)
    w.v_cache = w.v_cache.view(torch.uint8)[inv].view(torch.float8_e4m3fn)
    w.block_table = perm[w.block_table.long()].to(torch.int32)
    b = run(orc, w)
    assert np.array_equal(a, b), "page relabelling changed the oracle output"


def pin_qlen1_decode(orc):
    w = make_workload([1, 1, 1], [50, 16, 3], 8, 1, "bf16", seed=13)
    got = run(orc, w)
    for b in range(3):
        ref = sdpa_reference(w, b, causal=False)
        _close(got[b:b + 1], ref)


def pin_constant_keys(orc):
    """Every key equal => every visible logit equal => out = mean of visible V."""
    ql, kl = [4, 3], [29, 18]
    w = make_workload(ql, kl, 4, 1, "fp8_e4m3", seed=17)
    row = w.k_cache.view(torch.uint8)[0, 0, 0].clone()
    w.k_cache = w.k_cache.view(torch.uint8).clone()
    w.k_cache[:] = row
    w.k_cache = w.k_cache.view(torch.float8_e4m3fn)
    got = run(orc, w)
    for b in range(2):
        _, v = dense_kv(w, b)
        S, L, q0 = kl[b], ql[b], int(w.cu_seqlens_q[b])
        for t in range(L):
            n = S - L + t + 1
            ref = v[:n, 0, :].mean(dim=0).numpy()
            for h in range(4):
                _close(got[q0 + t, h], ref)


def pin_zero_scale(orc):
    """softmax_scale 0 => every visible logit 0 => out = mean of visible V,
    whatever Q and K hold (the kernels turn 0 into a tiny positive scale)."""
    ql, kl = [4, 2], [37, 20]
    w = make_workload(ql, kl, 8, 2, "fp8_e4m3", seed=27, softmax_scale=0.0, k_descale=1.7)
    got = run(orc, w)
    for b in range(2):
        _, v = dense_kv(w, b)
        S, L, q0 = kl[b], ql[b], int(w.cu_seqlens_q[b])
        for t in range(L):
            n = S - L + t + 1
            for h in range(8):
                _close(got[q0 + t, h], v[:n, h // 4, :].mean(dim=0).numpy())


def pin_negative_scale_sdpa(orc):
    """A negative softmax scale (the softmax of the negated logits) against
    torch's float64 SDPA with the same scale."""
    w = make_workload([4, 3], [90, 41], 16, 1, "bf16", seed=29, softmax_scale=-1 / 16)
    got = run(orc, w)
    for b in range(2):
        q0, L = int(w.cu_seqlens_q[b]), int(w.cu_seqlens_q[b + 1] - w.cu_seqlens_q[b])
        _close(got[q0:q0 + L], sdpa_reference(w, b), tol=1e-10)


def pin_spike_boundary(orc):
    """All-zero keys except one large key at position p = S - 2: with L = 4,
    tokens 0 and 1 do not see it (uniform mean over their keys), tokens 2 and 3
    see it and it dominates by e^128 (closed form: V[p])."""
    L, S = 4, 37
    w = make_workload([L], [S], 2, 1, "bf16", seed=19)
    w.q = torch.ones_like(w.q)
    k = torch.zeros_like(w.k_cache)
    p = S - 2
    page = int(w.block_table[0, p // 16])
    k[page, p % 16] = 8.0                                 # logit = 256 * 8 / 16 = 128
    w.k_cache = k
    got = run(orc, w)
    _, v = dense_kv(w, 0)
    for t in range(L):
        n = S - L + t + 1
        ref = v[p, 0].numpy() if n > p else v[:n, 0].mean(dim=0).numpy()
        for h in range(2):
            _close(got[t, h], ref, 1e-12)


def pin_descale(orc):
    w = make_workload([2, 3], [33, 20], 8, 2, "fp8_e4m3", seed=23)
    base = run(orc, w)
    w.v_descale = torch.tensor([1.75])
    _close(run(orc, w), 1.75 * base, 1e-13)
    w.v_descale = None
    w.k_descale = torch.tensor([0.5])
    a = run(orc, w)
    w.k_descale = None
    w.softmax_scale = w.softmax_scale * 0.5
    b = run(orc, w)
    _close(a, b, 1e-13)


def pin_empty_rows(orc):
    """S < L: tokens with no visible key give exactly 0; the rest match SDPA."""
    ql, kl = [4, 2], [2, 0]
    w = make_workload(ql, kl, 4, 1, "fp8_e4m3", seed=29)
    got = run(orc, w)
    ref = sdpa_reference(w, 0)                             # rows 0,1 NaN from SDPA
    assert np.all(got[0:2] == 0.0)
    _close(got[2:4], ref[2:4])
    assert np.all(got[4:6] == 0.0)


def pin_window_sdpa(orc):
    """Sliding window (window_size = (w, 0)): torch SDPA with the band mask, for
    windows from 0 (only the token's own key) to beyond the sequence."""
    ql, kl = [4, 2, 3], [70, 19, 5]
    w = make_workload(ql, kl, 8, 2, "bf16", seed=43)
    for win in (0, 1, 5, 16, 33, 200):
        got = run(orc, w, window_left=win)
        for b in range(3):
            q0, L = int(w.cu_seqlens_q[b]), ql[b]
            _close(got[q0:q0 + L], sdpa_reference(w, b, window_left=win))


def pin_window_never_reads_pages_before_it(orc):
    """Pages wholly before every row's window may be unmapped (a sliding-window
    page table): pointing them past the cache must not change the result."""
    ql, kl = [3, 2], [150, 90]
    w = make_workload(ql, kl, 4, 1, "fp8_e4m3", seed=47)
    win = 20
    ref = run(orc, w, window_left=win)
    bt = w.block_table.clone()
    for b in range(2):
        first = max(0, kl[b] - ql[b] - win)
        bt[b, :first // 16] = 10 ** 6                              # would raise if read
    w.block_table = bt
    try:
        got = run(orc, w, window_left=win)
    except IndexError as e:
        raise AssertionError(f"read a page before the window: {e}")
    _close(got, ref, 0.0)


def pin_softcap_closed_forms(orc):
    """A huge cap changes nothing; constant keys still give the mean of the
    visible V; a spike key of logit 128 among zero logits with cap c weighs
    e^(c tanh(128 / c)) against 1 for each other key."""
    w = make_workload([2, 3], [40, 25], 4, 1, "bf16", seed=53)
    _close(run(orc, w, softcap=1e9), run(orc, w), 1e-9)
    L, S = 4, 37
    w = make_workload([L], [S], 2, 1, "bf16", seed=19)
    w.q = torch.ones_like(w.q)
    k = torch.zeros_like(w.k_cache)
    p = S - 2
    k[int(w.block_table[0, p // 16]), p % 16] = 8.0                # logit 256 * 8 / 16 = 128
    w.k_cache = k
    cap = 2.0
    got = run(orc, w, softcap=cap)
    _, v = dense_kv(w, 0)
    e = math.exp(cap * math.tanh(128.0 / cap))
    for t in range(L):
        n = S - L + t + 1
        if n > p:
            ref = ((v[:n, 0].sum(dim=0) - v[p, 0]) + e * v[p, 0]) / (n - 1 + e)
        else:
            ref = v[:n, 0].mean(dim=0)
        for h in range(2):
            _close(got[t, h], ref.numpy(), 1e-12)


def pin_sink_closed_forms(orc):
    """A sink of -inf changes nothing; with constant keys every visible logit
    is c = scale q.k, so out = mean(V) n e^c / (n e^c + e^sink)."""
    w = make_workload([2, 3], [40, 25], 4, 1, "fp8_e4m3", seed=59)
    _close(run(orc, w, sinks=np.full(4, -np.inf)), run(orc, w), 0.0)
    ql, kl = [4, 3], [29, 18]
    w = make_workload(ql, kl, 4, 1, "bf16", seed=61)
    row = w.k_cache[0, 0, 0].clone()
    w.k_cache = w.k_cache.clone()
    w.k_cache[:] = row
    sinks = np.array([-1.0, 0.5, 2.0, 7.0])
    got = run(orc, w, sinks=sinks)
    kvec = row.to(torch.float64)
    for b in range(2):
        _, v = dense_kv(w, b)
        S, L, q0 = kl[b], ql[b], int(w.cu_seqlens_q[b])
        for t in range(L):
            n = S - L + t + 1
            for h in range(4):
                c = w.softmax_scale * float(w.q[q0 + t, h].to(torch.float64) @ kvec)
                scale = n * math.exp(c) / (n * math.exp(c) + math.exp(sinks[h]))
                _close(got[q0 + t, h], (v[:n, 0].mean(dim=0) * scale).numpy(), 1e-12)


ALL_PINS = [pin_e4m3_exhaustive, pin_e4m3_spec_points, pin_bf16_exhaustive, pin_sdpa_bruteforce,
            pin_gqa_equals_mha, pin_page_permutation, pin_qlen1_decode, pin_constant_keys,
            pin_spike_boundary, pin_descale, pin_empty_rows, pin_window_sdpa,
            pin_window_never_reads_pages_before_it, pin_softcap_closed_forms, pin_sink_closed_forms,
            pin_zero_scale, pin_negative_scale_sdpa]
