"""Pins of the latent-cache (absorbed-MLA) oracle, oracle/mla_fp64.py, to
facts outside it, and planted mistakes (on the CPU) that each break a pin.

* torch's float64 scaled_dot_product_attention on dense tensors gathered and
  converted by torch: K = whole cache rows (latent | rope) times k_descale,
  V = the latent columns times v_descale, explicit bottom-right causal mask.
* The already-pinned GQA oracle on an equivalent GQA problem: K = the whole
  rows, V = the latent padded with zero rope columns, so that the GQA
  result's first NOPE_DIM columns are the MLA result and the rest are 0.
* A closed form that needs no softmax: every visible row identical gives
  exactly that row's latent; a spike key that differs only in its rope part
  is invisible to the token before it and dominates the tokens after it.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.attention_fp64 as gqa
import oracle.mla_fp64 as mla
from speculative_decoding_verify_split_gb300.workloads import make_mla_workload

NOPE = 512


def _raw(t):
    t = t.contiguous()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def run(orc, w, seqs=None):
    kd = None if w.k_descale is None else float(w.k_descale[0])
    vd = None if w.v_descale is None else float(w.v_descale[0])
    kv_dtype = "fp8_e4m3" if w.kv_cache.dtype == torch.float8_e4m3fn else "bf16"
    return orc.verify_attn_mla_oracle(_raw(w.q), _raw(w.kv_cache), kv_dtype, w.block_table.numpy(),
                                      w.cu_seqlens_q.numpy(), w.seqused_k.numpy(), w.softmax_scale,
                                      kd, vd, NOPE, seqs)


def sdpa_mla(w, b):
    """[L, Hq, NOPE] from torch SDPA (float64) on torch-gathered rows."""
    L = int(w.cu_seqlens_q[b + 1] - w.cu_seqlens_q[b])
    S = int(w.seqused_k[b])
    q0 = int(w.cu_seqlens_q[b])
    n = (S + 15) // 16
    rows = w.kv_cache[w.block_table[b, :n].long()].to(torch.float64).reshape(n * 16, -1)[:S]
    kd = 1.0 if w.k_descale is None else float(w.k_descale[0])
    vd = 1.0 if w.v_descale is None else float(w.v_descale[0])
    Hq = w.q.shape[1]
    k = (rows * kd)[None, None].expand(1, Hq, S, rows.shape[1])
    v = (rows[:, :NOPE] * vd)[None, None].expand(1, Hq, S, NOPE)
    q = w.q[q0:q0 + L].to(torch.float64).permute(1, 0, 2)[None]
    t = torch.arange(L)[:, None]
    j = torch.arange(S)[None, :]
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=j <= (S - L + t), scale=w.softmax_scale)
    return o[0].permute(1, 0, 2).numpy()


def small(seed, hq=8, q_lens=(4, 1, 3), kv_lens=(300, 17, 64), descale=True):
    return make_mla_workload(list(q_lens), list(kv_lens), hq, seed=seed,
                             k_descale=1.3 if descale else None, v_descale=0.7 if descale else None)


# ---------------------------------------------------------------------------


def pin_sdpa(orc):
    for seed, hq, ql, kl in [(1, 8, (4, 1, 3), (300, 17, 64)), (2, 16, (2, 4), (129, 1000)),
                             (3, 4, (1, 2, 4, 3), (16, 15, 33, 250))]:
        w = small(seed, hq, ql, kl)
        got = run(orc, w)
        for b in range(len(ql)):
            q0, L = int(w.cu_seqlens_q[b]), ql[b]
            ref = sdpa_mla(w, b)
            err = np.abs(got[q0:q0 + L] - ref).max()
            assert err <= 1e-11 * max(1.0, np.abs(ref).max()), (seed, b, err)


def pin_gqa_oracle_on_padded_values(orc):
    w = small(4, 16, (4, 2), (200, 40))
    raw_kv = _raw(w.kv_cache)                                      # [nb, 16, 1, 576] uint8
    v_pad = raw_kv.copy()
    v_pad[..., NOPE:] = 0                                          # e4m3 0x00 is +0
    kd, vd = float(w.k_descale[0]), float(w.v_descale[0])
    ref = gqa.verify_attn_oracle(_raw(w.q), raw_kv, v_pad, "fp8_e4m3", w.block_table.numpy(),
                                 w.cu_seqlens_q.numpy(), w.seqused_k.numpy(), w.softmax_scale,
                                 kd, vd)
    got = run(orc, w)
    assert np.abs(ref[..., NOPE:]).max() == 0.0
    err = np.abs(got - ref[..., :NOPE]).max()
    assert err <= 1e-11 * max(1.0, np.abs(ref).max()), err


def pin_constant_rows_and_rope_spike(orc):
    """Every cache row = base, except row j* = S - L + 1 whose rope part is
    large and aligned with q_pe and whose latent differs. Token 0 sees keys
    [0, S - L], all equal to base: its output is base's latent (times
    v_descale) exactly. Tokens t >= 1 see the spike, whose logit exceeds the
    others by > 60: their output is the spike's latent to ~1e-26."""
    S, L, hq = 70, 3, 4
    w = make_mla_workload([L], [S], hq, seed=5, permute=True, k_descale=1.0, v_descale=0.5)
    g = torch.Generator().manual_seed(9)
    base = torch.randn(NOPE + 64, generator=g).to(torch.float8_e4m3fn)
    spike = base.clone()
    spike[:NOPE] = torch.randn(NOPE, generator=g).to(torch.float8_e4m3fn)
    spike[NOPE:] = torch.full((64,), 8.0).to(torch.float8_e4m3fn)
    n = (S + 15) // 16
    pages = w.block_table[0, :n].long()
    flat = w.kv_cache[pages].reshape(n * 16, -1)
    flat[:S] = base
    flat[S - L + 1] = spike
    w.kv_cache[pages] = flat.reshape(n, 16, 1, -1)
    qv = w.q.to(torch.float32)
    qv[:, :, NOPE:] = 4.0                                          # q_pe . r_spike = 64 * 4 * 8
    qv[:, :, :NOPE] = 0.0
    w.q = qv.to(torch.bfloat16)
    out = run(orc, w)
    b64 = base.to(torch.float64).numpy()[:NOPE] * 0.5
    s64 = spike.to(torch.float64).numpy()[:NOPE] * 0.5
    for h in range(hq):
        assert np.array_equal(out[0, h], b64), "token 0 must see only identical rows"
        for t in range(1, L):
            assert np.abs(out[t, h] - s64).max() < 1e-12, "the rope spike must dominate"


def pin_sdpa_bf16(orc):
    """The same SDPA pin on a BF16 latent cache (the oracle's bf16 decode of
    the cache rows; torch converts the rows for SDPA by itself)."""
    for seed, (q_lens, kv_lens, hq) in enumerate([((4, 2, 3), (40, 17, 1), 16), ((1, 4), (33, 64), 8)]):
        w = make_mla_workload(list(q_lens), list(kv_lens), hq, "bf16", seed=40 + seed, k_descale=1.3,
                              v_descale=0.6)
        out = run(orc, w)
        for b in range(len(q_lens)):
            q0 = int(w.cu_seqlens_q[b])
            ref = sdpa_mla(w, b)
            assert np.abs(out[q0:q0 + q_lens[b]] - ref).max() < 1e-10


def pin_scale_sign_and_zero(orc):
    """A negative softmax scale against torch's float64 SDPA with that scale,
    and a zero one against the mean of the visible latent rows times
    v_descale (every logit 0)."""
    w = make_mla_workload([4, 2], [70, 33], 8, seed=47, k_descale=1.2, v_descale=0.9, softmax_scale=-0.08)
    out = run(orc, w)
    for b, L in enumerate([4, 2]):
        q0 = int(w.cu_seqlens_q[b])
        ref = sdpa_mla(w, b)
        assert np.abs(out[q0:q0 + L] - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max())
    w = make_mla_workload([3, 1], [40, 18], 4, seed=48, v_descale=0.9, softmax_scale=0.0)
    out = run(orc, w)
    for b, (L, S) in enumerate([(3, 40), (1, 18)]):
        q0 = int(w.cu_seqlens_q[b])
        n = (S + 15) // 16
        pages = w.block_table[b, :n].long()
        lat = w.kv_cache[pages].to(torch.float64).reshape(n * 16, -1)[:S, :w.nope_dim] * float(w.v_descale[0])
        for t in range(L):
            ref = lat[:S - L + t + 1].mean(dim=0).numpy()
            assert np.abs(out[q0 + t] - ref[None, :]).max() <= 1e-11 * max(1.0, np.abs(ref).max())


PINS = [pin_sdpa, pin_gqa_oracle_on_padded_values, pin_constant_rows_and_rope_spike, pin_sdpa_bf16,
        pin_scale_sign_and_zero]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(mla)


def test_rows_without_visible_keys_are_zero():
    w = small(6, 4, (4, 2), (2, 0))
    out = run(mla, w)
    assert np.all(out[0:2] == 0.0) and np.all(np.isfinite(out))    # S - L + t < 0: no key
    assert np.all(out[4:6] == 0.0)                                 # an empty cache


# ---- planted mistakes ------------------------------------------------------

_real_split = mla.latent_and_rope
_real_logits = mla.mla_logit_rows


def _rope_dropped(q_rows, cache_rows, nope_dim):
    qn, _ = mla.query_parts(q_rows, nope_dim)
    c, _ = mla.latent_and_rope(cache_rows, nope_dim)
    return qn @ c.T


def _values_from_the_tail(rows, nope_dim):
    c, r = _real_split(rows, nope_dim)
    return rows[:, -nope_dim:], r


def _query_parts_swapped(q_rows, nope_dim):
    return q_rows[:, -nope_dim:], q_rows[:, :q_rows.shape[1] - nope_dim]


def _visible_minus_one(S, L, t):
    return max(0, min(S, S - L + t))


_real_attend = mla._attend


def _attend_abs_scale(q_rows, K, V, n_vis, scale, nope_dim):
    return _real_attend(q_rows, K, V, n_vis, abs(scale), nope_dim)


MUTATIONS = [("mla_logit_rows", _rope_dropped), ("latent_and_rope", _values_from_the_tail),
             ("query_parts", _query_parts_swapped), ("visible_keys", _visible_minus_one),
             ("_attend", _attend_abs_scale)]


@pytest.mark.parametrize("name,fake", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(monkeypatch, name, fake):
    monkeypatch.setattr(mla, name, fake)
    failures = 0
    for pin in PINS:
        try:
            pin(mla)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake in {name}"
