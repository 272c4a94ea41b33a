"""Pins of the shard (context-parallel) oracle, oracle/partial_fp64.py, to
facts outside it, and planted mistakes that each break a pin.

* Merging the results of a sequence's KV cut into shards (page-aligned, some
  empty) gives the full verify attention of the already-pinned oracle.
* One shard holding everything: o is the full oracle's output and lse is
  torch's logsumexp of the logits computed by torch on torch-gathered keys.
* A shard wholly before the draft tokens (kv_extent >= S + L - 1) is seen in
  full: o is torch SDPA without a mask.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.attention_fp64 as orc
import oracle.partial_fp64 as part
from speculative_decoding_verify_split_gb300.workloads import make_workload, split_kv_shards


def _raw(t):
    t = t.contiguous()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def shard_result(w, bt, su, ext):
    kv_dtype = "fp8_e4m3" if w.k_cache.dtype == torch.float8_e4m3fn else "bf16"
    kd = None if w.k_descale is None else float(w.k_descale[0])
    vd = None if w.v_descale is None else float(w.v_descale[0])
    return part.verify_attn_partial_oracle(_raw(w.q), _raw(w.k_cache), _raw(w.v_cache), kv_dtype,
                                           bt.numpy(), w.cu_seqlens_q.numpy(), su.numpy(),
                                           None if ext is None else ext.numpy(), w.softmax_scale, kd, vd)


def full_result(w):
    kv_dtype = "fp8_e4m3" if w.k_cache.dtype == torch.float8_e4m3fn else "bf16"
    kd = None if w.k_descale is None else float(w.k_descale[0])
    vd = None if w.v_descale is None else float(w.v_descale[0])
    return orc.verify_attn_oracle(_raw(w.q), _raw(w.k_cache), _raw(w.v_cache), kv_dtype,
                                  w.block_table.numpy(), w.cu_seqlens_q.numpy(), w.seqused_k.numpy(),
                                  w.softmax_scale, kd, vd)


CASES = [([4, 1, 3], [300, 17, 64], 16, 1, "fp8_e4m3"), ([2, 3], [129, 1000], 8, 2, "bf16"),
         ([1, 4, 2, 3], [16, 250, 33, 5], 4, 1, "fp8_e4m3")]


def pin_shards_merge_to_full(mod):
    for ci, (ql, kl, hq, hkv, dt) in enumerate(CASES):
        w = make_workload(ql, kl, hq, hkv, dt, seed=70 + ci, k_descale=1.2, v_descale=0.8)
        ref = full_result(w)
        for n in (1, 2, 3, 4):
            res = [shard_result(w, bt, su, ext) for bt, su, ext in split_kv_shards(w, n, seed=n + ci)]
            got = mod.merge_partials([r[0] for r in res], [r[1] for r in res])
            err = np.abs(got - ref).max()
            assert err <= 1e-12 * max(1.0, np.abs(ref).max()), (ci, n, err)


def pin_one_shard_lse(mod):
    w = make_workload([4, 2], [200, 40], 8, 1, "fp8_e4m3", seed=81, k_descale=1.3)
    o, lse = shard_result(w, w.block_table, w.seqused_k, None)
    ref = full_result(w)
    assert np.abs(o - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    for b, (L, S) in enumerate(zip([4, 2], [200, 40])):
        n = (S + 15) // 16
        k = w.k_cache[w.block_table[b, :n].long()].to(torch.float64).reshape(n * 16, 1, -1)[:S, 0] * float(w.k_descale[0])
        q0 = int(w.cu_seqlens_q[b])
        for t in range(L):
            for h in range(8):
                lg = w.softmax_scale * (w.q[q0 + t, h].to(torch.float64) @ k[:S - L + t + 1].T)
                assert abs(float(torch.logsumexp(lg, 0)) - lse[q0 + t, h]) < 1e-10


def pin_early_shard_unmasked(mod):
    w = make_workload([3, 2], [100, 64], 4, 1, "fp8_e4m3", seed=83)
    ext = w.seqused_k + 50                                  # the draft tokens are far past this shard
    o, _ = shard_result(w, w.block_table, w.seqused_k, ext)
    for b, (L, S) in enumerate(zip([3, 2], [100, 64])):
        n = (S + 15) // 16
        pages = w.block_table[b, :n].long()
        k = w.k_cache[pages].to(torch.float64).reshape(n * 16, 1, -1)[:S].permute(1, 0, 2)[None]
        v = w.v_cache[pages].to(torch.float64).reshape(n * 16, 1, -1)[:S].permute(1, 0, 2)[None]
        q0 = int(w.cu_seqlens_q[b])
        q = w.q[q0:q0 + L].to(torch.float64).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(q, k.expand(1, 4, S, 256), v.expand(1, 4, S, 256),
                                             scale=w.softmax_scale)[0].permute(1, 0, 2).numpy()
        assert np.abs(o[q0:q0 + L] - ref).max() < 1e-12


PINS = [pin_shards_merge_to_full, pin_one_shard_lse, pin_early_shard_unmasked]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(part)


_real_vis = part.visible_in_shard
_real_rows = part.partial_rows
_real_merge = part.merge_partials


def _vis_off_by_one(E, S, L, t):
    return _real_vis(E, S, L, t - 1)


def _lse_log2(q_rows, K, V, n_vis, scale):
    o, lse = _real_rows(q_rows, K, V, n_vis, scale)
    return o, lse / np.log(2.0)


def _merge_uniform(os_, lses):
    return _real_merge(os_, [np.where(np.isfinite(l), 0.0, -np.inf) for l in lses])


def _vis_ignores_extent(E, S, L, t):
    return _real_vis(S, S, L, t)


MUTATIONS = [("visible_in_shard", _vis_off_by_one), ("partial_rows", _lse_log2),
             ("merge_partials", _merge_uniform), ("visible_in_shard", _vis_ignores_extent)]


@pytest.mark.parametrize("name,fake", MUTATIONS, ids=["vis_off_by_one", "lse_log2", "merge_uniform", "extent_ignored"])
def test_planted_mistake_fails_a_pin(monkeypatch, name, fake):
    monkeypatch.setattr(part, name, fake)
    failures = 0
    for pin in PINS:
        try:
            pin(part)
        except AssertionError:
            failures += 1
    assert failures > 0, name
