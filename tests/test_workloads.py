"""The seeded input recipes (speculative_decoding_verify_split_gb300/workloads.py)
against the five verify configurations they stand for, and the invariants of
the inputs the tests and the bench build from them: the paged layout and its
poison page, the flat token-slot form of the draft-extend pass, and the
page-aligned shards of the context-parallel path. Structure only, on the CPU;
the attention arithmetic lives in oracle/ and the kernels."""
import math

import pytest
import torch

from speculative_decoding_verify_split_gb300.workloads import (
    BF16, FP8, MLA_WORKLOADS, WORKLOADS, flat_kv_slots, make_workload, mla_workload_structure,
    named_workload, split_kv_shards, workload_sizes, workload_structure)

# name -> (batch, q_len values allowed, kv range inclusive, Hq, Hkv, kv dtype)
CONFIGS = {
    "tiny_verify": (2, None, None, 16, 1, FP8),
    "gqa_32q2kv": (8, {2, 3, 4}, (513, 4096), 32, 2, FP8),
    "mid_context_fp8": (64, {3}, (8192, 32768), 16, 1, FP8),
    "long_context_fp8": (16, {4}, (65536, 131072), 16, 1, FP8),
    "high_concurrency_bf16": (256, {2}, (2048, 16384), 8, 1, BF16),
}


def test_every_config_has_a_recipe():
    assert set(WORKLOADS) == set(CONFIGS)


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_structure_matches_config(name):
    B, qs, kv, hq, hkv, dt = CONFIGS[name]
    st = workload_structure(name)
    assert len(st["q_lens"]) == len(st["kv_lens"]) == B
    assert (st["Hq"], st["Hkv"], st["kv_dtype"]) == (hq, hkv, dt)
    if qs is not None:
        assert set(st["q_lens"]) <= qs
        assert all(kv[0] <= s <= kv[1] for s in st["kv_lens"])
    # reproducible from the seed, and the seed matters
    assert workload_structure(name)["kv_lens"] == st["kv_lens"]
    if kv is not None:
        assert workload_structure(name, seed=1)["kv_lens"] != st["kv_lens"]


def test_tiny_verify_is_the_stated_case():
    w = named_workload("tiny_verify")
    assert w.q_lens == [4, 2] and w.kv_lens == [1024, 769]
    assert torch.equal(w.block_table, torch.arange(2 * 65, dtype=torch.int32).view(2, 65))
    assert float(w.k_descale[0]) == 1.0 and float(w.v_descale[0]) == 1.0
    assert w.softmax_scale == 1 / 16
    assert w.q.dtype == torch.bfloat16 and w.k_cache.dtype == torch.float8_e4m3fn


def test_sizes_count_kv_once_per_kv_head():
    s = workload_sizes("long_context_fp8")
    kv = sum(s["kv_lens"]) * 1 * 256 * 2 * 1
    assert s["kv_bytes"] == kv
    assert s["algorithmic_bytes"] == kv + 2 * sum(s["q_lens"]) * 16 * 256 * 2
    b = workload_sizes("high_concurrency_bf16")
    assert b["kv_bytes"] == sum(b["kv_lens"]) * 256 * 2 * 2


@pytest.mark.parametrize("name", MLA_WORKLOADS)
def test_latent_structures_mirror_the_gqa_shapes(name):
    st = mla_workload_structure(name)
    base = {"mla_tiny": "tiny_verify", "mla_mid_context_fp8": "mid_context_fp8",
            "mla_long_context_fp8": "long_context_fp8", "mla_tiny_bf16": "tiny_verify",
            "mla_mid_context_bf16": "mid_context_fp8", "mla_long_context_bf16": "long_context_fp8"}[name]
    assert st.get("kv_dtype", FP8) == (BF16 if name.endswith("_bf16") else FP8)
    B, qs, kv, hq, _, _ = CONFIGS[base]
    assert len(st["q_lens"]) == B and st["Hq"] == hq
    if qs is not None:
        assert set(st["q_lens"]) <= qs and all(kv[0] <= s <= kv[1] for s in st["kv_lens"])


def small(seed=3, dt=FP8):
    return make_workload([4, 1, 3, 2], [700, 16, 33, 1], 8, 2, dt, seed=seed)


@pytest.mark.parametrize("dt", [FP8, BF16])
def test_paged_layout_and_poison(dt):
    w = small(dt=dt)
    pages = [math.ceil(s / 16) for s in w.kv_lens]
    used = torch.cat([w.block_table[b, :n] for b, n in enumerate(pages)])
    # every data page used exactly once; the poison page is the extra last one
    assert sorted(used.tolist()) == list(range(sum(pages)))
    assert w.poison_page == sum(pages) == w.k_cache.shape[0] - 1
    for b, n in enumerate(pages):
        assert (w.block_table[b, n:] == w.poison_page).all()
    bits = torch.uint8 if dt == FP8 else torch.int16
    k = w.k_cache.view(bits)
    poison = (k[w.poison_page].flatten().to(torch.int32) & 0x7F) == 0x7F if dt == FP8 else \
        (k[w.poison_page].flatten().to(torch.int32) & 0x7FFF) == 0x7FC0
    assert poison.all()
    # the slots past seqused_k in a sequence's last page are poisoned too
    b = 0
    last = int(w.block_table[b, pages[b] - 1])
    tail = w.kv_lens[b] - (pages[b] - 1) * 16
    vals = w.v_cache[last, tail:].float()
    assert torch.isnan(vals).all()
    assert not torch.isnan(w.v_cache[last, :tail].float()).any()


def test_flat_slots_match_the_block_table():
    w = small()
    indptr, slots = flat_kv_slots(w)
    assert indptr.tolist() == [0] + list(torch.tensor(w.kv_lens).cumsum(0).tolist())
    for b, S in enumerate(w.kv_lens):
        s = slots[indptr[b]:indptr[b + 1]].to(torch.int64)
        t = torch.arange(S)
        assert torch.equal(s // 16, w.block_table[b, t // 16].to(torch.int64))
        assert torch.equal(s % 16, t % 16)


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_shards_partition_each_sequence(n):
    w = small(seed=7)
    shards = split_kv_shards(w, n, seed=n)
    assert len(shards) == n
    for b, S in enumerate(w.kv_lens):
        pages = math.ceil(S / 16)
        offset, got = 0, []
        for bt, su, ext in shards:
            s, e = int(su[b]), int(ext[b])
            assert e == S - offset          # token t of the shard sits at offset + e - L + t
            assert offset % 16 == 0 or s == 0  # cuts fall on page boundaries
            got += bt[b, :math.ceil(s / 16)].tolist()
            offset += s
        assert offset == S
        assert got == w.block_table[b, :pages].tolist()
