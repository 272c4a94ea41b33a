"""The draft-extend path on the GPU, through the C-ABI: block table and KV
lengths built from the flat token-slot form (kv_indptr / kv_indices), then
the verify attention on them.

* The builder against the oracle (oracle/block_table.py): table, lengths and
  status bits bit for bit, on random ragged layouts, on cases built to set
  each status bit, on a strided output table, and on the full long-context
  layout (1.6 M tokens).
* The whole pass (draft_extend_attn) against verify_attn on the workload's
  own table: bit-identical outputs, and within the parity tolerance of the
  attention oracle."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import (flat_kv_slots, make_workload,
                                                               named_workload)
from oracle.block_table import block_table_from_indptr
from gpu_util import compare
from oracle.attention_fp64 import oracle_from_torch
from test_oracle_block_table import expand, random_layout

pytestmark = pytest.mark.gpu

PAD = -7


def gpu_build(indptr, slots, width, table=None):
    ip = torch.as_tensor(np.asarray(indptr), dtype=torch.int32, device="cuda")
    ix = torch.as_tensor(np.asarray(slots), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt, sk = va.block_table_from_indptr(ip, ix, width, PAD, block_table=table, status=status)
    torch.cuda.synchronize()
    return bt.cpu().numpy(), sk.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("seed", range(12))
def test_builder_matches_oracle_random(seed):
    rows, lengths, width = random_layout(np.random.default_rng(1000 + seed))
    indptr, slots = expand(rows, lengths)
    got = gpu_build(indptr, slots, width)
    ref = block_table_from_indptr(indptr, slots, width, PAD)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]) and got[2] == ref[2]


def test_builder_status_bits_match_oracle():
    good = list(range(112, 128)) + list(range(48, 52))
    swapped = list(good)
    swapped[4], swapped[5] = swapped[5], swapped[4]
    cases = [([0, 20], [113] + good[1:], 2), ([0, 20], swapped, 2), ([0, 20], good, 1),
             ([0, 20, 10], good, 2), ([0, 20, 25], good, 2), ([0, 20, 20], good, 0)]
    for indptr, slots, width in cases:
        got = gpu_build(indptr, slots, width)
        ref = block_table_from_indptr(indptr, slots, width, PAD)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
        assert got[2] == ref[2], (indptr, width, got[2], ref[2])


def test_builder_strided_table_and_empty_batch():
    rows, lengths, width = random_layout(np.random.default_rng(7))
    indptr, slots = expand(rows, lengths)
    big = torch.full((len(lengths), 2 * width + 3), 99, dtype=torch.int32, device="cuda")
    view = big[:, 1:2 * width + 1:2]                      # row stride 2w+3, column stride 2
    got = gpu_build(indptr, slots, width, table=view)
    ref = block_table_from_indptr(indptr, slots, width, PAD)
    assert np.array_equal(got[0], ref[0])
    rest = big.cpu().numpy().copy()
    rest[:, 1:2 * width + 1:2] = 99
    assert (rest == 99).all()                              # nothing else written
    got = gpu_build([0], [], 4)
    assert got[0].shape == (0, 4) and got[2] == 0


def test_builder_full_long_context_layout():
    w = named_workload("long_context_fp8", value_device="cuda").to("cuda")
    ip, ix = flat_kv_slots(w)
    width = w.block_table.shape[1]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt, sk = va.block_table_from_indptr(ip, ix, width, PAD, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert sk.cpu().tolist() == list(w.kv_lens)
    own = w.block_table.cpu().numpy()
    got = bt.cpu().numpy()
    for b, S in enumerate(w.kv_lens):
        n = (S + 15) // 16
        assert np.array_equal(got[b, :n], own[b, :n]) and (got[b, n:] == PAD).all()
    ref = block_table_from_indptr(ip.cpu().numpy(), ix.cpu().numpy(), width, PAD)
    assert np.array_equal(got, ref[0]) and ref[2] == 0


@pytest.mark.parametrize("case", [
    dict(q=[4, 2, 3, 1], kv=[3000, 769, 1500, 40], hq=16, hkv=1, dt="fp8_e4m3", kd=0.9, vd=1.3),
    dict(q=[2, 3, 2], kv=[2100, 513, 4000], hq=32, hkv=2, dt="fp8_e4m3", kd=None, vd=None),
    dict(q=[2] * 5, kv=[2048, 9000, 300, 17, 5000], hq=8, hkv=1, dt="bf16", kd=None, vd=None),
])
def test_draft_extend_equals_verify_on_own_table(case):
    w = make_workload(case["q"], case["kv"], case["hq"], case["hkv"], case["dt"], seed=41,
                      k_descale=case["kd"], v_descale=case["vd"]).to("cuda")
    ip, ix = flat_kv_slots(w)
    width = w.block_table.shape[1]
    ref = torch.full_like(w.q, float("nan"))           # same upper bound, so the same split
    va.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                   w.max_seqlen_q, width * 16, w.softmax_scale, w.k_descale, w.v_descale, out=ref)
    got = torch.full_like(w.q, float("nan"))
    va.draft_extend_attn(w.q, w.k_cache, w.v_cache, ip, ix, w.cu_seqlens_q, w.max_seqlen_q,
                         width, w.softmax_scale, w.k_descale, w.v_descale, out=got, pad_page=0)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    compare(got, oracle_from_torch(w.to("cpu")))
