"""Shards of each sequence's keys on the GPU (verify_attn_partial) and their
log-sum-exp merge (verify_attn_merge_partials), through the C-ABI:

* each shard's (o, lse) against the shard oracle (oracle/partial_fp64.py):
  o within the parity tolerance, lse within 2e-2 (and -inf exactly where a
  row sees no key of the shard);
* the merged output of 1-4 shards (page-aligned cuts, some empty) against
  the full verify-attention oracle, on both KV types and at forced splits;
* the long-context workload cut in two, merged, every sequence;
* argument errors."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import (make_workload, named_workload,
                                                               split_kv_shards)
from oracle.attention_fp64 import oracle_from_torch
from oracle.partial_fp64 import partial_oracle_from_torch
from gpu_util import compare

pytestmark = pytest.mark.gpu

CASES = [
    dict(q=[4, 2, 3, 1], kv=[3000, 769, 300, 5], hq=16, hkv=1, dt="fp8_e4m3", kd=1.1, vd=0.8),
    dict(q=[2, 3], kv=[2100, 513], hq=32, hkv=2, dt="fp8_e4m3", kd=None, vd=None),
    dict(q=[2, 2, 1], kv=[1500, 64, 700], hq=8, hkv=1, dt="bf16", kd=None, vd=None),
]


def workload(case, seed):
    return make_workload(case["q"], case["kv"], case["hq"], case["hkv"], case["dt"], seed=seed,
                         k_descale=case["kd"], v_descale=case["vd"])


def run_shard(wg, bt, su, ext, splits=0):
    width = bt.shape[1]
    n = va.workspace_size(wg.q, wg.k_cache, su, wg.max_seqlen_q, width * 16, splits)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    o, lse = va.verify_attn_partial(wg.q, wg.k_cache, wg.v_cache, bt, wg.cu_seqlens_q, su,
                                    wg.max_seqlen_q, width * 16, wg.softmax_scale, wg.k_descale,
                                    wg.v_descale, kv_extent=ext, workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    assert va.workspace_status(ws) == 0
    return o, lse


def shard_view(w, bt, su):
    """The workload as the shard sees it (CPU), for the shard oracle."""
    s = w.to("cpu")
    s.block_table, s.seqused_k = bt.cpu(), su.cpu()
    return s


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_each_shard_against_its_oracle(ci):
    w = workload(CASES[ci], 200 + ci)
    wg = w.to("cuda")
    for bt, su, ext in split_kv_shards(wg, 3, seed=ci):
        o, lse = run_shard(wg, bt, su, ext)
        ro, rl = partial_oracle_from_torch(shard_view(w, bt, su), ext.cpu())
        got_l = lse.cpu().numpy().astype(np.float64)
        assert np.array_equal(np.isinf(got_l), np.isinf(rl)), "rows without visible keys differ"
        fin = np.isfinite(rl)
        assert np.abs(got_l[fin] - rl[fin]).max(initial=0.0) < 2e-2
        compare(o, ro)


@pytest.mark.parametrize("ci", range(len(CASES)))
@pytest.mark.parametrize("n", [1, 2, 4])
def test_merged_shards_equal_full_attention(ci, n):
    w = workload(CASES[ci], 210 + ci)
    wg = w.to("cuda")
    ref = oracle_from_torch(w)
    for splits in (0, 5):
        parts = [run_shard(wg, bt, su, ext, splits) for bt, su, ext in split_kv_shards(wg, n, seed=n)]
        out = va.merge_partials(parts)
        torch.cuda.synchronize()
        compare(out, ref)


def test_one_shard_is_verify_attn():
    w = workload(CASES[0], 220)
    wg = w.to("cuda")
    o, lse = run_shard(wg, wg.block_table, wg.seqused_k, None)
    out = va.merge_partials([(o, lse)])
    full = va.verify_attn(wg.q, wg.k_cache, wg.v_cache, wg.block_table, wg.cu_seqlens_q, wg.seqused_k,
                          wg.max_seqlen_q, wg.max_seqlen_k, wg.softmax_scale, wg.k_descale, wg.v_descale)
    torch.cuda.synchronize()
    diff = (out.float() - full.float()).abs().max().item()
    assert diff <= 1e-2, diff
    compare(out, oracle_from_torch(w))


def test_long_context_in_two_shards_every_sequence():
    w = named_workload("long_context_fp8", value_device="cuda").to("cuda")
    parts = [run_shard(w, bt, su, ext) for bt, su, ext in split_kv_shards(w, 2, seed=9)]
    out = va.merge_partials(parts)
    torch.cuda.synchronize()
    print("two shards", compare(out, oracle_from_torch(w.to("cpu"))))


def test_errors():
    w = workload(CASES[0], 230).to("cuda")
    with pytest.raises(va.VerifyAttnError) as e:
        va.verify_attn_partial(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                               w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale,
                               o=torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 3
    o = torch.zeros(w.q.shape, dtype=torch.float32, device="cuda")
    lse = torch.zeros(w.q.shape[:2], dtype=torch.float32, device="cuda")
    with pytest.raises(va.VerifyAttnError) as e:
        va.merge_partials([(o, lse)] * 17)
    assert e.value.status == 4
    with pytest.raises(va.VerifyAttnError) as e:
        va.merge_partials([(o, lse[:, :3])])
    assert e.value.status == 2
