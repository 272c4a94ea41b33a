"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle,
element by element on the same seeded inputs, within atol = rtol = 1e-2 on
the bf16 output, plus the invariants that must hold exactly on the GPU."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from gpu_util import check_against_oracle, compare, run_gpu, to_gpu
from spikes import plant_boundary_spikes
from oracle.attention_fp64 import oracle_from_torch
from speculative_decoding_verify_split_gb300.workloads import make_workload, named_workload

pytestmark = pytest.mark.gpu


# --- the five verify workloads ---------------------------------------------

def test_tiny_verify_full():
    w = named_workload("tiny_verify")
    s = check_against_oracle(w)
    print("tiny_verify", s)


def test_gqa_32q2kv_full():
    w = named_workload("gqa_32q2kv")
    s = check_against_oracle(w)
    print("gqa_32q2kv", s)


FULL = ["mid_context_fp8", "long_context_fp8", "high_concurrency_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_sequence(name):
    """Full-size workload on the GPU (values drawn on the device) in the launch
    configuration the benchmark times, every sequence against the oracle."""
    w_gpu = named_workload(name, value_device="cuda").to("cuda")
    got = run_gpu(w_gpu)
    w_cpu = w_gpu.to("cpu")
    s = compare(got, oracle_from_torch(w_cpu))
    print(name, s)


@pytest.mark.parametrize("name", FULL)
def test_full_size_mask_boundary_spikes(name):
    """The same workloads with a dominant key at every sequence's mask
    boundary (visible to draft tokens t >= 1 only): a one-key mask error
    changes whole rows at any length."""
    w_gpu = plant_boundary_spikes(named_workload(name, value_device="cuda").to("cuda"))
    got = run_gpu(w_gpu)
    s = compare(got, oracle_from_torch(w_gpu.to("cpu")))
    print(name, "spiked", s)


# --- sweeps over the row packing --------------------------------------------

@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "bf16"])
@pytest.mark.parametrize("group,hkv", [(1, 1), (2, 2), (4, 1), (8, 2), (16, 1), (16, 2)])
@pytest.mark.parametrize("qlen", [1, 2, 3, 4])
def test_sweep_rows(kv_dtype, group, hkv, qlen):
    kv = [1, 15, 16, 17, 100, 333, 700]
    ql = [qlen] * len(kv)
    ql[0] = min(qlen, 1)
    w = make_workload(ql, kv, group * hkv, hkv, kv_dtype, seed=group * 10 + qlen,
                      k_descale=0.8 if kv_dtype == "fp8_e4m3" else None,
                      v_descale=1.3 if kv_dtype == "fp8_e4m3" else None)
    check_against_oracle(w)


def test_mixed_qlens_and_large_group():
    w = make_workload([4, 1, 3, 2, 4], [2000, 5, 513, 64, 1031], 16, 1, "fp8_e4m3", seed=3)
    check_against_oracle(w)


# --- split-KV decomposition -------------------------------------------------

@pytest.mark.parametrize("splits", [1, 2, 7, 64, 500])
def test_forced_splits_match_oracle(splits):
    w = make_workload([4, 2, 3], [3000, 769, 1500], 16, 1, "fp8_e4m3", seed=5)
    check_against_oracle(w, ex=True, num_splits=splits)


def test_split_count_invariance():
    w = to_gpu(make_workload([4, 4], [5000, 4000], 16, 1, "fp8_e4m3", seed=6))
    outs = [run_gpu(w, ex=True, num_splits=s).float() for s in (1, 2, 7, 64, 300)]
    for o in outs[1:]:
        assert torch.allclose(o, outs[0], atol=2e-3, rtol=2e-2)


def test_run_to_run_bit_identical():
    w = to_gpu(make_workload([4, 3, 2], [4000, 2500, 900], 16, 1, "fp8_e4m3", seed=8))
    a = run_gpu(w)
    for _ in range(3):
        assert torch.equal(run_gpu(w).view(torch.int16), a.view(torch.int16))


def test_page_permutation_bit_identical():
    w = make_workload([4, 3], [1500, 900], 16, 1, "fp8_e4m3", seed=9)
    a = run_gpu(to_gpu(w))
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(4))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    w.k_cache = w.k_cache.view(torch.uint8)[inv].view(torch.float8_e4m3fn)
    w.v_cache = w.v_cache.view(torch.uint8)[inv].view(torch.float8_e4m3fn)
    w.block_table = perm[w.block_table.long()].to(torch.int32)
    b = run_gpu(to_gpu(w))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_gqa_equals_expanded_mha_on_gpu():
    w = make_workload([3, 2], [400, 230], 8, 2, "fp8_e4m3", seed=7)
    m = make_workload([3, 2], [400, 230], 8, 2, "fp8_e4m3", seed=7)
    m.k_cache = w.k_cache.view(torch.uint8).repeat_interleave(4, dim=2).view(torch.float8_e4m3fn)
    m.v_cache = w.v_cache.view(torch.uint8).repeat_interleave(4, dim=2).view(torch.float8_e4m3fn)
    a = run_gpu(to_gpu(w)).float()
    b = run_gpu(to_gpu(m)).float()
    assert torch.allclose(a, b, atol=2e-3, rtol=2e-2)


# --- edge cases ---------------------------------------------------------------

def test_rows_without_visible_keys_are_zero():
    w = make_workload([4, 2, 3], [2, 0, 40], 16, 1, "fp8_e4m3", seed=10)
    out = run_gpu(to_gpu(w))
    assert torch.all(out[0:2] == 0) and torch.all(out[4:6] == 0)
    ref = oracle_from_torch(w)
    compare(out, ref)


def test_sequence_without_draft_tokens():
    w = make_workload([3, 0, 2], [100, 50, 70], 16, 1, "fp8_e4m3", seed=12)
    check_against_oracle(w)


def test_empty_batch_and_empty_query():
    w = to_gpu(make_workload([], [], 16, 1, "fp8_e4m3", seed=1))
    out = torch.empty(0, 16, 256, dtype=torch.bfloat16, device="cuda")
    va.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                   1, 0, 0.0625, out=out)
    torch.cuda.synchronize()


def test_descales_are_applied():
    w = make_workload([3, 4], [600, 300], 16, 1, "fp8_e4m3", seed=13, k_descale=0.55, v_descale=1.9)
    check_against_oracle(w)


def test_strided_q_and_out():
    w = make_workload([4, 2], [300, 200], 16, 1, "fp8_e4m3", seed=14)
    ref = oracle_from_torch(w)
    wg = to_gpu(w)
    big = torch.zeros(wg.q.shape[0], 16, 512, dtype=torch.bfloat16, device="cuda")
    big[..., :256] = wg.q
    wg.q = big[..., :256]
    out_big = torch.full((wg.q.shape[0], 16, 768), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = out_big[..., 256:512]
    va.run_workload(wg, out=out)
    torch.cuda.synchronize()
    compare(out, ref)
    assert torch.isnan(out_big[..., :256].float()).all()


@pytest.mark.parametrize("splits", [0, 1])
def test_out_rows_16_byte_aligned(splits):
    """Output rows 16- but not 32-byte aligned (row stride 528 B, base 16 B into
    a row): rows written directly (one split: every item) take 16-byte stores."""
    w = make_workload([4, 2, 3], [300, 200, 1000], 16, 1, "fp8_e4m3", seed=16)
    ref = oracle_from_torch(w)
    wg = to_gpu(w)
    out_big = torch.full((wg.q.shape[0], 16, 264), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = out_big[..., 8:264]
    va.run_workload_ex(wg, out=out, num_splits=splits)
    torch.cuda.synchronize()
    compare(out, ref)
    assert torch.isnan(out_big[..., :8].float()).all()


def test_side_stream():
    w = make_workload([4, 2], [800, 600], 16, 1, "fp8_e4m3", seed=15)
    s = torch.cuda.Stream()
    wg = to_gpu(w)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = torch.full_like(wg.q, float("nan"))
        va.run_workload(wg, out=out, stream=s)
    s.synchronize()
    compare(out, oracle_from_torch(w))


def test_bad_arguments_raise_before_launch():
    w = to_gpu(make_workload([4, 2], [100, 60], 16, 1, "fp8_e4m3", seed=16))
    with pytest.raises(va.VerifyAttnError) as e:
        va.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                       5, w.max_seqlen_k, 0.0625)
    assert e.value.status == 4
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(va.VerifyAttnError) as e:
        va.run_workload_ex(w, workspace=ws)
    assert e.value.status == 5


def test_out_of_range_page_ids_do_not_fault():
    """A corrupt block table (ids past the cache) must not read out of bounds;
    the affected rows are unspecified but the call completes."""
    w = make_workload([2], [64], 16, 1, "fp8_e4m3", seed=17)
    w.block_table[0, 1] = 10**6
    wg = to_gpu(w)
    run_gpu(wg)


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "bf16"])
def test_more_items_than_threads(kv_dtype):
    """1000 (sequence, KV head) items: more than one per thread of a CTA, so
    the work scan takes its two-pass path."""
    g = torch.Generator().manual_seed(77)
    B = 500
    q_lens = torch.randint(1, 5, (B,), generator=g).tolist()
    kv_lens = torch.randint(1, 400, (B,), generator=g).tolist()
    w = make_workload(q_lens, kv_lens, 8, 2, kv_dtype, seed=78)
    assert w.num_seqs * w.num_kv_heads > 416
    check_against_oracle(w)


def test_one_sequence_of_a_million_keys():
    """A single work item split over every SM: the merge combines one segment
    per CTA; the block table is 62,500 pages wide."""
    w = make_workload([4], [1_000_000], 16, 1, "fp8_e4m3", seed=79, value_device="cuda")
    wg = w.to("cuda")
    got = run_gpu(wg)
    ref = oracle_from_torch(wg.to("cpu"))
    compare(got, ref)


def test_no_bounded_wait_timed_out():
    """The tensor-core kernel bounds every wait; a timeout sets a status bit in
    the workspace. None may be set on a normal run."""
    w = to_gpu(make_workload([4, 3, 2, 4], [9000, 2500, 900, 70], 16, 1, "fp8_e4m3", seed=18))
    n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    for splits in (0, 3, 40):
        va.run_workload_ex(w, out=torch.empty_like(w.q), workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    assert va.workspace_status(ws) == 0
