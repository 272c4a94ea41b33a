"""The FP8 main kernel's two layouts. Batches of at least 16 key tiles per
CTA run with Q and P in tensor memory (one S tile, four K ring slots: the
plan's kernel 2); smaller batches and the variant options with Q in shared
memory (two S tiles, each P written over its S: kernel 1). A split count
forced low puts small inputs on the first layout, so that the row-packing
sweep, the bit-identity invariants and agreement with the other layout are
checked on it as well."""
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from gpu_util import check_against_oracle, compare, run_gpu, to_gpu
from oracle.attention_fp64 import oracle_from_torch
from speculative_decoding_verify_split_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


def _layout(w, splits):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return va.plan(w.num_seqs, w.k_cache.shape[2], w.q.shape[1], w.max_seqlen_q, w.max_seqlen_k,
                   w.kv_dtype, sms, force_splits=splits)["kernel"]


@pytest.mark.parametrize("group,hkv", [(1, 1), (2, 2), (4, 1), (8, 2), (16, 1), (16, 2)])
@pytest.mark.parametrize("qlen", [1, 2, 3, 4])
def test_sweep_rows_q_in_tmem(group, hkv, qlen):
    kv = [1, 15, 16, 17, 100, 333, 700, 2100]
    ql = [qlen] * len(kv)
    ql[0] = min(qlen, 1)
    w = make_workload(ql, kv, group * hkv, hkv, "fp8_e4m3", seed=100 + group * 10 + qlen,
                      k_descale=0.8, v_descale=1.3)
    assert _layout(w, 2) == 2
    check_against_oracle(w, ex=True, num_splits=2)


def test_run_to_run_bit_identical_q_in_tmem():
    w = make_workload([4, 3, 2], [4000, 2500, 900], 16, 1, "fp8_e4m3", seed=8)
    assert _layout(w, 3) == 2
    wg = to_gpu(w)
    a = run_gpu(wg, ex=True, num_splits=3)
    for _ in range(3):
        assert torch.equal(run_gpu(wg, ex=True, num_splits=3).view(torch.int16), a.view(torch.int16))
    compare(a, oracle_from_torch(w))


def test_page_permutation_bit_identical_q_in_tmem():
    w = make_workload([4, 3], [3000, 1900], 16, 1, "fp8_e4m3", seed=9)
    assert _layout(w, 2) == 2
    a = run_gpu(to_gpu(w), ex=True, num_splits=2)
    nb = w.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(4))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    w.k_cache = w.k_cache.view(torch.uint8)[inv].view(torch.float8_e4m3fn)
    w.v_cache = w.v_cache.view(torch.uint8)[inv].view(torch.float8_e4m3fn)
    w.block_table = perm[w.block_table.long()].to(torch.int32)
    b = run_gpu(to_gpu(w), ex=True, num_splits=2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("splits", [1, 2])
def test_layouts_agree(splits):
    """The same split once with Q in tensor memory (a plain call) and once with
    Q in shared memory (the variant kernel, with a window wider than every
    sequence so that no key is masked): the same products and sums in the same
    order, so the same bits."""
    w = make_workload([4, 2, 3], [3000, 769, 1500], 16, 1, "fp8_e4m3", seed=5, k_descale=1.2)
    assert _layout(w, splits) == 2
    wg = to_gpu(w)
    a = run_gpu(wg, ex=True, num_splits=splits)
    b = torch.full_like(wg.q, float("nan"))
    ws = torch.zeros(va.workspace_size(wg.q, wg.k_cache, wg.seqused_k, wg.max_seqlen_q, wg.max_seqlen_k,
                                       splits) + 256, dtype=torch.uint8, device="cuda")
    va.verify_attn_opt(wg.q, wg.k_cache, wg.v_cache, wg.block_table, wg.cu_seqlens_q, wg.seqused_k,
                       wg.max_seqlen_q, wg.max_seqlen_k, wg.softmax_scale, wg.k_descale, wg.v_descale,
                       out=b, window_left=1 << 20, workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    diff = (a.float() - b.float()).abs().max().item()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"max |diff| {diff}"
    compare(a, oracle_from_torch(w))
