"""The latent-cache (absorbed-MLA) path on the GPU, through the C-ABI
(verify_attn_mla), against the CPU oracle oracle/mla_fp64.py with the parity
tolerance (atol = rtol = 1e-2 on the bf16 output):

* the small workload whole, at the library's split and at forced split
  counts from 1 CTA to more CTAs than tiles;
* seeded random batches: ragged lengths (0, 1, page and tile edges), 1-4
  draft tokens, 1 to 64 heads, descales, forced splits;
* bit-identical results run to run, under a relabelling of the physical
  pages, and between CUDA-graph replays and eager calls;
* the long-context workload (16 sequences of 64K-128K keys), every
  sequence, in the launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import make_mla_workload, named_mla_workload
from oracle.mla_fp64 import mla_oracle_from_torch
from gpu_util import compare

pytestmark = pytest.mark.gpu


def run(w, num_splits=0, ws=True):
    out = torch.full((w.q.shape[0], w.q.shape[1], va.MLA_NOPE), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    workspace = None
    if ws:
        n = va.mla_workspace_size(w.q, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, num_splits)
        workspace = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    va.run_mla_workload(w, out=out, workspace=workspace, num_splits=num_splits)
    torch.cuda.synchronize()
    if workspace is not None:
        assert va.workspace_status(workspace) == 0
    return out


@pytest.fixture(scope="module")
def tiny():
    w = named_mla_workload("mla_tiny")
    return w, w.to("cuda"), mla_oracle_from_torch(w)


@pytest.mark.parametrize("splits", [0, 1, 2, 7, 64, 1000])
def test_tiny_whole(tiny, splits):
    w, wg, ref = tiny
    compare(run(wg, splits), ref)


def test_library_workspace(tiny):
    w, wg, ref = tiny
    compare(run(wg, ws=False), ref)


def test_run_to_run_and_page_relabelling_bit_identical():
    w = make_mla_workload([4, 3, 1], [3000, 700, 129], 16, seed=21, k_descale=0.8, v_descale=1.7)
    wg = w.to("cuda")
    a = run(wg)
    for _ in range(3):
        assert torch.equal(run(wg).view(torch.int16), a.view(torch.int16))
    # move every page to a new physical slot
    nb = wg.kv_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(3)).to("cuda")
    kv2 = torch.empty_like(wg.kv_cache)
    kv2[perm] = wg.kv_cache
    w2 = w.to("cuda")
    w2.kv_cache = kv2
    w2.block_table = perm.to(torch.int32)[wg.block_table.long()]
    assert torch.equal(run(w2).view(torch.int16), a.view(torch.int16))
    compare(a, mla_oracle_from_torch(w))


@pytest.mark.parametrize("seed", range(14))
def test_random_shapes(seed):
    g = torch.Generator().manual_seed(500 + seed)
    B = int(torch.randint(1, 7, (1,), generator=g))
    hq = [1, 2, 4, 8, 16, 32, 64][int(torch.randint(0, 7, (1,), generator=g))]
    qmax = min(4, 64 // hq)
    q_lens = torch.randint(1, qmax + 1, (B,), generator=g).tolist()
    choices = [0, 1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 500, 1000, 2500]
    kv_lens = [choices[int(i)] for i in torch.randint(0, len(choices), (B,), generator=g)]
    kd = float(torch.rand(1, generator=g) * 1.5 + 0.5)
    vd = float(torch.rand(1, generator=g) * 1.5 + 0.5)
    w = make_mla_workload(q_lens, kv_lens, hq, seed=600 + seed, k_descale=kd, v_descale=vd)
    splits = [0, 1, 3, 200][seed % 4]
    compare(run(w.to("cuda"), splits), mla_oracle_from_torch(w))


def test_peaked_softmax_and_rescales():
    """Queries scaled up so that row maxima jump across tiles (O^T rescales)
    and single keys dominate (P near the top of its range)."""
    w = make_mla_workload([4, 2, 3], [2000, 4100, 600], 16, seed=31)
    w.q = (w.q.to(torch.float32) * 6).to(torch.bfloat16)
    for splits in (1, 0, 11):
        compare(run(w.to("cuda"), splits), mla_oracle_from_torch(w))


def test_long_context_every_sequence():
    w = named_mla_workload("mla_long_context_fp8", value_device="cuda")
    got = run(w.to("cuda"))
    print("mla_long_context_fp8", compare(got, mla_oracle_from_torch(w.to("cpu"))))


def test_many_sequences_eight_row_merge():
    """64 short sequences of 3 draft tokens x 16 heads: 768 four-row merge
    CTAs, more than one wave, so the merge takes eight rows per CTA."""
    g = np.random.default_rng(5)
    kv = [int(x) for x in g.integers(64, 600, size=64)]
    w = make_mla_workload([3] * 64, kv, 16, seed=23, k_descale=1.2, v_descale=0.9)
    compare(run(w.to("cuda")), mla_oracle_from_torch(w))


def test_errors():
    w = make_mla_workload([2], [100], 16, seed=41).to("cuda")
    with pytest.raises(va.VerifyAttnError) as e:   # 16 heads x 5 tokens > 64 rows
        va.verify_attn_mla(w.q, w.kv_cache, w.block_table, w.cu_seqlens_q, w.seqused_k, 5,
                           w.max_seqlen_k, w.softmax_scale)
    assert e.value.status == 4
    with pytest.raises(va.VerifyAttnError) as e:   # an fp32 latent cache
        va.verify_attn_mla(w.q, w.kv_cache.to(torch.float32), w.block_table, w.cu_seqlens_q,
                           w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale)
    assert e.value.status == 3


# --- a BF16 latent cache (the BF16 kernel: 32-key tiles, Q in shared memory) ---

@pytest.mark.parametrize("splits", [0, 1, 2, 7, 64, 1000])
def test_bf16_tiny_whole(splits):
    w = named_mla_workload("mla_tiny_bf16")
    compare(run(w.to("cuda"), splits), mla_oracle_from_torch(w))


@pytest.mark.parametrize("seed", range(10))
def test_bf16_random_shapes(seed):
    """Ragged lengths (0, 1, page and tile edges), 1-4 draft tokens, 1 to 64
    heads, descales, forced splits, on a BF16 latent cache."""
    g = torch.Generator().manual_seed(900 + seed)
    B = int(torch.randint(1, 7, (1,), generator=g))
    hq = [1, 2, 4, 8, 16, 32, 64][int(torch.randint(0, 7, (1,), generator=g))]
    qmax = min(4, 64 // hq)
    q_lens = torch.randint(1, qmax + 1, (B,), generator=g).tolist()
    choices = [0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 500, 1000, 2500]
    kv_lens = [choices[int(i)] for i in torch.randint(0, len(choices), (B,), generator=g)]
    kd = float(torch.rand(1, generator=g) * 1.5 + 0.5)
    vd = float(torch.rand(1, generator=g) * 1.5 + 0.5)
    w = make_mla_workload(q_lens, kv_lens, hq, "bf16", seed=950 + seed, k_descale=kd, v_descale=vd)
    splits = [0, 1, 3, 200][seed % 4]
    compare(run(w.to("cuda"), splits), mla_oracle_from_torch(w))


def test_bf16_peaked_softmax_and_bit_identity():
    """Queries scaled up so that row maxima jump across tiles (O^T rescales);
    results bit-identical run to run and under a relabelling of the pages."""
    w = make_mla_workload([4, 2, 3], [2000, 4100, 600], 16, "bf16", seed=931)
    w.q = (w.q.to(torch.float32) * 6).to(torch.bfloat16)
    ref = mla_oracle_from_torch(w)
    wg = w.to("cuda")
    a = run(wg, 11)
    compare(a, ref)
    assert torch.equal(run(wg, 11).view(torch.int16), a.view(torch.int16))
    nb = wg.kv_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5)).to("cuda")
    kv2 = torch.empty_like(wg.kv_cache)
    kv2[perm] = wg.kv_cache
    w2 = w.to("cuda")
    w2.kv_cache = kv2
    w2.block_table = perm.to(torch.int32)[wg.block_table.long()]
    assert torch.equal(run(w2, 11).view(torch.int16), a.view(torch.int16))


def test_bf16_long_context_every_sequence():
    w = named_mla_workload("mla_long_context_bf16", value_device="cuda")
    got = run(w.to("cuda"))
    print("mla_long_context_bf16", compare(got, mla_oracle_from_torch(w.to("cpu"))))


@pytest.mark.parametrize("hq,q_lens", [(64, [1, 1, 1]), (32, [2, 1]), (1, [4, 3, 1]), (2, [1, 4])])
def test_head_counts(hq, q_lens):
    """Group sizes from 1 to 64 query heads on the one latent (rows = heads x
    draft tokens <= 64), at the library's split and split over many CTAs."""
    w = make_mla_workload(q_lens, [700, 129, 2000][:len(q_lens)], hq, seed=50 + hq, k_descale=1.2,
                          v_descale=0.9)
    ref = mla_oracle_from_torch(w)
    for splits in (0, 37):
        compare(run(w.to("cuda"), splits), ref)


def test_cuda_graph_replay_bit_identical():
    """With a caller workspace the call allocates and synchronises nothing, so
    it can be captured; replays on new query values match eager calls bit
    for bit."""
    w = make_mla_workload([4, 2, 3], [3000, 200, 1100], 16, seed=61).to("cuda")
    n = va.mla_workspace_size(w.q, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    out = torch.empty(w.q.shape[0], w.q.shape[1], va.MLA_NOPE, dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        va.run_mla_workload(w, out=out, workspace=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        va.run_mla_workload(w, out=out, workspace=ws, stream=torch.cuda.current_stream())
    gen = torch.Generator(device="cuda").manual_seed(7)
    for _ in range(3):
        w.q.copy_(torch.randn(w.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        ref = torch.empty_like(out)
        va.run_mla_workload(w, out=ref, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
