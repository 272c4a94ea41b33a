"""The generic attention's variants on the GPU, through the C-ABI
(verify_attn_opt): sliding window, logit soft cap, attention sinks, alone and
together, on both KV types, against the CPU oracle with the parity tolerance
(atol = rtol = 1e-2 on the bf16 output)."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import make_workload, named_workload
from oracle.attention_fp64 import oracle_from_torch
from gpu_util import compare

pytestmark = pytest.mark.gpu


def run_opt(w, **kw):
    out = torch.full_like(w.q, float("nan"))
    va.verify_attn_opt(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                       w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale, w.v_descale,
                       out=out, **kw)
    torch.cuda.synchronize()
    return out


def oracle(w, seqs=None, window_left=-1, softcap=0.0, sinks=None):
    s = None if sinks is None else sinks.cpu().numpy().astype(np.float64)
    return oracle_from_torch(w.to("cpu"), seqs, window_left=window_left, softcap=softcap, sinks=s)


CASES = [
    dict(q=[4, 2, 3, 1, 4], kv=[1000, 769, 300, 5, 3], hq=16, hkv=1, dt="fp8_e4m3", kd=1.1, vd=0.8),
    dict(q=[2, 3, 4], kv=[2100, 513, 130], hq=32, hkv=2, dt="fp8_e4m3", kd=None, vd=None),
    dict(q=[2, 2, 1, 2], kv=[1500, 17, 64, 700], hq=8, hkv=1, dt="bf16", kd=None, vd=None),
]


def workload(case, seed):
    return make_workload(case["q"], case["kv"], case["hq"], case["hkv"], case["dt"], seed=seed,
                         k_descale=case["kd"], v_descale=case["vd"]).to("cuda")


@pytest.mark.parametrize("ci", range(len(CASES)))
@pytest.mark.parametrize("win", [0, 1, 15, 16, 17, 100, 257, 1000, 100000])
def test_window(ci, win):
    w = workload(CASES[ci], 71 + ci)
    compare(run_opt(w, window_left=win), oracle(w, window_left=win))


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_window_leaves_pages_before_it_unread(ci):
    """Pages wholly before every token's window may be unmapped in a
    sliding-window page table: invalid ids, or a page of NaN, give the same
    result as the real table."""
    w = workload(CASES[ci], 91 + ci)
    win = 40
    ref = oracle(w, window_left=win)
    bt = w.block_table.clone()
    poison = w.poison_page                                 # the workload's NaN page
    for b, (L, S) in enumerate(zip(CASES[ci]["q"], CASES[ci]["kv"])):
        first = max(0, S - L - win) // 16
        bt[b, :first] = torch.where(torch.arange(first, device="cuda") % 2 == 0,
                                    torch.full((first,), -1, dtype=torch.int32, device="cuda"),
                                    torch.full((first,), poison, dtype=torch.int32, device="cuda"))
    w.block_table = bt
    for splits in (0, 1, 7):
        n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, splits)
        ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
        got = run_opt(w, window_left=win, workspace=ws, num_splits=splits)
        compare(got, ref)
        assert va.workspace_status(ws) == 0


@pytest.mark.parametrize("ci", range(len(CASES)))
@pytest.mark.parametrize("cap", [1.5, 30.0])
def test_softcap(ci, cap):
    w = workload(CASES[ci], 101 + ci)
    w.q = w.q * 4                                          # logits large enough for the cap to bite
    compare(run_opt(w, softcap=cap), oracle(w, softcap=cap))


@pytest.mark.parametrize("ci", range(len(CASES)))
@pytest.mark.parametrize("splits", [1, 0, 9])
def test_sinks(ci, splits):
    """Direct rows (one split) and merged rows (several) add the sink once."""
    w = workload(CASES[ci], 111 + ci)
    hq = w.q.shape[1]
    g = torch.Generator().manual_seed(5)
    sinks = (torch.rand(hq, generator=g) * 10 - 5).to("cuda")
    sinks[0] = 12.0                                        # a sink that takes most of the mass
    n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, splits)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    got = run_opt(w, sinks=sinks, workspace=ws, num_splits=splits)
    compare(got, oracle(w, sinks=sinks))


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_all_variants_with_forced_splits(ci):
    w = workload(CASES[ci], 121 + ci)
    hq = w.q.shape[1]
    sinks = torch.linspace(-3, 3, hq, device="cuda")
    ref = oracle(w, window_left=300, softcap=20.0, sinks=sinks)
    for splits in (1, 2, 7, 64):
        n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, splits)
        ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
        got = run_opt(w, window_left=300, softcap=20.0, sinks=sinks, workspace=ws,
                      num_splits=splits)
        compare(got, ref)


def test_long_context_window_every_sequence():
    w = named_workload("long_context_fp8", value_device="cuda").to("cuda")
    got = run_opt(w, window_left=4096)
    print("window 4096", compare(got, oracle(w, window_left=4096)))


def test_options_are_validated():
    w = workload(CASES[0], 131)
    hq = w.q.shape[1]
    bad = [dict(window_left=-2), dict(softcap=-1.0), dict(softcap=float("inf")),
           dict(sinks=torch.zeros(hq + 1, device="cuda")),
           dict(sinks=torch.zeros(hq, dtype=torch.bfloat16, device="cuda"))]
    for kw in bad:
        with pytest.raises(va.VerifyAttnError):
            run_opt(w, **kw)


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes_and_variants(seed):
    """Seeded random batches: ragged lengths (including 0, 1 and page/tile
    edges), query lengths 1-4, head groupings, both KV types, random variant
    settings and forced split counts."""
    g = torch.Generator().manual_seed(1000 + seed)
    B = int(torch.randint(1, 9, (1,), generator=g))
    hkv = [1, 2, 4][int(torch.randint(0, 3, (1,), generator=g))]
    group = [1, 2, 4, 8, 16][int(torch.randint(0, 5, (1,), generator=g))]
    qmax = min(4, 64 // group)
    q_lens = torch.randint(1, qmax + 1, (B,), generator=g).tolist()
    choices = [0, 1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 500, 1000, 2500]
    kv_lens = [choices[int(i)] for i in torch.randint(0, len(choices), (B,), generator=g)]
    dt = ["fp8_e4m3", "bf16"][seed % 2]
    kd = float(torch.rand(1, generator=g) * 1.5 + 0.5) if dt == "fp8_e4m3" else None
    w = make_workload(q_lens, kv_lens, group * hkv, hkv, dt, seed=2000 + seed, k_descale=kd,
                      v_descale=kd).to("cuda")
    kw = {}
    if seed % 3 == 0:
        kw["window_left"] = int(torch.randint(0, 300, (1,), generator=g))
    if seed % 4 == 1:
        kw["softcap"] = float(torch.rand(1, generator=g) * 40 + 2)
    if seed % 2 == 1:
        kw["sinks"] = (torch.rand(group * hkv, generator=g) * 6 - 3).to("cuda")
    splits = [0, 1, 3, 200][seed % 4]
    n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, splits)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    got = run_opt(w, workspace=ws, num_splits=splits, **kw)
    compare(got, oracle(w, **kw))
    assert va.workspace_status(ws) == 0
