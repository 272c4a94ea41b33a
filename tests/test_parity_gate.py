"""The parity gates (tests/parity_gate.py) against plausible wrong results at
long-context lengths, on the CPU: oracle outputs of two sequences with the
long-context workload's lengths (64K-128K keys, 16 query heads on one FP8 KV
head, 4 draft tokens), and wrong results built from the oracle itself.

* one KV segment's keys dropped from one sequence (what a merge or partial
  indexing bug does), and the output at half its size: the pages'
  elementwise bound 1e-2 + 1e-2 |ref| passes both, the output-scaled gates
  fail both;
* the causal mask off by one on random keys: at these lengths the extra (or
  missing) key moves a row by ~1e-3 of its size, below the kernels' own
  rounding, so no tolerance sees it; the mask boundary is pinned exactly by
  inputs with a dominant key at the boundary. On such an input (a key that
  only the draft tokens t >= 1 may see, with a logit ~100 above the rest)
  both off-by-one directions fail the gates by orders of magnitude.
The GPU full-size parity tests use the same spiked input."""
import numpy as np
import pytest
import torch

from oracle.attention_fp64 import oracle_from_torch
from oracle.partial_fp64 import merge_partials, partial_oracle_from_torch
from parity_gate import REL_L2_MAX, gate_stats, gates_pass
from spikes import plant_boundary_spikes
from speculative_decoding_verify_split_gb300.workloads import PAGE_SIZE, make_workload

ATOL = RTOL = 1e-2
KV = [70001, 120003]     # within the long-context workload's range [65536, 131072]
SEGMENT = 10496          # one CTA's share of that workload's 1.6M keys over 152 SMs


def old_bound_passes(got, ref):
    return bool(np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)))


def shard_inputs(w, b, lo, hi):
    """Block table, lengths and extents of the shard holding keys [lo, hi) of
    sequence b (every other sequence whole)."""
    bt = w.block_table.clone()
    su = w.seqused_k.clone()
    ext = w.seqused_k.clone()
    p0 = lo // PAGE_SIZE
    n = (hi - lo + PAGE_SIZE - 1) // PAGE_SIZE
    bt[b, :n] = w.block_table[b, p0:p0 + n]
    su[b] = hi - lo
    ext[b] = w.kv_lens[b] - lo
    s = w.to("cpu")
    s.block_table, s.seqused_k = bt, su
    return s, ext


@pytest.fixture(scope="module")
def long_pair():
    w = make_workload([4, 4], KV, 16, 1, "fp8_e4m3", seed=41)
    return w, oracle_from_torch(w)


def test_dropped_segment_and_half_output(long_pair):
    w, ref = long_pair
    # the 120K-key sequence in three shards, the middle one a CTA's segment
    # (page-aligned). On the 70K-key one the elementwise bound flags 7 of its
    # 32,768 elements; here none (largest error 0.62 of the bound).
    a = 54000
    parts = []
    for lo, hi in ((0, a), (a, a + SEGMENT), (a + SEGMENT, KV[1])):
        s, ext = shard_inputs(w, 1, lo, hi)
        parts.append(partial_oracle_from_torch(s, ext, seqs=[1]))
    rows = slice(4, 8)
    full = merge_partials([o[rows] for o, _ in parts], [l[rows] for _, l in parts])
    assert np.abs(full - ref[rows]).max() < 1e-12   # the shards are exact
    dropped = ref.copy()
    dropped[rows] = merge_partials([parts[0][0][rows], parts[2][0][rows]],
                                   [parts[0][1][rows], parts[2][1][rows]])
    assert old_bound_passes(dropped, ref)
    assert not gates_pass(dropped, ref), gate_stats(dropped, ref)

    half = ref.copy()
    half[rows] *= 0.5          # that sequence's rows at half their size
    assert old_bound_passes(half, ref)
    assert not gates_pass(half, ref), gate_stats(half, ref)
    # a result rounded to bf16 (the kernels' output type) passes
    bf = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()
    assert gates_pass(bf, ref), gate_stats(bf, ref)


def test_mask_off_by_one_random_keys_is_below_rounding(long_pair):
    w, ref = long_pair
    ext = w.seqused_k + 1    # token t sees keys [0, S - L + t + 1]
    wrong, _ = partial_oracle_from_torch(w, ext)
    assert old_bound_passes(wrong, ref)
    s = gate_stats(wrong, ref)
    assert s["rel_l2"] < 0.5 * REL_L2_MAX, s    # no tolerance separates it from rounding


@pytest.mark.parametrize("shift", [+1, -1])
def test_mask_off_by_one_on_boundary_spikes(shift):
    w = plant_boundary_spikes(make_workload([4, 4], KV, 16, 1, "fp8_e4m3", seed=42))
    ref = oracle_from_torch(w)
    # the spike dominates the rows that see it: their output is its value row
    cu = w.cu_seqlens_q.tolist()
    for b, L in enumerate(w.q_lens):
        S = w.kv_lens[b]
        j = S - L + 1
        page = int(w.block_table[b, j // PAGE_SIZE])
        v = w.v_cache[page, j % PAGE_SIZE, 0].to(torch.float64).numpy()
        for t in range(1, L):
            assert np.abs(ref[cu[b] + t] - v[None, :]).max() < 1e-9
        assert np.abs(ref[cu[b]] - v[None, :]).max() > 0.5     # token 0 must not see it
    if shift > 0:    # token t sees keys [0, S - L + t + 1]
        wrong, _ = partial_oracle_from_torch(w, w.seqused_k + 1)
    else:            # token t sees keys [0, S - L + t - 1]: S one short
        short = w.to("cpu")
        short.seqused_k = w.seqused_k - 1
        wrong = oracle_from_torch(short)
    assert not gates_pass(wrong, ref), gate_stats(wrong, ref)
