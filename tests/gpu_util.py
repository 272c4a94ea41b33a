"""Helpers for the GPU parity tests: run the CUDA path through the C-ABI
binding and compare with the CPU oracle on the same bytes."""
from __future__ import annotations

import numpy as np
import torch

import speculative_decoding_verify_split_gb300 as va
from oracle.attention_fp64 import oracle_from_torch
from parity_gate import check_gates

# Tolerance on the bf16 output, from the pages' parity test (sglang PR 36330
# digest, unit test: assert_close(actual, expected, atol=1e-2, rtol=1e-2)).
ATOL = 1e-2
RTOL = 1e-2


def to_gpu(w):
    return w.to("cuda")


def run_gpu(w_gpu, ex=False, num_splits=0, stream=None) -> torch.Tensor:
    out = torch.full_like(w_gpu.q, float("nan"))
    if ex:
        va.run_workload_ex(w_gpu, out=out, num_splits=num_splits, stream=stream)
    else:
        va.run_workload(w_gpu, out=out, stream=stream)
    torch.cuda.synchronize()
    return out


def rows_of(w, seqs):
    cu = w.cu_seqlens_q.cpu().tolist()
    idx = []
    for b in seqs:
        idx.extend(range(cu[b], cu[b + 1]))
    return np.array(idx, dtype=np.int64)


def compare(got_bf16: torch.Tensor, ref: np.ndarray, rows=None) -> dict:
    """The pages' elementwise bound |got - ref| <= ATOL + RTOL * |ref| on the
    given q rows, and beside it the gates that scale with the output
    (parity_gate.check_gates: relative L2 error of the whole output and of
    every (token, head) row)."""
    got = got_bf16.to(torch.float64).cpu().numpy()
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert not np.isnan(ref).any(), "oracle rows missing"
    assert not np.isnan(got).any(), "NaN in GPU output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    stats = dict(max_abs=float(err.max()) if err.size else 0.0, n=int(err.size))
    stats.update(check_gates(got, ref))
    assert not bad.any(), f"{int(bad.sum())} of {err.size} elements out of tolerance; {stats}"
    return stats


def check_against_oracle(w_cpu, seqs=None, **run_kw) -> dict:
    w_gpu = to_gpu(w_cpu)
    got = run_gpu(w_gpu, **run_kw)
    ref = oracle_from_torch(w_cpu, seqs)
    rows = None if seqs is None else rows_of(w_cpu, seqs)
    return compare(got, ref, rows)
