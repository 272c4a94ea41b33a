"""Parity gates that scale with the output, applied beside the pages'
elementwise bound |got - ref| <= 1e-2 + 1e-2 |ref| (sglang PR 36330 digest,
"Key code excerpts": the unit test's assert_close(atol=1e-2, rtol=1e-2)).

Why a second gate: an attention row over n visible keys has entries of size
about 1 / sqrt(n) (about 0.005 at 70K keys), so at long context the
elementwise bound is looser than the output itself. A result at half its
right size, or one that lost a whole KV segment's keys, passes it. These
gates bound the error relative to the output:

* REL_L2_MAX: ||got - ref|| / ||ref|| over the whole compared output;
* ROW_REL_L2_MAX: the same per (token, head) row (the last axis), so that one
  wrong sequence among hundreds cannot hide in the total;
* a row whose reference is exactly 0 (it sees no key) must be exactly 0.

The kernels' own error is about 2e-3 relative (bf16 output rounding alone is
up to 2^-9 per element); the limits leave it a factor of 5 or more.
Numpy only: the CPU tests use it on oracle outputs."""
from __future__ import annotations

import numpy as np

REL_L2_MAX = 1e-2
ROW_REL_L2_MAX = 2e-2


def gate_stats(got: np.ndarray, ref: np.ndarray) -> dict:
    """Relative L2 errors of the whole array and of its rows (last axis)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    width = ref.shape[-1] if ref.ndim else 1
    d2 = d.reshape(-1, width)
    r2 = ref.reshape(-1, width)
    row_err = np.linalg.norm(d2, axis=1)
    row_ref = np.linalg.norm(r2, axis=1)
    zero = row_ref == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        row_rel = np.where(zero, 0.0, row_err / np.where(zero, 1.0, row_ref))
    tot_ref = float(np.linalg.norm(r2))
    return dict(rel_l2=float(np.linalg.norm(d2)) / tot_ref if tot_ref > 0 else float(np.linalg.norm(d2)),
                row_rel_l2_max=float(row_rel.max()) if row_rel.size else 0.0,
                zero_rows=int(zero.sum()),
                zero_rows_nonzero=int((zero & (row_err > 0)).sum()))


def gates_pass(got: np.ndarray, ref: np.ndarray) -> bool:
    s = gate_stats(got, ref)
    return (s["rel_l2"] <= REL_L2_MAX and s["row_rel_l2_max"] <= ROW_REL_L2_MAX
            and s["zero_rows_nonzero"] == 0)


def check_gates(got: np.ndarray, ref: np.ndarray) -> dict:
    """Asserts the gates; returns the statistics."""
    s = gate_stats(got, ref)
    assert s["rel_l2"] <= REL_L2_MAX, f"relative L2 error {s['rel_l2']:.3e} > {REL_L2_MAX}; {s}"
    assert s["row_rel_l2_max"] <= ROW_REL_L2_MAX, \
        f"a row's relative L2 error {s['row_rel_l2_max']:.3e} > {ROW_REL_L2_MAX}; {s}"
    assert s["zero_rows_nonzero"] == 0, f"rows that see no key are not 0; {s}"
    return s
