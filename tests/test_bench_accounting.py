"""bench.py's byte accounting, on the CPU: the per-sequence bytes the CPU
baseline is scaled by sum to the workload's algorithmic bytes (K and V once
per KV head, Q in and out), for the GQA and latent layouts, and a sliding
window's bytes reach them exactly when the window covers every key."""
import importlib.util
import os
from types import SimpleNamespace

import pytest

from speculative_decoding_verify_split_gb300.workloads import (
    MLA_WORKLOADS, WORKLOADS, make_mla_workload, make_workload, mla_workload_structure,
    workload_sizes)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_for_accounting", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _shape(name):
    s = workload_sizes(name)
    return SimpleNamespace(kv_dtype=s["kv_dtype"], kv_lens=s["kv_lens"], q_lens=s["q_lens"],
                           num_kv_heads=s["Hkv"], num_q_heads=s["Hq"]), s["algorithmic_bytes"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_sequence_bytes_sum_to_the_workload(name):
    bench = _bench()
    w, total = _shape(name)
    assert sum(bench.seq_bytes(w, b, False) for b in range(len(w.kv_lens))) == total


def test_sequence_bytes_of_built_workloads():
    bench = _bench()
    w = make_workload([4, 1, 3], [700, 16, 33], 8, 2, "fp8_e4m3", seed=1)
    assert sum(bench.seq_bytes(w, b, False) for b in range(3)) == w.algorithmic_bytes()
    m = make_mla_workload([4, 2], [300, 17], 16, seed=2)
    assert sum(bench.seq_bytes(m, b, True) for b in range(2)) == m.algorithmic_bytes()


@pytest.mark.parametrize("name", WORKLOADS)
def test_window_bytes(name):
    bench = _bench()
    w, total = _shape(name)
    assert bench.window_bytes(w, max(w.kv_lens)) == total
    assert bench.window_bytes(w, 4096) <= total
    # a zero window: each draft token sees only itself, so the last q_len keys
    e = 1 if w.kv_dtype == "fp8_e4m3" else 2
    kv0 = sum(min(s, l) for s, l in zip(w.kv_lens, w.q_lens)) * w.num_kv_heads * 256 * 2 * e
    qo = 2 * sum(w.q_lens) * w.num_q_heads * 256 * 2
    assert bench.window_bytes(w, 0) == kv0 + qo


def test_throughput_is_whole_job():
    bench = _bench()
    assert bench.throughput(10**9, 1, 1.0) == pytest.approx(1000.0)
    assert bench.throughput(10**9, 4, 2.0) == pytest.approx(2000.0)


@pytest.mark.parametrize("name", ["tiny_verify", "gqa_32q2kv", "mla_tiny", "mla_tiny_bf16"])
@pytest.mark.parametrize("world", [1, 4])
def test_reference_arm_reports_our_config(name, world):
    """The reference arm (the oracle on the host cores) reports the same
    config block as our arm, computed from the seeded structure alone."""
    from speculative_decoding_verify_split_gb300.workloads import named_mla_workload, named_workload
    b = _bench()
    w = named_mla_workload(name) if name.startswith("mla_") else named_workload(name)
    assert b.reference_config(name, world) == b.workload_config(w, name, world)


@pytest.mark.parametrize("name", sorted(WORKLOADS) + list(MLA_WORKLOADS))
def test_reference_bytes_match_the_structure(name):
    b = _bench()
    _, _, alg = b.reference_structure(name)
    if name in WORKLOADS:
        assert alg == workload_sizes(name)["algorithmic_bytes"]
    else:
        st = mla_workload_structure(name)
        w = make_mla_workload([1] * len(st["q_lens"]), [1] * len(st["kv_lens"]), st["Hq"],
                              st.get("kv_dtype", "fp8_e4m3"), seed=0)
        e = 1 if st.get("kv_dtype", "fp8_e4m3") == "fp8_e4m3" else 2
        per_key, per_token = 576 * e, st["Hq"] * (576 + 512) * 2
        assert w.algorithmic_bytes() == len(st["kv_lens"]) * per_key + len(st["q_lens"]) * per_token
        assert alg == sum(st["kv_lens"]) * per_key + sum(st["q_lens"]) * per_token
