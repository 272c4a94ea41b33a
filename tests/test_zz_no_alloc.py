"""verify_attn_noalloc: the entry point for callers that cannot allocate
device memory (a runtime whose memory pool is fixed after start-up, an
allocator callback that must not re-enter the allocator). It keeps the
split-KV partials in an array built into the library instead of a workspace.

Checked through the C-ABI against verify_attn on the same inputs, on two
calls in a row (the second call finds the first call's partials still in the
array). Both entry points run the same plan and the same kernels, so the
outputs must be bit-identical; one case is also compared with the CPU oracle
within the parity tolerance the other GPU tests use. Collected last so that a
run stopping at the first failure has already run every other test; it also
passes alone in a fresh process."""
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from gpu_util import compare
from oracle.attention_fp64 import oracle_from_torch
from speculative_decoding_verify_split_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


def _call(fn, w, out):
    return fn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
              w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale, w.v_descale, out=out)


CASES = [
    dict(q=[4, 2, 3], kv=[3000, 769, 1500], hq=16, hkv=1, dt="fp8_e4m3", kd=0.9, vd=1.4),
    dict(q=[2, 3, 4, 2], kv=[2100, 513, 4000, 64], hq=32, hkv=2, dt="fp8_e4m3", kd=None, vd=None),
    dict(q=[2] * 6, kv=[2048, 9000, 300, 16, 17, 5000], hq=8, hkv=1, dt="bf16", kd=None, vd=None),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_noalloc_matches_verify_attn_twice(ci):
    case = CASES[ci]
    w_cpu = make_workload(case["q"], case["kv"], case["hq"], case["hkv"], case["dt"], seed=21,
                          k_descale=case["kd"], v_descale=case["vd"])
    w = w_cpu.to("cuda")
    ref = torch.empty_like(w.q)
    _call(va.verify_attn, w, ref)
    for _ in range(2):
        out = torch.full_like(w.q, float("nan"))
        _call(va.verify_attn_noalloc, w, out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    if ci == 0:
        compare(out, oracle_from_torch(w_cpu))


def test_noalloc_rejects_shapes_beyond_its_array():
    # 300 sequences x 64 packed rows need ~29 MiB of partials > 16 MiB.
    w = make_workload([4] * 300, [256] * 300, 16, 1, "fp8_e4m3", seed=22).to("cuda")
    out = torch.empty_like(w.q)
    with pytest.raises(va.VerifyAttnError) as e:
        _call(va.verify_attn_noalloc, w, out)
    assert e.value.status == 5      # VA_ERR_WORKSPACE, nothing launched
