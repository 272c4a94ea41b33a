"""The timeout path of the kernels' bounded waits, on the GPU, through the
C-ABI. Every wait of the main kernels (a ring slot, a copy landing, an MMA
finishing) gives up after a time limit; the kernel then stops issuing work,
lets its copies and MMAs in flight finish, frees its tensor memory and
returns, leaving a status bit in the workspace. Here the limit is cut to
1 ns (verify_attn_set_wait_limit), so waits run out on any input, and each
test checks that:

* the call returns and the stream synchronises without a CUDA error;
* verify_attn_last_device_error reports the bits, then reads 0 (cleared);
* with the default limit restored, the next call on the same workspace and
  on a fresh one matches the CPU oracle.

Covered: the GQA kernel on both KV types (many CTAs and one), the variant
kernel, a shard call, the latent-cache kernels (FP8 and BF16 caches), the
library's own workspace and the no-alloc array."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from gpu_util import compare
from oracle.attention_fp64 import oracle_from_torch
from oracle.mla_fp64 import mla_oracle_from_torch
from speculative_decoding_verify_split_gb300.workloads import make_mla_workload, make_workload

pytestmark = pytest.mark.gpu


class short_waits:
    """Every bounded wait of the launches inside runs out after 1 ns."""

    def __enter__(self):
        va.set_wait_limit(1)

    def __exit__(self, *exc):
        va.set_wait_limit(0)
        return False


def workspace_for(w, splits=0):
    n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, splits)
    return torch.zeros(n + 256, dtype=torch.uint8, device="cuda")


def timed_out_then_clear(ws=None):
    bits = va.last_device_error(ws)
    assert bits != 0, "no bounded wait reported running out"
    assert va.last_device_error(ws) == 0, "the status word was not cleared"
    return bits


@pytest.mark.parametrize("dt", ["fp8_e4m3", "bf16"])
def test_gqa_kernel_timeout(dt):
    w_cpu = make_workload([4, 3, 2, 4], [3000, 1500, 700, 9], 16, 1, dt, seed=301,
                          k_descale=0.9 if dt == "fp8_e4m3" else None)
    w = w_cpu.to("cuda")
    ws = workspace_for(w)
    with short_waits():
        for splits in (0, 1, 5):   # every SM, one CTA, a few
            va.run_workload_ex(w, out=torch.empty_like(w.q), workspace=ws, num_splits=splits)
        torch.cuda.synchronize()
    print(dt, "status bits", hex(timed_out_then_clear(ws)))
    ref = oracle_from_torch(w_cpu)
    for wsx in (ws, workspace_for(w)):
        out = torch.full_like(w.q, float("nan"))
        va.run_workload_ex(w, out=out, workspace=wsx)
        torch.cuda.synchronize()
        compare(out, ref)
        assert va.last_device_error(wsx) == 0


def test_variant_kernel_and_shard_timeout():
    w_cpu = make_workload([4, 2], [2000, 800], 16, 1, "fp8_e4m3", seed=302)
    w = w_cpu.to("cuda")
    ws = workspace_for(w)
    sinks = torch.zeros(16, dtype=torch.float32, device="cuda")
    with short_waits():
        va.verify_attn_opt(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                           w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, out=torch.empty_like(w.q),
                           window_left=300, softcap=20.0, sinks=sinks, workspace=ws)
        va.verify_attn_partial(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                               w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, workspace=ws)
        torch.cuda.synchronize()
    timed_out_then_clear(ws)
    got = torch.full_like(w.q, float("nan"))
    va.verify_attn_opt(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                       w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, out=got, window_left=300,
                       softcap=20.0, sinks=sinks, workspace=ws)
    torch.cuda.synchronize()
    compare(got, oracle_from_torch(w_cpu, window_left=300, softcap=20.0,
                                   sinks=np.zeros(16, dtype=np.float64)))
    assert va.last_device_error(ws) == 0


@pytest.mark.parametrize("dt", ["fp8_e4m3", "bf16"])
def test_latent_kernel_timeout(dt):
    m_cpu = make_mla_workload([4, 2, 3], [2500, 700, 130], 16, dt, seed=303, k_descale=1.1, v_descale=0.8)
    m = m_cpu.to("cuda")
    n = va.mla_workspace_size(m.q, m.seqused_k, m.max_seqlen_q, m.max_seqlen_k)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    with short_waits():
        for splits in (0, 1):
            va.run_mla_workload(m, workspace=ws, num_splits=splits)
        torch.cuda.synchronize()
    timed_out_then_clear(ws)
    out = torch.full((m.q.shape[0], m.q.shape[1], va.MLA_NOPE), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    va.run_mla_workload(m, out=out, workspace=ws)
    torch.cuda.synchronize()
    compare(out, mla_oracle_from_torch(m_cpu))
    assert va.last_device_error(ws) == 0


def test_library_scratch_timeout():
    """Calls without a workspace (the library's own) and the no-alloc entry:
    their status words are read and cleared through a NULL workspace."""
    w_cpu = make_workload([4, 3], [1200, 600], 16, 1, "fp8_e4m3", seed=304)
    w = w_cpu.to("cuda")
    ref = oracle_from_torch(w_cpu)
    va.run_workload(w, out=torch.empty_like(w.q))      # the library workspace exists
    torch.cuda.synchronize()
    va.last_device_error()                             # start from a clear word
    for fn in (va.verify_attn, va.verify_attn_noalloc):
        with short_waits():
            fn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
               w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, out=torch.empty_like(w.q))
            torch.cuda.synchronize()
        timed_out_then_clear(None)
        out = torch.full_like(w.q, float("nan"))
        fn(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
           w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, out=out)
        torch.cuda.synchronize()
        compare(out, ref)
        assert va.last_device_error() == 0


def test_status_query_argument_errors():
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    bits = __import__("ctypes").c_int32(0)
    lib = va.library()
    assert lib.verify_attn_last_device_error(None, None, None) == 1          # VA_ERR_NULL
    misaligned = va._workspace_addr(ws) + 4
    assert lib.verify_attn_last_device_error(misaligned, __import__("ctypes").byref(bits), None) == 5
