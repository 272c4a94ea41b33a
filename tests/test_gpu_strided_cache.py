"""Caches that are views, as serving frameworks lay them out: K and V as the
two halves of one combined [pages, 2, 16, Hkv, D] tensor (page stride twice a
page), rows padded past the head dimension, and a latent cache whose 576-byte
rows sit in 640-byte ones. The tensor maps take the caller's strides, so the
kernels must read exactly the bytes of the contiguous layout: outputs equal
the contiguous call's bit for bit, and the oracle within the parity
tolerance."""
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from gpu_util import compare, to_gpu
from oracle.attention_fp64 import oracle_from_torch
from oracle.mla_fp64 import mla_oracle_from_torch
from speculative_decoding_verify_split_gb300.workloads import make_mla_workload, make_workload

pytestmark = pytest.mark.gpu


def _run(w):
    out = torch.full_like(w.q, float("nan"))
    va.run_workload(w, out=out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dt,hq,hkv", [("fp8_e4m3", 16, 1), ("bf16", 8, 1), ("fp8_e4m3", 32, 2)])
def test_combined_kv_tensor(dt, hq, hkv):
    w = make_workload([4, 2, 3, 1], [2100, 769, 130, 17], hq, hkv, dt, seed=41,
                      k_descale=0.9 if dt == "fp8_e4m3" else None)
    wg = to_gpu(w)
    ref_out = _run(wg)
    # one tensor holding K then V for every page
    kv = torch.empty((wg.k_cache.shape[0], 2) + tuple(wg.k_cache.shape[1:]), dtype=wg.k_cache.dtype,
                     device="cuda")
    kv[:, 0] = wg.k_cache
    kv[:, 1] = wg.v_cache
    wg.k_cache, wg.v_cache = kv[:, 0], kv[:, 1]
    assert not wg.k_cache.is_contiguous()
    got = _run(wg)
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16))
    compare(got, oracle_from_torch(w))


@pytest.mark.parametrize("dt", ["fp8_e4m3", "bf16"])
def test_padded_rows(dt):
    w = make_workload([4, 3], [1500, 600], 16, 1, dt, seed=43)
    wg = to_gpu(w)
    ref_out = _run(wg)
    pad = 32 if dt == "fp8_e4m3" else 16        # rows of 288 bytes (fp8) or 544 bytes (bf16)
    for name in ("k_cache", "v_cache"):
        c = getattr(wg, name)
        big = torch.zeros(tuple(c.shape[:-1]) + (c.shape[-1] + pad,), dtype=c.dtype, device="cuda")
        big[..., :c.shape[-1]] = c
        setattr(wg, name, big[..., :c.shape[-1]])
    got = _run(wg)
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16))
    compare(got, oracle_from_torch(w))


def _run_mla(w):
    out = torch.full((w.q.shape[0], w.q.shape[1], va.MLA_NOPE), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    va.run_mla_workload(w, out=out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dt", ["fp8_e4m3", "bf16"])
def test_latent_rows_in_wider_rows(dt):
    w = make_mla_workload([4, 2, 3], [1900, 700, 65], 16, kv_dtype=dt, seed=45, k_descale=1.1,
                          v_descale=0.8)
    wg = w.to("cuda")
    ref_out = _run_mla(wg)
    c = wg.kv_cache
    big = torch.zeros(tuple(c.shape[:-1]) + (640,), dtype=c.dtype, device="cuda")
    big[..., :576] = c
    wg.kv_cache = big[..., :576]
    got = _run_mla(wg)
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16))
    compare(got, mla_oracle_from_torch(w))
