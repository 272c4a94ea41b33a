"""The logit scale's degenerate cases on the GPU, against the CPU oracle with
the parity tolerance: a negative softmax scale (softmax of the negated
logits) and a zero one (uniform weights over each row's visible keys), beside
the usual positive scale, for the GQA kernel on both KV types, its variant
build (soft cap, window) and the latent-cache kernel on both cache types. The
kernels take the row max of the raw dot products and apply the scale after, so
a negative scale is folded into Q as it is staged; these cases pin that."""
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import make_mla_workload, make_workload
from oracle.attention_fp64 import oracle_from_torch
from oracle.mla_fp64 import mla_oracle_from_torch
from gpu_util import compare, run_gpu

pytestmark = pytest.mark.gpu

SCALES = [1 / 16, -1 / 16, 0.0]


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("dt,hq,hkv", [("fp8_e4m3", 16, 1), ("bf16", 8, 1), ("fp8_e4m3", 32, 2)])
def test_gqa(scale, dt, hq, hkv):
    w = make_workload([4, 2, 3, 1], [700, 129, 33, 1], hq, hkv, dt, seed=17, softmax_scale=scale,
                      k_descale=1.3 if dt == "fp8_e4m3" else None)
    compare(run_gpu(w.to("cuda")), oracle_from_torch(w))


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("kw", [dict(softcap=30.0), dict(window_left=100)])
def test_gqa_variants(scale, kw):
    w = make_workload([4, 2, 3], [900, 300, 17], 16, 1, "fp8_e4m3", seed=19, softmax_scale=scale)
    wg = w.to("cuda")
    out = torch.full_like(wg.q, float("nan"))
    va.verify_attn_opt(wg.q, wg.k_cache, wg.v_cache, wg.block_table, wg.cu_seqlens_q, wg.seqused_k,
                       wg.max_seqlen_q, wg.max_seqlen_k, wg.softmax_scale, wg.k_descale, wg.v_descale,
                       out=out, **kw)
    torch.cuda.synchronize()
    compare(out, oracle_from_torch(w, **kw))


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("dt", ["fp8_e4m3", "bf16"])
def test_latent(scale, dt):
    w = make_mla_workload([4, 2, 1], [700, 65, 3], 16, seed=23, kv_dtype=dt, softmax_scale=scale)
    wg = w.to("cuda")
    out = torch.full((wg.q.shape[0], wg.q.shape[1], va.MLA_NOPE), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    va.run_mla_workload(wg, out=out)
    torch.cuda.synchronize()
    compare(out, mla_oracle_from_torch(w))
