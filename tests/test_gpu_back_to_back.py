"""Back-to-back calls with no synchronisation between them.

The main kernels are programmatic dependents of the stream's previous kernel:
they initialise their barriers, allocate TMEM and prefetch the tensor-map
descriptors while that kernel ends, and wait for its completion before they
read Q, the lengths or the block table or touch the workspace. Here every call
is preceded, in the same stream, by copies of another batch's cache and block
table and by small torch kernels that rewrite seqused_k and Q in place (Q last,
so the kernel right before each call writes what it reads), and consecutive
calls share one workspace. Each output must equal bit for bit the same call
made alone after a synchronize; a main kernel that read before the previous
kernel finished would see the other batch's Q or lengths, and one that wrote
the workspace early would corrupt the previous call's merge."""
import dataclasses

import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import make_mla_workload, make_workload

pytestmark = pytest.mark.gpu

Q_LENS = [4, 2, 3, 1, 4]
KV_LENS = [3000, 769, 1500, 40, 2100]
SHORTER = [37, 300, 5, 0, 1999]   # batch B's seqused_k = batch A's minus these


def _batches(make):
    a = make(seed=41).to("cuda")
    b = make(seed=42).to("cuda")
    su = torch.tensor([max(k - d, q) for k, d, q in zip(KV_LENS, SHORTER, Q_LENS)], dtype=torch.int32)
    b.seqused_k = su.to("cuda")
    b.kv_lens = su.tolist()
    assert a.block_table.shape == b.block_table.shape and a.q.shape == b.q.shape
    return a, b


def _run_alternating(a, b, names, call, n_calls=8):
    """Calls `call(dst, out, ws)` n_calls times on dst buffers alternately
    refilled from a and b, with no synchronisation; returns the outputs and
    the two references (each batch called alone)."""
    dst = dataclasses.replace(a, **{k: getattr(a, k).clone() for k in names})
    n = call.workspace_size(dst)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    refs = []
    for src in (a, b):
        out = call(src, None, ws)
        torch.cuda.synchronize()
        refs.append(out.clone())
    outs = []
    for i in range(n_calls):
        src = a if i % 2 == 0 else b
        for k in names:
            if k not in ("q", "seqused_k"):
                getattr(dst, k).copy_(getattr(src, k))
        torch.add(src.seqused_k, 0, out=dst.seqused_k)          # a kernel, not a copy
        torch.mul(src.q, 1.0, out=dst.q)                          # exact in bf16
        outs.append(call(dst, None, ws))
    torch.cuda.synchronize()
    assert va.workspace_status(ws) == 0
    return outs, refs


class _Gqa:
    def __init__(self, splits=0):
        self.splits = splits

    def workspace_size(self, w):
        return va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, self.splits)

    def __call__(self, w, out, ws):
        return va.verify_attn_ex(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                                 w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale,
                                 w.k_descale, w.v_descale, out=out, workspace=ws,
                                 num_splits=self.splits)


class _Mla:
    @staticmethod
    def workspace_size(w):
        return va.mla_workspace_size(w.q, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k)

    def __call__(self, w, out, ws):
        return va.verify_attn_mla(w.q, w.kv_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                                  w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale,
                                  w.v_descale, out=out, workspace=ws)


# (KV dtype, forced split count): FP8 with 8 splits runs the kernel with Q in
# tensor memory (at least 16 key tiles per CTA), the others Q in shared memory
@pytest.mark.parametrize("dt,splits", [("fp8_e4m3", 0), ("bf16", 0), ("fp8_e4m3", 8)])
def test_back_to_back_gqa(dt, splits):
    fp8 = dt == "fp8_e4m3"
    a, b = _batches(lambda seed: make_workload(Q_LENS, KV_LENS, 16, 2, dt, seed=seed,
                                               k_descale=1.1 if fp8 else None,
                                               v_descale=0.8 if fp8 else None))
    if splits:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert va.plan(a.num_seqs, 2, 16, a.max_seqlen_q, a.max_seqlen_k, dt, sms, splits)["kernel"] == 2
    outs, refs = _run_alternating(a, b, ["q", "k_cache", "v_cache", "block_table", "seqused_k"],
                                  _Gqa(splits))
    assert not torch.equal(refs[0], refs[1])
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), refs[i % 2].view(torch.int16)), f"call {i}"


class _Variants(_Gqa):
    """verify_attn_opt with a window, a soft cap and sinks (the VAR main
    kernel and the SINKS merge)."""

    def __init__(self, hq):
        super().__init__()
        self.sinks = torch.linspace(-1.5, 1.5, hq, device="cuda")

    def __call__(self, w, out, ws):
        return va.verify_attn_opt(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                                  w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale,
                                  w.k_descale, w.v_descale, out=out, workspace=ws, window_left=700,
                                  softcap=20.0, sinks=self.sinks)


def test_back_to_back_variants():
    a, b = _batches(lambda seed: make_workload(Q_LENS, KV_LENS, 16, 2, "fp8_e4m3", seed=seed,
                                               k_descale=1.1, v_descale=0.8))
    outs, refs = _run_alternating(a, b, ["q", "k_cache", "v_cache", "block_table", "seqused_k"],
                                  _Variants(a.q.shape[1]))
    assert not torch.equal(refs[0], refs[1])
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), refs[i % 2].view(torch.int16)), f"call {i}"


def test_back_to_back_shards():
    """Two shards and their merge per call (verify_attn_partial twice, then
    verify_attn_merge_partials), calls unsynchronised, each shard with its
    own workspace reused across calls."""
    from speculative_decoding_verify_split_gb300.workloads import split_kv_shards
    a, b = _batches(lambda seed: make_workload(Q_LENS, KV_LENS, 16, 1, "fp8_e4m3", seed=seed))
    width = a.block_table.shape[1]
    plans = {id(x): split_kv_shards(x, 2, seed=3) for x in (a, b)}
    wss = []
    for bt, su, ext in plans[id(a)]:
        n = va.workspace_size(a.q, a.k_cache, su, a.max_seqlen_q, width * 16)
        wss.append(torch.zeros(n + 256, dtype=torch.uint8, device="cuda"))

    def call(w):
        parts = []
        for (bt, su, ext), ws in zip(plans[id(w)], wss):
            parts.append(va.verify_attn_partial(w.q, w.k_cache, w.v_cache, bt, w.cu_seqlens_q, su,
                                                w.max_seqlen_q, width * 16, w.softmax_scale,
                                                w.k_descale, w.v_descale, kv_extent=ext, workspace=ws))
        return va.merge_partials(parts)

    refs = []
    for w in (a, b):
        refs.append(call(w).clone())
        torch.cuda.synchronize()
    outs = [call(a if i % 2 == 0 else b) for i in range(6)]
    torch.cuda.synchronize()
    assert not torch.equal(refs[0], refs[1])
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), refs[i % 2].view(torch.int16)), f"call {i}"
    for ws in wss:
        assert va.workspace_status(ws) == 0


def test_back_to_back_latent():
    a, b = _batches(lambda seed: make_mla_workload(Q_LENS, KV_LENS, 16, seed=seed, k_descale=0.9,
                                                   v_descale=1.2))
    outs, refs = _run_alternating(a, b, ["q", "kv_cache", "block_table", "seqused_k"], _Mla())
    assert not torch.equal(refs[0], refs[1])
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), refs[i % 2].view(torch.int16)), f"call {i}"
