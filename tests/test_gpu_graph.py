"""verify_attn_ex inside a CUDA graph.

The call with a caller workspace allocates nothing, synchronises nothing and
reads no device data on the host, so a serving loop can capture it once per
batch shape and replay it. Captured through the C-ABI (both kernels, the merge
as a programmatic dependent of the main kernel), replayed on new Q values and
descales written into the same buffers, and compared bit for bit with an eager
call on those values."""
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


def _ex(w, out, ws, stream=None, splits=0):
    return va.verify_attn_ex(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                             w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale,
                             w.k_descale, w.v_descale, out=out, workspace=ws, num_splits=splits,
                             stream=stream)


# (KV dtype, forced split count): FP8 with 4 splits runs the kernel with Q in
# tensor memory (at least 16 key tiles per CTA), the others Q in shared memory
@pytest.mark.parametrize("dt,splits", [("fp8_e4m3", 0), ("bf16", 0), ("fp8_e4m3", 4)])
def test_graph_replay_matches_eager(dt, splits):
    w = make_workload([4, 2, 3, 1], [3000, 769, 1500, 40], 16, 1, dt, seed=31,
                      k_descale=1.1 if dt == "fp8_e4m3" else None,
                      v_descale=0.8 if dt == "fp8_e4m3" else None).to("cuda")
    if splits:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert va.plan(w.num_seqs, 1, 16, w.max_seqlen_q, w.max_seqlen_k, dt, sms, splits)["kernel"] == 2
    n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k, splits)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device="cuda")
    out = torch.full_like(w.q, float("nan"))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _ex(w, out, ws, stream=side, splits=splits)   # warm-up: library state, kernel attributes
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _ex(w, out, ws, stream=torch.cuda.current_stream(), splits=splits)

    # new values in the same buffers: another Q and, for fp8, other descales
    w.q.copy_(torch.randn(w.q.shape, generator=torch.Generator(device="cuda").manual_seed(5),
                          device="cuda").to(w.q.dtype))
    if dt == "fp8_e4m3":
        w.k_descale.fill_(1.3)
        w.v_descale.fill_(0.6)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()

    ref = torch.full_like(w.q, float("nan"))
    _ex(w, ref, ws, splits=splits)
    torch.cuda.synchronize()
    assert not torch.isnan(got.float()).any()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert va.workspace_status(ws) == 0
