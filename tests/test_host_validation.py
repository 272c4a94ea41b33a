"""Host-only checks of the boundary: the validation matrix (each shape gate
of the pages turned into a status code) and the split heuristic. No CUDA
call is made: verify_attn_check and verify_attn_plan are pure host code."""
import pytest
import torch

import speculative_decoding_verify_split_gb300 as va
from speculative_decoding_verify_split_gb300.build import build_library
from speculative_decoding_verify_split_gb300.workloads import make_workload

OK, NULL, SHAPE, DTYPE, UNSUP, WS, CUDA, LAYOUT = range(8)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_library()


def _args(w, **over):
    a = dict(q=w.q, k_cache=w.k_cache, v_cache=w.v_cache, block_table=w.block_table,
             cu_seqlens_q=w.cu_seqlens_q, seqused_k=w.seqused_k, max_seqlen_q=w.max_seqlen_q,
             max_seqlen_k=w.max_seqlen_k, k_descale=w.k_descale, v_descale=w.v_descale,
             out=torch.empty_like(w.q))
    a.update(over)
    return a


@pytest.fixture(scope="module")
def w():
    return make_workload([4, 2], [100, 37], 16, 1, "fp8_e4m3", seed=1, k_descale=1.0, v_descale=2.0)


def test_valid(w):
    assert va.check(**_args(w)) == OK


def test_valid_bf16_and_gqa():
    w2 = make_workload([2, 3], [50, 70], 32, 2, "bf16", seed=2)
    assert va.check(**_args(w2)) == OK


def test_null_descriptor(w):
    assert va.check(**_args(w, q=None)) == NULL
    assert va.check(**_args(w, out=None)) == NULL
    assert va.check(**_args(w, block_table=None)) == NULL


def test_dtypes(w):
    assert va.check(**_args(w, q=w.q.view(torch.int16).to(torch.int32))) == DTYPE
    assert va.check(**_args(w, v_cache=w.v_cache.to(torch.bfloat16))) == DTYPE
    assert va.check(**_args(w, block_table=w.block_table.float())) == DTYPE
    assert va.check(**_args(w, k_descale=torch.ones(1, dtype=torch.int32))) == DTYPE


def test_head_dim_and_page_size_are_gated(w):
    k = w.k_cache[..., :128].contiguous()
    assert va.check(**_args(w, k_cache=k, v_cache=k)) == UNSUP
    k8 = w.k_cache.reshape(-1, 8, 1, 256)
    assert va.check(**_args(w, k_cache=k8, v_cache=k8)) == UNSUP
    q = w.q[..., :128].contiguous()
    assert va.check(**_args(w, q=q, out=torch.empty_like(q))) == UNSUP


def test_head_ratio(w):
    q = torch.zeros(w.q.shape[0], 12, 256, dtype=torch.bfloat16)
    k = torch.zeros(4, 16, 8, 256, dtype=torch.float8_e4m3fn)
    assert va.check(**_args(w, q=q, out=torch.empty_like(q), k_cache=k, v_cache=k)) == SHAPE


def test_row_budget(w):
    assert va.check(**_args(w, max_seqlen_q=5)) == UNSUP      # 16 * 5 > 64
    assert va.check(**_args(w, max_seqlen_q=0)) == UNSUP
    assert va.check(**_args(w, max_seqlen_k=-1)) == UNSUP


def test_shapes(w):
    assert va.check(**_args(w, cu_seqlens_q=w.cu_seqlens_q[:2])) == SHAPE
    assert va.check(**_args(w, block_table=w.block_table[:1])) == SHAPE
    assert va.check(**_args(w, max_seqlen_k=w.block_table.shape[1] * 16 + 1)) == SHAPE
    assert va.check(**_args(w, out=torch.empty(w.q.shape[0], 8, 256, dtype=torch.bfloat16))) == SHAPE
    assert va.check(**_args(w, v_descale=torch.ones(2))) == SHAPE


def test_layout(w):
    big = torch.zeros(w.q.shape[0], w.q.shape[1], 512, dtype=torch.bfloat16)
    q_strided = big[..., ::2]
    assert va.check(**_args(w, q=q_strided, out=torch.empty_like(w.q))) == LAYOUT
    q_padded = big[..., :256]                       # head stride 512: still 16-byte rows
    assert va.check(**_args(w, q=q_padded, out=torch.empty_like(w.q))) == OK
    odd = torch.zeros(w.q.numel() + 1, dtype=torch.bfloat16)[1:].view(w.q.shape)
    assert va.check(**_args(w, q=odd, out=torch.empty_like(w.q))) == LAYOUT


def test_plan_fills_the_sms():
    p = va.plan(16, 1, 16, 4, 131072, "fp8_e4m3", 152)
    assert p["num_splits"] == 152 and p["max_rows"] == 64 and p["num_work"] == 16
    assert p["workspace_bytes"] >= (16 + 152) * 64 * 256 * 4


def test_plan_spreads_small_batches_one_tile_per_cta():
    # one CTA per key tile of the upper-bound workload, up to one per SM
    p = va.plan(1, 1, 16, 2, 16, "fp8_e4m3", 152)
    assert p["num_splits"] == 1
    for dt in ("fp8_e4m3", "bf16"):
        p = va.plan(2, 1, 16, 4, 1024, dt, 152)
        assert p["num_splits"] == 2 * (1024 // p["tile_keys"])
        p = va.plan(8, 2, 32, 4, 4096, dt, 152)
        assert p["num_splits"] == 152


def test_plan_force_and_clamp():
    assert va.plan(2, 1, 16, 4, 1024, "fp8_e4m3", 152, force_splits=7)["num_splits"] == 7
    for dt in ("fp8_e4m3", "bf16"):
        p = va.plan(2, 1, 16, 4, 1024, dt, 152, force_splits=10**6)
        assert p["num_splits"] == 2 * (1024 // p["tile_keys"])
    assert va.plan(3, 1, 16, 4, 0, "fp8_e4m3", 152)["num_splits"] == 1


def test_plan_picks_the_layout():
    """FP8 batches of at least 16 key tiles per CTA run the kernel with Q and
    P in tensor memory (plan kernel 2); BF16 and small FP8 batches the one
    with Q in shared memory (1)."""
    assert va.plan(16, 1, 16, 4, 131072, "fp8_e4m3", 152)["kernel"] == 2
    assert va.plan(64, 1, 16, 3, 32768, "fp8_e4m3", 152)["kernel"] == 2
    assert va.plan(2, 1, 16, 4, 1024, "fp8_e4m3", 152)["kernel"] == 1
    assert va.plan(8, 2, 32, 4, 4096, "fp8_e4m3", 152)["kernel"] == 1
    assert va.plan(16, 1, 16, 4, 131072, "bf16", 152)["kernel"] == 1
    # the boundary: 16 tiles per CTA
    assert va.plan(1, 1, 16, 4, 16 * 128, "fp8_e4m3", 152, force_splits=1)["kernel"] == 2
    assert va.plan(1, 1, 16, 4, 16 * 128 - 128, "fp8_e4m3", 152, force_splits=1)["kernel"] == 1
    assert va.plan(2, 1, 16, 4, 1024, "fp8_e4m3", 152, force_splits=1)["kernel"] == 2


def test_plan_rejects():
    for bad in [(1, 1, 16, 5, 100, "fp8_e4m3", 152), (1, 3, 16, 1, 100, "fp8_e4m3", 152),
                (1, 1, 16, 1, 100, "fp8_e4m3", 0), (1, 1, 16, 0, 100, "bf16", 152)]:
        with pytest.raises(va.VerifyAttnError):
            va.plan(*bad)


def _bt_call(indptr, indices, table, seqused):
    import ctypes
    d = [va.desc(t) for t in (indptr, indices, table, seqused)]
    return va.library().verify_attn_block_table_from_indptr(
        *[None if x is None else ctypes.byref(x) for x in d], 0, None, None)


def test_block_table_builder_rejects_bad_descriptors_before_launch():
    # host validation only: every case returns before anything is launched
    i32 = torch.int32
    ip, ix = torch.zeros(4, dtype=i32), torch.zeros(10, dtype=i32)
    bt, sk = torch.zeros(3, 5, dtype=i32), torch.zeros(3, dtype=i32)
    assert _bt_call(ip, ix, bt, None) == 1                                   # NULL
    assert _bt_call(ip.float(), ix, bt, sk) == 3                             # dtype
    assert _bt_call(ip, ix, torch.zeros(2, 5, dtype=i32), sk) == 2           # B mismatch
    assert _bt_call(ip, ix, bt, torch.zeros(4, dtype=i32)) == 2
    assert _bt_call(ip, ix, bt.view(-1), sk) == 2                            # table not 2D
    assert _bt_call(torch.zeros(8, dtype=i32)[::2], ix, bt, sk) == 7         # strided indptr
    assert _bt_call(ip, torch.zeros(20, dtype=i32)[::2], bt, sk) == 7        # strided indices
    big = torch.zeros(65537, dtype=i32)
    assert _bt_call(big, ix, torch.zeros(65536, 1, dtype=i32), torch.zeros(65536, dtype=i32)) == 4


# ---- the latent-cache entry point (validation runs before any CUDA call) ----

def _mla_status(w, **over):
    """verify_attn_mla's status for invalid arguments: returned by the host
    checks before the library touches CUDA."""
    import ctypes
    a = dict(q=w.q, kv=w.kv_cache, bt=w.block_table, cu=w.cu_seqlens_q, su=w.seqused_k,
             mq=w.max_seqlen_q, mk=w.max_seqlen_k, kd=w.k_descale, vd=w.v_descale,
             out=torch.empty(w.q.shape[0], w.q.shape[1], 512, dtype=torch.bfloat16))
    a.update(over)
    ds = [va.desc(a[k]) for k in ("q", "kv", "bt", "cu", "su", "kd", "vd", "out")]
    r = [None if d is None else ctypes.byref(d) for d in ds]
    return va.library().verify_attn_mla(r[0], r[1], r[2], r[3], r[4], int(a["mq"]), int(a["mk"]),
                                        0.1, r[5], r[6], r[7], None, 0, 0, None, None)


@pytest.fixture(scope="module")
def wm():
    from speculative_decoding_verify_split_gb300.workloads import make_mla_workload
    return make_mla_workload([4, 2], [100, 37], 16, seed=1, k_descale=1.0, v_descale=2.0)


def test_mla_validation(wm):
    assert _mla_status(wm, q=None) == NULL
    assert _mla_status(wm, out=None) == NULL
    # a BF16 latent cache passes the cache checks (then the mismatched out is reported)
    assert _mla_status(wm, kv=wm.kv_cache.to(torch.bfloat16),
                       out=torch.empty(6, 8, 512, dtype=torch.bfloat16)) == SHAPE
    assert _mla_status(wm, kv=wm.kv_cache.to(torch.float32)) == DTYPE
    assert _mla_status(wm, kv=wm.kv_cache.view(torch.uint8).to(torch.int32)) == DTYPE
    two = torch.cat([wm.kv_cache, wm.kv_cache], dim=2)
    assert _mla_status(wm, kv=two) == UNSUP                                # one latent head
    assert _mla_status(wm, kv=wm.kv_cache[..., :512].contiguous()) == UNSUP
    assert _mla_status(wm, q=wm.q[..., :512].contiguous()) == UNSUP
    assert _mla_status(wm, out=torch.empty(6, 16, 576, dtype=torch.bfloat16)) == UNSUP
    assert _mla_status(wm, out=torch.empty(6, 8, 512, dtype=torch.bfloat16)) == SHAPE
    assert _mla_status(wm, mq=5) == UNSUP                                  # 16 heads x 5 > 64 rows
    assert _mla_status(wm, mk=100000) == SHAPE                             # table too narrow
    assert _mla_status(wm, kd=torch.ones(2)) == SHAPE
    shifted = torch.empty(wm.q.numel() + 1, dtype=torch.bfloat16)[1:].view(wm.q.shape)
    assert _mla_status(wm, q=shifted) == LAYOUT                            # not 16-byte aligned
    assert _mla_status(wm, cu=wm.cu_seqlens_q[:2]) == SHAPE
