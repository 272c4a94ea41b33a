"""Decode-context-parallel verify attention (speculative_decoding_verify_split_gb300.dcp):
every sequence's keys split over the ranks of a process group, each rank's
shard result exchanged by an all-gather and merged by log-sum-exp.

* CPU (gloo, two ranks): the exchange alone. Each rank's shard result comes
  from the shard oracle; the gathered parts must be every rank's own result
  in rank order, and their merge (the oracle's) the full verify attention.
* GPU (gloo, two processes on one GPU, whose kernels never wait on each
  other): the whole path, verify_attn_partial on each rank's shard, the
  exchange staged through host memory, verify_attn_merge_partials; both
  ranks' bf16 outputs must be bit-identical and match the full oracle
  element by element within the parity tolerance."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    dict(q=[4, 2, 3, 1], kv=[3000, 769, 1500, 20], hq=16, hkv=1, dt="fp8_e4m3", kd=1.2, vd=0.7),
    dict(q=[2, 2, 2], kv=[2000, 4100, 64], hq=8, hkv=1, dt="bf16", kd=None, vd=None),
    dict(q=[3, 4], kv=[1100, 2600], hq=32, hkv=2, dt="fp8_e4m3", kd=None, vd=None),
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload(ci):
    from speculative_decoding_verify_split_gb300.workloads import make_workload
    c = CASES[ci]
    return make_workload(c["q"], c["kv"], c["hq"], c["hkv"], c["dt"], seed=700 + ci,
                         k_descale=c["kd"], v_descale=c["vd"])


def _shard_view(w, bt, su):
    s = w.to("cpu")
    s.block_table, s.seqused_k = bt.cpu(), su.cpu()
    return s


def _cpu_rank(rank, world, port, ci, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle.partial_fp64 import merge_partials, partial_oracle_from_torch
    from speculative_decoding_verify_split_gb300.dcp import gather_shard_results
    from speculative_decoding_verify_split_gb300.workloads import split_kv_shards
    w = _workload(ci)
    bt, su, ext = split_kv_shards(w, world, seed=ci)[rank]
    o, lse = partial_oracle_from_torch(_shard_view(w, bt, su), ext)
    o_t = torch.from_numpy(o).to(torch.float32)
    l_t = torch.from_numpy(lse).to(torch.float32)
    parts = gather_shard_results(o_t, l_t)
    own = torch.equal(parts[rank][0], o_t) and torch.equal(parts[rank][1], l_t)
    merged = merge_partials([p.double().numpy() for p, _ in parts],
                            [l.double().numpy() for _, l in parts])
    q.put((rank, own, merged))
    dist.barrier()
    dist.destroy_process_group()


def _run(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port) + args + (q,)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return sorted(res, key=lambda r: r[0])


@pytest.mark.parametrize("ci", [0, 1])
def test_exchange_gloo_cpu(ci):
    from oracle.attention_fp64 import oracle_from_torch
    res = _run(_cpu_rank, 2, ci)
    assert all(r[1] for r in res), "a rank's own part is not in its rank's place"
    ref = oracle_from_torch(_workload(ci))
    for _, _, merged in res:
        assert np.abs(merged - ref).max() < 1e-6   # fp32 shard results, fp64 merge


def _gpu_rank(rank, world, port, ci, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    from speculative_decoding_verify_split_gb300.dcp import dcp_verify_attn
    from speculative_decoding_verify_split_gb300.workloads import split_kv_shards
    w = _workload(ci).to("cuda")
    bt, su, ext = split_kv_shards(w, world, seed=ci)[rank]
    out = dcp_verify_attn(w.q, w.k_cache, w.v_cache, bt, w.cu_seqlens_q, su, ext, w.max_seqlen_q,
                          bt.shape[1] * 16, w.softmax_scale, w.k_descale, w.v_descale)
    torch.cuda.synchronize()
    # by value (the bf16 bits as a numpy array): a torch tensor would go
    # through a file descriptor this process shares, gone if it exits first
    q.put((rank, out.cpu().view(torch.int16).numpy().copy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_dcp_two_processes_on_one_gpu(ci):
    from gpu_util import compare
    from oracle.attention_fp64 import oracle_from_torch
    res = _run(_gpu_rank, 2, ci)
    a, b = (torch.from_numpy(r[1]).view(torch.bfloat16) for r in res)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "ranks disagree"
    print("dcp", ci, compare(a, oracle_from_torch(_workload(ci))))
