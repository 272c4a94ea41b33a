#!/usr/bin/env python
"""Benchmark of target-verify attention (split-KV main kernel + segment merge).

One step = one verify_attn call over the whole batch of the long-context FP8
verify workload (16 sequences, 4 draft tokens, kv_len U[65536, 131072],
16 query heads per KV head, head_dim 256, page 16, FP8 E4M3 KV), inputs
resident in HBM. The inputs (~0.8 GB) exceed the 129 MB L2, so no flush is
needed between steps.

Prints one JSON line. ``value`` = algorithmic bytes (K+V read once per KV
head, plus Q and out) of all ranks / max-over-ranks time, in GB/s.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
Multi-GPU runs are independent replicas (the operation has no exchange step).
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-attn µs/call and achieved HBM GB/s (fraction of ~8 TB/s) on 1 GB300"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# main kernel by KV dtype and, for the GQA kernel, the layout the plan picks
# (verify_attn_plan's `kernel`: 2 = FP8 with Q in tensor memory)
MAIN_KERNEL = {("fp8_e4m3", 1): "va_main_tc_kernel<true, false, false>",
               ("fp8_e4m3", 2): "va_main_tc_kernel<true, false, true>",
               ("bf16", 1): "va_main_tc_kernel<false, false, false>",
               "mla": "va_mla_tc_kernel", "mla_bf16": "va_mla_bf16_tc_kernel"}


def is_mla(name):
    """Workloads over an absorbed-MLA latent cache (verify_attn_mla)."""
    return name.startswith("mla_")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context_fp8")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def env_int(name, default):
    v = os.environ.get(name)
    return int(v) if v is not None else default


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments and whitespace runs (string and
    character literals kept as they are), so that a change of wording alone
    does not count as a change of the kernels."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_sha():
    """A hash of the CUDA/C++ sources' code (comments and whitespace removed):
    DRAM traffic recorded by ncu is reported only for the code it was taken
    on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verify_split_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*"))):
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(strip_c_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per main-kernel launch from a committed ncu summary, only if
    it was taken on the kernel sources as they are now."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            recs = json.load(f)
    except Exception:
        return None
    sha = kernel_source_sha()
    for r in recs:
        if r.get("workload") == workload and r.get("kernel_source_sha") == sha:
            return r.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_id), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def gpu_identifier(torch, dev):
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return dev


L2_BYTES = 129 * 2**20
FLUSH_BYTES = 256 * 2**20


def needs_flush(w):
    """Inputs that could stay L2-resident between steps get an L2 flush."""
    return w.algorithmic_bytes() < 2 * L2_BYTES


def max_over_ranks(x: float, world: int, dist, device) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself on
    one rank. A collective of the timing only: the ranks' work is
    independent (replicas)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(alg_bytes: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank's algorithmic bytes over the slowest step time."""
    return alg_bytes * world / (ms_per_step / 1e3) / 1e9


def config_block(name, q_lens, kv_lens, hq, hkv, kv_dtype, alg_bytes, world):
    """The JSON line's config: the workload by name, its seeded lengths and
    sizes. Both arms print it (the reference arm from the same seeded
    structure, without drawing the cache)."""
    layout = ({"layout": "absorbed-MLA latent cache, rows [latent 512 | rope 64], values = latent",
               "row_width": 576, "value_dim": 512} if is_mla(name) else {"head_dim": 256})
    return {"workload": name, "num_seqs": len(q_lens), "q_lens": sorted(set(q_lens)),
            "kv_len_range": [min(kv_lens), max(kv_lens)], "kv_tokens": sum(kv_lens),
            "num_q_heads": hq, "num_kv_heads": hkv, **layout,
            "page_size": 16, "kv_dtype": kv_dtype, "algorithmic_bytes": alg_bytes,
            "l2": ("inputs under 2x the 129 MB L2: a 256 MB buffer is written before every step, "
                   "outside the per-step CUDA events" if alg_bytes < 2 * L2_BYTES else
                   "inputs exceed the 129 MB L2; steps back to back, no flush"),
            "accumulate": "f32",
            "parallelism": f"replicas x{world}", "seed": 0}


def workload_config(w, name, world):
    return config_block(name, w.q_lens, w.kv_lens, w.num_q_heads, w.num_kv_heads, w.kv_dtype,
                        w.algorithmic_bytes(), world)


def reference_structure(name):
    """The seeded structure of a workload (lengths, heads, cache type) and its
    algorithmic bytes as Workload / MlaWorkload count them, without drawing
    any values."""
    from speculative_decoding_verify_split_gb300.workloads import mla_workload_structure, workload_structure
    mla = is_mla(name)
    if mla:
        st = dict(mla_workload_structure(name, 0), Hkv=1)
        st.setdefault("kv_dtype", "fp8_e4m3")
    else:
        st = workload_structure(name, 0)
    e = 1 if st["kv_dtype"] == "fp8_e4m3" else 2
    key_bytes = 576 * e if mla else st["Hkv"] * 512 * e  # cache bytes per key
    q_bytes = st["Hq"] * ((576 + 512) * 2 if mla else 2 * 256 * 2)  # per draft token: Q in, out
    alg = sum(st["kv_lens"]) * key_bytes + sum(st["q_lens"]) * q_bytes
    return st, key_bytes, alg


def reference_config(name, world):
    st, _, alg = reference_structure(name)
    return config_block(name, st["q_lens"], st["kv_lens"], st["Hq"], st["Hkv"], st["kv_dtype"], alg, world)


def seq_bytes(w, b, mla):
    """Algorithmic bytes of sequence b of a workload (its share of
    Workload.algorithmic_bytes / MlaWorkload.algorithmic_bytes)."""
    e = 1 if w.kv_dtype == "fp8_e4m3" else 2
    if mla:
        return w.kv_lens[b] * 576 * e + w.q_lens[b] * w.num_q_heads * (576 + 512) * 2
    return w.kv_lens[b] * w.num_kv_heads * 256 * 2 * e + 2 * w.q_lens[b] * w.num_q_heads * 256 * 2


def cpu_baseline(w_cpu, seconds, mla=False):
    """The fp64 oracle as it stands, on sequences of the workload in order,
    until `seconds` of wall time have passed (at least one sequence)."""
    if mla:
        from oracle.mla_fp64 import mla_oracle_from_torch as run_oracle
    else:
        from oracle.attention_fp64 import oracle_from_torch as run_oracle
    done, nbytes = [], 0
    t0 = time.perf_counter()
    c0 = time.process_time()
    for b in range(w_cpu.num_seqs):
        run_oracle(w_cpu, [b])
        done.append(b)
        nbytes += seq_bytes(w_cpu, b, mla)
        if time.perf_counter() - t0 >= seconds:
            break
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    return {"value": nbytes / wall / 1e9, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "cpu_time_over_wall": round(cpu / wall, 2),
            "sample": f"{len(done)} of {w_cpu.num_seqs} sequences ({sum(w_cpu.kv_lens[b] for b in done)} "
                      f"keys), fp64 numpy, {wall:.1f} s wall"}


def replay_us(torch, fn, reps, K, scratch=None, warm=None):
    """Device time per call of fn, from CUDA-graph replays (host marshalling is
    not in the figure). fn is captured `reps` times into one graph after three
    warm-up calls (of `warm`, default fn) on a side stream. Without `scratch`
    the graph is replayed back to back; with it (for work whose bytes fit in
    L2) fn is captured once and every replay is timed alone with CUDA events
    after `scratch` is written, outside the events, so each call starts with a
    cold L2."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            (warm or fn)()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    reps = 1 if scratch is not None else reps
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    if scratch is not None:
        n = max(K, 5)
        s0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        s1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            scratch.fill_(i & 0xFF)
            s0[i].record()
            g.replay()
            s1[i].record()
        torch.cuda.synchronize()
        return statistics.mean(s0[i].elapsed_time(s1[i]) for i in range(n)) * 1e3
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_rep = max(K // reps, 5)
    a.record()
    for _ in range(n_rep):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (n_rep * reps) * 1e3


def l2_scratch(torch, nbytes, device):
    """A buffer to write between timed calls when `nbytes` (what a call
    reads) could stay in L2 from one call to the next; None otherwise."""
    if nbytes < 2 * L2_BYTES:
        return torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    return None


def draft_extend_timing(va, w, stream, torch, K):
    """The draft-extend pass on the same workload, given in flat token-slot
    form: the block-table builder alone, and builder + attention per call.
    Measured after the timed region from CUDA-graph replays, so host-side
    marshalling is not part of the figure."""
    from speculative_decoding_verify_split_gb300.workloads import flat_kv_slots
    ip, ix = flat_kv_slots(w)
    width = w.block_table.shape[1]
    B = w.num_seqs
    bt = torch.empty((B, width), dtype=torch.int32, device=ip.device)
    sk = torch.empty((B,), dtype=torch.int32, device=ip.device)
    out = torch.empty_like(w.q)

    # device time: each measured sequence is captured once in a CUDA graph
    # (both entry points are capturable with caller buffers) and replayed
    n_ws = va.workspace_size(w.q, w.k_cache, sk, w.max_seqlen_q, width * 16)
    ws = torch.zeros(n_ws + 256, dtype=torch.uint8, device=ip.device)

    def call_ex():
        build_cur()
        va.verify_attn_ex(w.q, w.k_cache, w.v_cache, bt, w.cu_seqlens_q, sk, w.max_seqlen_q,
                          width * 16, w.softmax_scale, w.k_descale, w.v_descale, out=out,
                          workspace=ws, stream=torch.cuda.current_stream())

    def build_cur():
        va.block_table_from_indptr(ip, ix, width, 0, block_table=bt, seqused_k=sk,
                                   stream=torch.cuda.current_stream())

    nnz = ix.numel()
    builder_bytes = 4 * nnz + 4 * (B + 1) + 4 * B * width + 4 * B
    res = {"builder": replay_us(torch, build_cur, 20, K, l2_scratch(torch, builder_bytes, ip.device)),
           "call": replay_us(torch, call_ex, 4, K, l2_scratch(torch, w.algorithmic_bytes(), ip.device))}
    return {"builder_us": round(res["builder"], 2), "builder_bytes": builder_bytes,
            "builder_gbs": round(builder_bytes / res["builder"] / 1e3, 1),
            "call_us": round(res["call"], 2), "kv_tokens": nnz,
            "note": "block table + seqused_k from kv_indptr/kv_indices, then verify_attn_ex with "
                    "max_seqlen_k = width * 16; device time from CUDA-graph replays "
                    "(20 builder launches, or 4 builder+attention calls, per graph; a call "
                    "whose bytes fit in L2 is replayed alone after an L2 flush)"}


def shard_timing(va, w, torch, K):
    """The same workload with each sequence's keys cut into two page-aligned
    shards (verify_attn_partial twice, then verify_attn_merge_partials), from
    CUDA-graph replays so that host marshalling is not in the figure. Also the
    shard merge alone."""
    from speculative_decoding_verify_split_gb300.workloads import split_kv_shards
    shards = split_kv_shards(w, 2, seed=0)
    width = w.block_table.shape[1]
    o = [torch.empty(w.q.shape, dtype=torch.float32, device=w.q.device) for _ in shards]
    lse = [torch.empty(w.q.shape[:2], dtype=torch.float32, device=w.q.device) for _ in shards]
    out = torch.empty_like(w.q)
    wss = []
    for bt, su, ext in shards:
        n = va.workspace_size(w.q, w.k_cache, su, w.max_seqlen_q, width * 16)
        wss.append(torch.zeros(n + 256, dtype=torch.uint8, device=w.q.device))

    def partials():
        for i, (bt, su, ext) in enumerate(shards):
            va.verify_attn_partial(w.q, w.k_cache, w.v_cache, bt, w.cu_seqlens_q, su, w.max_seqlen_q,
                                   width * 16, w.softmax_scale, w.k_descale, w.v_descale, kv_extent=ext,
                                   o=o[i], lse=lse[i], workspace=wss[i],
                                   stream=torch.cuda.current_stream())

    def merge():
        va.merge_partials(list(zip(o, lse)), out=out, stream=torch.cuda.current_stream())

    def both():
        partials()
        merge()

    merge_bytes = 2 * (w.q.numel() * 4 + w.q.shape[0] * w.q.shape[1] * 4) + w.q.numel() * 2
    res = {"two_shards_and_merge": replay_us(torch, both, 2, K,
                                             l2_scratch(torch, w.algorithmic_bytes(), w.q.device)),
           "merge": replay_us(torch, merge, 20, K, l2_scratch(torch, merge_bytes, w.q.device),
                              warm=both)}
    return {"two_shards_and_merge_us": round(res["two_shards_and_merge"], 2),
            "shard_merge_us": round(res["merge"], 2), "shard_merge_bytes": merge_bytes,
            "note": "each sequence's keys cut into two page-aligned shards (verify_attn_partial on each, "
                    "then verify_attn_merge_partials); device time from CUDA-graph replays; a call "
                    "whose bytes fit in L2 is replayed alone after an L2 flush"}


def window_bytes(w, window_left):
    """Bytes a call with a sliding window of `window_left` keys reads at
    most: each sequence's last window_left + q_len keys (all keys when
    shorter) for every KV head, plus Q and the output."""
    e = 1 if w.kv_dtype == "fp8_e4m3" else 2
    kv = sum(min(s, window_left + l) for s, l in zip(w.kv_lens, w.q_lens))
    return kv * w.num_kv_heads * 256 * 2 * e + 2 * sum(w.q_lens) * w.num_q_heads * 256 * 2


def variant_timing(va, w, torch, K):
    """The generic attention's variants on the same workload (verify_attn_opt
    with a caller workspace): no option, a 4096-key sliding window, a logit
    soft cap of 30, per-head sinks, and all three, from CUDA-graph replays.
    A call whose bytes fit in L2 (the window on most workloads) is timed
    alone after an L2 flush."""
    hq = w.q.shape[1]
    sinks = torch.linspace(-2.0, 2.0, hq, device=w.q.device)
    out = torch.empty_like(w.q)
    cases = {"plain": {}, "window_4096": dict(window_left=4096), "softcap_30": dict(softcap=30.0),
             "sinks": dict(sinks=sinks), "all_three": dict(window_left=4096, softcap=30.0, sinks=sinks)}
    res = {}
    for name, kw in cases.items():
        n = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k)
        ws = torch.zeros(n + 256, dtype=torch.uint8, device=w.q.device)

        def call():
            va.verify_attn_opt(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k,
                               w.max_seqlen_q, w.max_seqlen_k, w.softmax_scale, w.k_descale,
                               w.v_descale, out=out, workspace=ws, stream=torch.cuda.current_stream(),
                               **kw)
        nbytes = window_bytes(w, kw["window_left"]) if "window_left" in kw else w.algorithmic_bytes()
        scratch = l2_scratch(torch, nbytes, w.q.device)
        res[name + "_us"] = round(replay_us(torch, call, 4, K, scratch), 2)
        res[name + "_l2_flushed"] = scratch is not None
        del scratch
    res["note"] = ("verify_attn_opt per call (main kernel with the variant code + merge), device time "
                   "from CUDA-graph replays; the window reads only the keys it sees; *_l2_flushed: "
                   "replayed one call at a time after an L2 flush, since its bytes fit in L2")
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = env_int("RANK", 0), env_int("WORLD_SIZE", 1), env_int("LOCAL_RANK", 0)
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        from speculative_decoding_verify_split_gb300.build import build_library
        build_library()
    if world > 1:
        dist.barrier()
    import speculative_decoding_verify_split_gb300 as va
    from speculative_decoding_verify_split_gb300.workloads import named_mla_workload, named_workload

    mla = is_mla(args.workload)
    stream = torch.cuda.current_stream(dev)
    if mla:
        w = named_mla_workload(args.workload, seed=0, value_device=str(dev)).to(dev)
        out = torch.empty(w.q.shape[0], w.q.shape[1], va.MLA_NOPE, dtype=torch.bfloat16, device=dev)
        n_ws = va.mla_workspace_size(w.q, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k)
        inputs = ("q", "kv_cache", "block_table", "cu_seqlens_q", "seqused_k")
        kernel = MAIN_KERNEL["mla" if w.kv_dtype == "fp8_e4m3" else "mla_bf16"]
    else:
        w = named_workload(args.workload, seed=0, value_device=str(dev)).to(dev)
        out = torch.empty_like(w.q)
        n_ws = va.workspace_size(w.q, w.k_cache, w.seqused_k, w.max_seqlen_q, w.max_seqlen_k)
        inputs = ("q", "k_cache", "v_cache", "block_table", "cu_seqlens_q", "seqused_k")
        layout = va.plan(w.num_seqs, w.k_cache.shape[2], w.q.shape[1], w.max_seqlen_q, w.max_seqlen_k,
                         w.kv_dtype, torch.cuda.get_device_properties(dev).multi_processor_count)["kernel"]
        kernel = MAIN_KERNEL[(w.kv_dtype, layout)]
    alg = w.algorithmic_bytes()
    ws = torch.zeros(n_ws + 256, dtype=torch.uint8, device=dev)

    def step(ev_mid=None):
        if mla:
            va.run_mla_workload(w, out=out, workspace=ws, stream=stream, event_after_main=ev_mid)
        else:
            va.run_workload_ex(w, out=out, workspace=ws, stream=stream, event_after_main=ev_mid)

    def public_call():
        # the plain entry points, library-owned workspace
        if mla:
            va.run_mla_workload(w, out=out, stream=stream)
        else:
            va.run_workload(w, out=out, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_identifier(torch, local))
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    flush = needs_flush(w)
    scratch = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    ev_a = torch.cuda.Event(enable_timing=True)
    ev_b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if flush:
        # each step alone, after an L2 flush that stays outside its events
        s0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        s1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ev_a.record(stream)
        for i in range(K):
            scratch.fill_(i & 0xFF)
            s0[i].record(stream)
            step()
            s1[i].record(stream)
        ev_b.record(stream)
        torch.cuda.synchronize()
        total_ms = sum(s0[i].elapsed_time(s1[i]) for i in range(K))
    else:
        # whole steps back to back: main kernel + merge, nothing between them
        ev_a.record(stream)
        for i in range(K):
            step()
        ev_b.record(stream)
        torch.cuda.synchronize()
        total_ms = ev_a.elapsed_time(ev_b)
    if world > 1:
        dist.barrier()
    # the main kernel alone: an event recorded on the launching stream right
    # after it (this also keeps the merge from overlapping its launch, so it is
    # a separate loop)
    Km = min(K, 300)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(Km)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(Km)]
    for i in range(Km):
        if flush:
            scratch.fill_(i & 0xFF)
        e0[i].record(stream)
        step(e1[i])
    torch.cuda.synchronize()
    main_ms = statistics.mean(e0[i].elapsed_time(e1[i]) for i in range(Km))
    # keep the GPU busy a little longer so the clock sampler sees the load
    t_end = time.time() + 1.0
    while time.time() < t_end:
        for _ in range(20):
            step()
        torch.cuda.synchronize()
    clocks = sampler.stop()

    total_ms = max_over_ranks(total_ms, world, dist if world > 1 else None, dev)
    ms_per_step = total_ms / K
    value = throughput(alg, world, ms_per_step)

    # End to end through the public API with host buffers: every step copies
    # all inputs from pinned host memory and reads the output back.
    host = {k: getattr(w, k).cpu().pin_memory() for k in inputs}
    for k in ("k_descale", "v_descale"):
        if getattr(w, k) is not None:
            host[k] = getattr(w, k).cpu().pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        for k, t in host.items():
            getattr(w, k).copy_(t, non_blocking=True)
        public_call()
        out_host.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    E = max(args.e2e_steps, 3)
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    ea.record(stream)
    for _ in range(E):
        e2e_step()
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / E
    e2e_ms = max_over_ranks(e2e_ms, world, dist if world > 1 else None, dev)

    draft = None if mla else draft_extend_timing(va, w, stream, torch, min(K, 200))
    shards = None if mla else shard_timing(va, w, torch, min(K, 200))
    variants = None if mla else variant_timing(va, w, torch, min(K, 200))

    peak, peak_src = peak_hbm()
    achieved = alg / (main_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3" if w.kv_dtype == "fp8_e4m3" else "bf16", "data": "synthetic",
        "config": workload_config(w, args.workload, world),
        "us_per_call": round(ms_per_step * 1e3, 2),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "main_kernel_us": round(main_ms * 1e3, 2),
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_src} (HBM copy bandwidth)",
                     "traffic": recorded_traffic(args.workload),
                     "bytes_per_launch": alg},
        "e2e": {"value": round(throughput(alg, world, e2e_ms), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": 2 * K,
        **({} if draft is None else {"draft_extend": draft}),
        **({} if shards is None else {"kv_shards": shards}),
        **({} if variants is None else {"variants": variants}),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w_cpu = w.to("cpu")
        line["cpu_baseline"] = cpu_baseline(w_cpu, args.cpu_seconds, mla)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle on the host cores: each step is one sequence of the workload's
    shape (its q_len and heads), with the KV length capped so the whole run
    stays within a few minutes."""
    rank = env_int("RANK", 0)
    if rank != 0:
        return
    from speculative_decoding_verify_split_gb300.workloads import make_mla_workload, make_workload
    mla = is_mla(args.workload)
    if mla:
        from oracle.mla_fp64 import mla_oracle_from_torch as oracle_from_torch
    else:
        from oracle.attention_fp64 import oracle_from_torch
    st, key_bytes, _ = reference_structure(args.workload)
    q_lens, kv_lens = st["q_lens"], st["kv_lens"]

    def sample(b, cap, seed):
        S = min(kv_lens[b], cap)
        if mla:
            w = make_mla_workload([q_lens[b]], [S], st["Hq"], st["kv_dtype"], seed=seed)
        else:
            w = make_workload([q_lens[b]], [S], st["Hq"], st["Hkv"], st["kv_dtype"], seed=seed)
        return w, seq_bytes(w, 0, mla)

    # calibrate the cap so that all steps fit in about two minutes
    w, nb = sample(0, 4096, 1000)
    t = time.perf_counter()
    oracle_from_torch(w)
    rate = nb / (time.perf_counter() - t)
    budget = max(0.05, min(20.0, 120.0 / (args.steps + args.warmup)))
    cap = int(max(256, min(max(kv_lens), budget * rate / key_bytes)))

    times, nbytes_total = [], 0
    for i in range(args.warmup + args.steps):
        b = i % len(kv_lens)
        w, nb = sample(b, cap, 2000 + i)
        t = time.perf_counter()
        oracle_from_torch(w)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            times.append(dt)
            nbytes_total += nb
    total = sum(times)
    value = nbytes_total / total / 1e9
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": reference_config(args.workload, args.gpus),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step one sequence of the workload's shape with kv_len "
                                       f"capped at {cap}"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
