"""Seeded synthetic inputs for target-verify attention.

This module only draws inputs. It holds none of the attention arithmetic, so
both the CPU oracle (through ``tests/``) and the CUDA path can consume the same
bytes without sharing any code that computes the result.

Shapes and value distributions follow the unit test printed on the digest of
sglang PR 36330 ("Key code excerpts", the ``_check_matches_aiter`` test):
bf16 queries drawn from N(0, 1); K and V drawn from N(0, 1) in bf16 and cast
to float8 e4m3 (OCP "FN"); page size 16; head_dim 256; per-tensor descales of
shape [1] in fp32; ``softmax_scale = head_dim ** -0.5``.

Recipe (fixed, so that a workload is reproducible on any machine):

* structure is always drawn on the CPU from ``torch.Generator().manual_seed(seed)``
  in this order: q_lens, kv_lens, physical page permutation, descales;
* the bulk values (Q, then K, then V) are drawn by a second generator on
  ``value_device`` seeded with ``seed + 1``; on the CPU they are drawn in
  fixed chunks of ``_CHUNK`` elements so that memory stays bounded;
* pages are handed out to sequences in order, then permuted by the drawn
  permutation (``block_table = arange`` when ``permute=False``);
* one extra physical page, the poison page, is filled with NaN bytes. Every
  block-table slot beyond a sequence's last page points to it, and (when
  ``poison=True``) the token slots past ``seqused_k[b]`` inside a sequence's
  last page are NaN too. A correct kernel never lets these values reach the
  output.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

PAGE_SIZE = 16
HEAD_DIM = 256
_CHUNK = 1 << 24

FP8 = "fp8_e4m3"
BF16 = "bf16"

# NaN bit patterns: e4m3fn has a single NaN encoding per sign (S.1111.111);
# bf16 quiet NaN 0x7FC0.
_POISON_FP8 = 0x7F
_POISON_BF16 = 0x7FC0


@dataclass
class Workload:
    """One batch of verify-attention inputs (torch tensors on one device)."""

    name: str
    q: torch.Tensor                 # [total_q, Hq, D] bf16
    k_cache: torch.Tensor           # [num_blocks, 16, Hkv, D] float8_e4m3fn or bf16
    v_cache: torch.Tensor           # same as k_cache
    block_table: torch.Tensor       # [B, W] int32
    cu_seqlens_q: torch.Tensor      # [B + 1] int32
    seqused_k: torch.Tensor         # [B] int32
    max_seqlen_q: int
    max_seqlen_k: int
    softmax_scale: float
    k_descale: Optional[torch.Tensor]  # [1] fp32 or None (= 1.0)
    v_descale: Optional[torch.Tensor]
    q_lens: list = field(default_factory=list)
    kv_lens: list = field(default_factory=list)
    poison_page: int = -1

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_cache.shape[2])

    @property
    def kv_dtype(self) -> str:
        return FP8 if self.k_cache.dtype == torch.float8_e4m3fn else BF16

    def algorithmic_bytes(self) -> int:
        """K+V read once per KV head, plus Q read and out written."""
        e = 1 if self.kv_dtype == FP8 else 2
        d = int(self.q.shape[2])
        kv = sum(self.kv_lens) * self.num_kv_heads * d * 2 * e
        qo = 2 * int(self.q.shape[0]) * self.num_q_heads * d * 2
        return kv + qo

    def algorithmic_flops(self) -> int:
        d = int(self.q.shape[2])
        tot = 0
        for L, S in zip(self.q_lens, self.kv_lens):
            for t in range(L):
                tot += max(0, min(S, S - L + t + 1))
        return 4 * d * self.num_q_heads * tot

    def to(self, device) -> "Workload":
        def mv(x):
            return None if x is None else x.to(device)
        return Workload(self.name, mv(self.q), mv(self.k_cache), mv(self.v_cache),
                        mv(self.block_table), mv(self.cu_seqlens_q), mv(self.seqused_k),
                        self.max_seqlen_q, self.max_seqlen_k, self.softmax_scale,
                        mv(self.k_descale), mv(self.v_descale), list(self.q_lens),
                        list(self.kv_lens), self.poison_page)


def _randn(n: int, gen: torch.Generator, device) -> torch.Tensor:
    """n draws of N(0,1) rounded to bf16, in fixed-size chunks."""
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_workload(
    q_lens: Sequence[int],
    kv_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    kv_dtype: str = FP8,
    *,
    seed: int = 0,
    permute: bool = True,
    poison: bool = True,
    k_descale: Optional[float] = None,
    v_descale: Optional[float] = None,
    softmax_scale: Optional[float] = None,
    table_width: Optional[int] = None,
    max_seqlen_k: Optional[int] = None,
    value_device: str = "cpu",
    name: str = "custom",
    head_dim: int = HEAD_DIM,
) -> Workload:
    """Builds a workload with explicit per-sequence lengths (CPU structure)."""
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    B = len(q_lens)
    g = torch.Generator().manual_seed(seed)
    pages_per_seq = [math.ceil(s / PAGE_SIZE) for s in kv_lens]
    n_used = sum(pages_per_seq)
    perm = torch.randperm(n_used, generator=g) if permute else torch.arange(n_used)
    return _assemble(name, q_lens, kv_lens, num_q_heads, num_kv_heads, kv_dtype, seed,
                     perm, poison, k_descale, v_descale, softmax_scale, table_width,
                     max_seqlen_k, value_device, head_dim)


def _assemble(name, q_lens, kv_lens, Hq, Hkv, kv_dtype, seed, perm, poison,
              k_descale, v_descale, softmax_scale, table_width, max_seqlen_k,
              value_device, head_dim, arange_table=False):
    B = len(q_lens)
    D = head_dim
    pages_per_seq = [math.ceil(s / PAGE_SIZE) for s in kv_lens]
    n_used = sum(pages_per_seq)
    W = table_width if table_width is not None else max([1] + pages_per_seq)
    if arange_table:
        num_blocks = B * W
        block_table = torch.arange(num_blocks, dtype=torch.int32).view(B, W)
        poison_page = -1
    else:
        poison_page = n_used
        num_blocks = n_used + 1
        block_table = torch.full((B, W), poison_page, dtype=torch.int32)
        off = 0
        for b, n in enumerate(pages_per_seq):
            block_table[b, :n] = perm[off:off + n].to(torch.int32)
            off += n
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    total_q = int(cu[-1])
    seqused = torch.tensor(kv_lens, dtype=torch.int32)

    gv = torch.Generator(device=value_device).manual_seed(seed + 1)
    q = _randn(total_q * Hq * D, gv, value_device).view(total_q, Hq, D)
    kv_shape = (num_blocks, PAGE_SIZE, Hkv, D)
    n_kv = num_blocks * PAGE_SIZE * Hkv * D
    k = _randn(n_kv, gv, value_device).view(kv_shape)
    v = _randn(n_kv, gv, value_device).view(kv_shape)
    if kv_dtype == FP8:
        k = k.to(torch.float8_e4m3fn)
        v = v.to(torch.float8_e4m3fn)
        bits, pv = torch.uint8, _POISON_FP8
    elif kv_dtype == BF16:
        bits, pv = torch.int16, _POISON_BF16
    else:
        raise ValueError(f"unknown kv dtype {kv_dtype}")

    if poison_page >= 0:
        for t in (k, v):
            t.view(bits)[poison_page].fill_(pv)
    if poison and not arange_table:
        for b in range(B):
            S, n = kv_lens[b], pages_per_seq[b]
            tail = S - (n - 1) * PAGE_SIZE
            if n > 0 and tail < PAGE_SIZE:
                p = int(block_table[b, n - 1])
                for t in (k, v):
                    t.view(bits)[p, tail:].fill_(pv)

    kd = None if k_descale is None else torch.tensor([k_descale], dtype=torch.float32)
    vd = None if v_descale is None else torch.tensor([v_descale], dtype=torch.float32)
    msk = max_seqlen_k if max_seqlen_k is not None else max([0] + kv_lens)
    scale = softmax_scale if softmax_scale is not None else D ** -0.5
    return Workload(name, q, k, v, block_table, cu, seqused, max([0] + q_lens), msk,
                    scale, kd, vd, list(q_lens), list(kv_lens), poison_page)


# ----------------------------------------------------------------------------
# The five verify workloads. Each draws its structure from one CPU generator
# (seed 0 unless given) in the order q_lens, kv_lens, permutation, descales.
# ----------------------------------------------------------------------------

WORKLOADS = (
    "tiny_verify",            # 2 seqs, q [4,2], kv [1024,769], 16q:1kv, fp8, arange table
    "gqa_32q2kv",             # 8 seqs, q in {2,3,4}, kv U[513,4096], 32q:2kv, fp8
    "mid_context_fp8",        # 64 seqs, q 3, kv U[8192,32768], 16q:1kv, fp8, descale U[0.5,2]
    "long_context_fp8",       # 16 seqs, q 4, kv U[65536,131072], 16q:1kv, fp8
    "high_concurrency_bf16",  # 256 seqs, q 2, kv U[2048,16384], 8q:1kv, bf16 KV
)


def workload_structure(name: str, seed: int = 0):
    """Returns (q_lens, kv_lens, Hq, Hkv, kv_dtype, descales, generator-state
    used for the permutation) for one of the named workloads."""
    g = torch.Generator().manual_seed(seed)
    if name == "tiny_verify":
        return dict(q_lens=[4, 2], kv_lens=[1024, 769], Hq=16, Hkv=1, kv_dtype=FP8,
                    gen=g, arange_table=True, table_width=65, descale=(1.0, 1.0))
    if name == "gqa_32q2kv":
        B = 8
        q_lens = torch.randint(2, 5, (B,), generator=g).tolist()
        kv_lens = torch.randint(513, 4097, (B,), generator=g).tolist()
        return dict(q_lens=q_lens, kv_lens=kv_lens, Hq=32, Hkv=2, kv_dtype=FP8, gen=g,
                    descale=(1.0, 1.0))
    if name == "mid_context_fp8":
        B = 64
        q_lens = [3] * B
        kv_lens = torch.randint(8192, 32769, (B,), generator=g).tolist()
        return dict(q_lens=q_lens, kv_lens=kv_lens, Hq=16, Hkv=1, kv_dtype=FP8, gen=g,
                    descale="uniform")
    if name == "long_context_fp8":
        B = 16
        q_lens = [4] * B
        kv_lens = torch.randint(65536, 131073, (B,), generator=g).tolist()
        return dict(q_lens=q_lens, kv_lens=kv_lens, Hq=16, Hkv=1, kv_dtype=FP8, gen=g,
                    descale=(1.0, 1.0))
    if name == "high_concurrency_bf16":
        B = 256
        q_lens = [2] * B
        kv_lens = torch.randint(2048, 16385, (B,), generator=g).tolist()
        return dict(q_lens=q_lens, kv_lens=kv_lens, Hq=8, Hkv=1, kv_dtype=BF16, gen=g,
                    descale=None)
    raise KeyError(f"unknown workload {name!r}; known: {WORKLOADS}")


def named_workload(name: str, seed: int = 0, value_device: str = "cpu") -> Workload:
    st = workload_structure(name, seed)
    g = st["gen"]
    arange = st.get("arange_table", False)
    n_used = sum(math.ceil(s / PAGE_SIZE) for s in st["kv_lens"])
    perm = torch.arange(n_used) if arange else torch.randperm(n_used, generator=g)
    ds = st["descale"]
    if ds == "uniform":
        kd = float(torch.rand(1, generator=g) * 1.5 + 0.5)
        vd = float(torch.rand(1, generator=g) * 1.5 + 0.5)
    elif ds is None:
        kd = vd = None
    else:
        kd, vd = ds
    return _assemble(name, st["q_lens"], st["kv_lens"], st["Hq"], st["Hkv"], st["kv_dtype"],
                     seed, perm, True, kd, vd, None, st.get("table_width"), None,
                     value_device, HEAD_DIM, arange_table=arange)


def flat_kv_slots(w: Workload):
    """The workload's KV layout in the flat token-slot form of the
    draft-extend pass (sglang PR 30105 digest, "Fix 2"): kv_indptr [B+1]
    (token offsets) and kv_indices (the cache slot of every token,
    page * 16 + position), both int32 on the workload's device. Input
    construction only: each sequence's first ceil(S/16) table entries are
    written out token by token."""
    bt = w.block_table.cpu().to(torch.int64)
    indptr, chunks = [0], []
    pos = torch.arange(PAGE_SIZE, dtype=torch.int64)
    for b, S in enumerate(w.kv_lens):
        pages = bt[b, :(S + PAGE_SIZE - 1) // PAGE_SIZE]
        chunks.append((pages[:, None] * PAGE_SIZE + pos[None, :]).reshape(-1)[:S])
        indptr.append(indptr[-1] + S)
    dev = w.block_table.device
    slots = torch.cat(chunks) if chunks else torch.zeros(0, dtype=torch.int64)
    return (torch.tensor(indptr, dtype=torch.int32, device=dev),
            slots.to(torch.int32).to(dev))


def workload_sizes(name: str, seed: int = 0) -> dict:
    """Structure-only summary (no value draws): lengths and byte counts."""
    st = workload_structure(name, seed)
    e = 1 if st["kv_dtype"] == FP8 else 2
    kv = sum(st["kv_lens"]) * st["Hkv"] * HEAD_DIM * 2 * e
    qo = 2 * sum(st["q_lens"]) * st["Hq"] * HEAD_DIM * 2
    return dict(num_seqs=len(st["q_lens"]), q_lens=st["q_lens"], kv_lens=st["kv_lens"],
                Hq=st["Hq"], Hkv=st["Hkv"], kv_dtype=st["kv_dtype"], kv_bytes=kv,
                algorithmic_bytes=kv + qo)


# ----------------------------------------------------------------------------
# Absorbed-MLA latent-cache workloads (sglang PR 34517 digest, "Implementation
# breakdown" item 1: one TP-local KV head that is the MLA latent, NOPE_DIM
# latent columns plus PE_DIM = 64 RoPE columns). Same recipe as above: one
# CPU generator draws q_lens, kv_lens, the page permutation and descales; a
# value generator seeded with seed + 1 draws Q then the cache rows, N(0, 1)
# rounded to bf16 (then cast to e4m3 for an FP8 cache). The latent width is
# not on the pages: 512, as in the DeepSeek-V3 / Kimi-K2 MLA family. The
# default softmax scale is that family's, 1 / sqrt(128 + 64) (the query-key
# head width before absorption).
# ----------------------------------------------------------------------------

MLA_NOPE_DIM = 512
MLA_PE_DIM = 64


@dataclass
class MlaWorkload:
    """One batch of verify-attention inputs over a latent cache."""

    name: str
    q: torch.Tensor                 # [total_q, Hq, NOPE + PE] bf16: [q_nope | q_pe]
    kv_cache: torch.Tensor          # [num_blocks, 16, 1, NOPE + PE]: [latent | rope key]
    block_table: torch.Tensor       # [B, W] int32
    cu_seqlens_q: torch.Tensor      # [B + 1] int32
    seqused_k: torch.Tensor         # [B] int32
    max_seqlen_q: int
    max_seqlen_k: int
    softmax_scale: float
    k_descale: Optional[torch.Tensor]
    v_descale: Optional[torch.Tensor]
    q_lens: list = field(default_factory=list)
    kv_lens: list = field(default_factory=list)
    poison_page: int = -1
    nope_dim: int = MLA_NOPE_DIM

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return 1

    @property
    def kv_dtype(self) -> str:
        return FP8 if self.kv_cache.dtype == torch.float8_e4m3fn else BF16

    def algorithmic_bytes(self) -> int:
        """Each cache row read once (its latent serves as K and V), plus Q
        read and out (NOPE_DIM wide) written."""
        e = 1 if self.kv_dtype == FP8 else 2
        dq = int(self.q.shape[2])
        tq = int(self.q.shape[0])
        return sum(self.kv_lens) * dq * e + tq * self.num_q_heads * (dq + self.nope_dim) * 2

    def algorithmic_flops(self) -> int:
        dq = int(self.q.shape[2])
        tot = 0
        for L, S in zip(self.q_lens, self.kv_lens):
            for t in range(L):
                tot += max(0, min(S, S - L + t + 1))
        return 2 * (dq + self.nope_dim) * self.num_q_heads * tot

    def to(self, device) -> "MlaWorkload":
        def mv(x):
            return None if x is None else x.to(device)
        return MlaWorkload(self.name, mv(self.q), mv(self.kv_cache), mv(self.block_table),
                           mv(self.cu_seqlens_q), mv(self.seqused_k), self.max_seqlen_q,
                           self.max_seqlen_k, self.softmax_scale, mv(self.k_descale),
                           mv(self.v_descale), list(self.q_lens), list(self.kv_lens),
                           self.poison_page, self.nope_dim)


def make_mla_workload(
    q_lens: Sequence[int],
    kv_lens: Sequence[int],
    num_q_heads: int,
    kv_dtype: str = FP8,
    *,
    seed: int = 0,
    permute: bool = True,
    poison: bool = True,
    k_descale: Optional[float] = None,
    v_descale: Optional[float] = None,
    softmax_scale: Optional[float] = None,
    max_seqlen_k: Optional[int] = None,
    value_device: str = "cpu",
    name: str = "custom_mla",
    nope_dim: int = MLA_NOPE_DIM,
    pe_dim: int = MLA_PE_DIM,
    _gen: Optional[torch.Generator] = None,
) -> MlaWorkload:
    """Builds a latent-cache workload with explicit per-sequence lengths."""
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    B = len(q_lens)
    g = _gen if _gen is not None else torch.Generator().manual_seed(seed)
    pages_per_seq = [math.ceil(s / PAGE_SIZE) for s in kv_lens]
    n_used = sum(pages_per_seq)
    perm = torch.randperm(n_used, generator=g) if permute else torch.arange(n_used)
    if k_descale == "uniform":
        k_descale = float(torch.rand(1, generator=g) * 1.5 + 0.5)
        v_descale = float(torch.rand(1, generator=g) * 1.5 + 0.5)
    W = max([1] + pages_per_seq)
    poison_page = n_used
    num_blocks = n_used + 1
    block_table = torch.full((B, W), poison_page, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        block_table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    total_q = int(cu[-1])
    D = nope_dim + pe_dim
    gv = torch.Generator(device=value_device).manual_seed(seed + 1)
    q = _randn(total_q * num_q_heads * D, gv, value_device).view(total_q, num_q_heads, D)
    kv = _randn(num_blocks * PAGE_SIZE * D, gv, value_device).view(num_blocks, PAGE_SIZE, 1, D)
    if kv_dtype == FP8:
        kv = kv.to(torch.float8_e4m3fn)
        bits, pv = torch.uint8, _POISON_FP8
    elif kv_dtype == BF16:
        bits, pv = torch.int16, _POISON_BF16
    else:
        raise ValueError(f"unknown kv dtype {kv_dtype}")
    kv.view(bits)[poison_page].fill_(pv)
    if poison:
        for b in range(B):
            S, n = kv_lens[b], pages_per_seq[b]
            tail = S - (n - 1) * PAGE_SIZE
            if n > 0 and tail < PAGE_SIZE:
                kv.view(bits)[int(block_table[b, n - 1]), tail:].fill_(pv)
    kd = None if k_descale is None else torch.tensor([k_descale], dtype=torch.float32)
    vd = None if v_descale is None else torch.tensor([v_descale], dtype=torch.float32)
    msk = max_seqlen_k if max_seqlen_k is not None else max([0] + kv_lens)
    scale = softmax_scale if softmax_scale is not None else (128 + 64) ** -0.5
    return MlaWorkload(name, q, kv, block_table, cu, torch.tensor(kv_lens, dtype=torch.int32),
                       max([0] + q_lens), msk, scale, kd, vd, q_lens, kv_lens, poison_page,
                       nope_dim)


MLA_WORKLOADS = (
    "mla_tiny",                # 2 seqs, q [4,2], kv [1024,769], 16 heads, fp8 latent
    "mla_mid_context_fp8",     # 64 seqs, q 3, kv U[8192,32768], 16 heads, descale U[0.5,2]
    "mla_long_context_fp8",    # 16 seqs, q 4, kv U[65536,131072], 16 heads, fp8 latent
    "mla_tiny_bf16",           # the same shapes on a bf16 latent cache
    "mla_mid_context_bf16",
    "mla_long_context_bf16",
)


def mla_workload_structure(name: str, seed: int = 0) -> dict:
    """q_lens, kv_lens, heads and descales of a named latent-cache workload
    (the shapes of the GQA workloads of the same names, on a latent cache)."""
    g = torch.Generator().manual_seed(seed)
    if name.endswith("_bf16"):  # the FP8 workload's structure on a bf16 cache
        st = mla_workload_structure(name[:-len("_bf16")] + ("" if name == "mla_tiny_bf16" else "_fp8"), seed)
        st["kv_dtype"] = BF16
        return st
    if name == "mla_tiny":
        return dict(q_lens=[4, 2], kv_lens=[1024, 769], Hq=16, gen=g, descale=None)
    if name == "mla_mid_context_fp8":
        return dict(q_lens=[3] * 64, kv_lens=torch.randint(8192, 32769, (64,), generator=g).tolist(),
                    Hq=16, gen=g, descale="uniform")
    if name == "mla_long_context_fp8":
        return dict(q_lens=[4] * 16, kv_lens=torch.randint(65536, 131073, (16,), generator=g).tolist(),
                    Hq=16, gen=g, descale=None)
    raise KeyError(f"unknown workload {name!r}; known: {MLA_WORKLOADS}")


def named_mla_workload(name: str, seed: int = 0, value_device: str = "cpu") -> MlaWorkload:
    st = mla_workload_structure(name, seed)
    return make_mla_workload(st["q_lens"], st["kv_lens"], st["Hq"], st.get("kv_dtype", FP8), seed=seed,
                             k_descale=st["descale"], value_device=value_device, name=name,
                             _gen=st["gen"])


def split_kv_shards(w: Workload, n: int, seed: int = 0):
    """Input construction for the sharded (context-parallel) path: each
    sequence's keys cut into n contiguous, page-aligned shards of random sizes
    (some may be empty). Returns a list of n (block_table, seqused_k,
    kv_extent) triples on the workload's device: shard i of sequence b holds
    the keys [o, o + S_i) of the sequence through its own table rows (the
    sequence's pages [o / 16, ...)), and kv_extent = S_b - o."""
    g = torch.Generator().manual_seed(seed)
    bt = w.block_table.cpu()
    B, W = bt.shape
    dev = w.block_table.device
    tables = [torch.full((B, W), max(w.poison_page, 0), dtype=torch.int32) for _ in range(n)]
    used = [torch.zeros(B, dtype=torch.int32) for _ in range(n)]
    ext = [torch.zeros(B, dtype=torch.int32) for _ in range(n)]
    for b, S in enumerate(w.kv_lens):
        pages = (S + PAGE_SIZE - 1) // PAGE_SIZE
        cuts = sorted(torch.randint(0, pages + 1, (n - 1,), generator=g).tolist()) if n > 1 else []
        bounds = [0] + [c * PAGE_SIZE for c in cuts] + [S]
        for i in range(n):
            lo, hi = min(bounds[i], S), min(bounds[i + 1], S)
            hi = max(hi, lo)
            p0, p1 = lo // PAGE_SIZE, (hi + PAGE_SIZE - 1) // PAGE_SIZE
            tables[i][b, :p1 - p0] = bt[b, p0:p1]
            used[i][b] = hi - lo
            ext[i][b] = S - lo
    return [(t.to(dev), u.to(dev), e.to(dev)) for t, u, e in zip(tables, used, ext)]
