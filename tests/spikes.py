"""Input construction for mask-boundary checks at any length: a key that only
some draft tokens may see, with a logit far above every other key's. A
one-key error in the causal mask then changes whole rows, whatever the
sequence length (on random keys it would move a row by ~1/S)."""
import torch

PAGE_SIZE = 16


def plant_boundary_spikes(w):
    """Every sequence's draft-token queries set to one vector u (its first
    token's first head), and the key at position S - L + 1 of every KV head
    (visible to tokens t >= 1 only) set to 8 sign(u): its logit is
    softmax_scale * k_descale * 8 sum|u| (~100 at head_dim 256, scale 1/16)
    against about N(0, 1) for the others. Sequences with L < 2 are left
    alone. Works on CPU or GPU tensors; returns w."""
    cu = w.cu_seqlens_q.tolist()
    for b, (L, S) in enumerate(zip(w.q_lens, w.kv_lens)):
        if L < 2 or S < L:
            continue
        u = w.q[cu[b], 0].clone()
        w.q[cu[b]:cu[b + 1]] = u
        j = S - L + 1
        page = int(w.block_table[b, j // PAGE_SIZE])
        spike = torch.where(u.float() >= 0, 8.0, -8.0).to(w.k_cache.dtype)
        w.k_cache[page, j % PAGE_SIZE, :] = spike
    return w
