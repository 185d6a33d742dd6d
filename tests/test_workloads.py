"""The synthetic workloads match the geometry they are built for (CPU).

Each generator is checked against its stated shape: the tiny decode (2
sequences of 37 and 100 keys, 4 query / 2 K/V heads of 64, a 16-page pool);
GQA decode (64 sequences, 32 / 8 heads of 128, L ~ U[512, 8192] cached keys
plus the new one, the pool 10 % larger than the used pages); chunked prefill
(8 sequences, 512 new tokens over U[2048, 16384] cached keys, causal); the
shared-prefix n-sample step (16 groups x 8 samples, a 4096-token prefix
referenced once per group, private tails U[1, 1024]); and the block-causal
video step (one sequence, 40 heads, 7800 keys = 5 blocks of 1560, 1568 query
rows of which 1560 are real, identity pages).  For every workload the new
tokens' slots are the last keys of their row through the block table, padding
rows have no slot, a sequence's pages are distinct, and K/V values are bf16
draws of N(0, 1)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import workloads as wl

P = 32


def _check_common(c, permuted=True):
    B = c.batch
    kv = c.kv_lens.numpy().astype(np.int64)
    qi = c.q_indptr.numpy().astype(np.int64)
    qr = c.q_real.numpy().astype(np.int64)
    table = c.block_table.numpy()
    slots = c.slots.numpy()
    used = []
    for b in range(B):
        pages = table[b, :(kv[b] + P - 1) // P]
        assert (pages >= 0).all() and (pages < c.num_pages).all()
        used.append(pages)
        # the new tokens are the last keys of the row; padding rows have no slot
        for i in range(qi[b + 1] - qi[b]):
            s = slots[qi[b] + i]
            if i < qr[b]:
                pos = kv[b] - qr[b] + i
                assert s == table[b, pos // P] * P + pos % P
            else:
                assert s == -1
    allp = np.concatenate(used)
    if permuted:
        assert len(np.unique(allp)) == len(allp), "a page serves two sequences"
        assert not np.array_equal(allp, np.arange(len(allp))), "pages are not permuted"
    # bf16 N(0, 1) values over the used pages
    k = c.k_pool[torch.from_numpy(np.unique(allp))].float()
    assert c.k_pool.dtype == torch.bfloat16 and c.v_pool.dtype == torch.bfloat16
    assert abs(k.mean().item()) < 0.02 and 0.97 < k.std().item() < 1.03
    assert c.q.dtype == torch.bfloat16 and abs(c.q.float().std().item() - 1.0) < 0.05


def test_tiny_decode():
    c = wl.tiny_decode()
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.page_size) == (4, 2, 64, P)
    assert c.batch == 2 and c.kv_lens.tolist() == [37, 100] and c.num_pages == 16
    assert c.q.shape[0] == 2 and c.q_real.tolist() == [1, 1]
    _check_common(c)
    # the two free slots of the standalone scatter belong to no sequence's keys
    table = c.block_table.numpy()
    keys = {int(table[b, j // P]) * P + j % P for b, n in enumerate([37, 100]) for j in range(n)}
    free = [int(s) for s in c.extra["free_slots"]]
    assert len(free) == 2 and not (set(free) & keys)


def test_gqa_decode():
    c = wl.gqa_decode()
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.batch) == (32, 8, 128, 64)
    kv = c.kv_lens.numpy()
    assert ((kv - 1 >= 512) & (kv - 1 <= 8192)).all()
    assert c.q.shape[0] == 64 and (c.q_real.numpy() == 1).all()
    used = int(sum((int(n) + P - 1) // P for n in kv))
    assert c.num_pages >= int(np.ceil(used * 1.10)) - 1 and c.num_pages <= used * 1.11 + 1
    assert c.mask == "causal"
    _check_common(c)


def test_chunked_prefill():
    c = wl.chunked_prefill()
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.batch) == (32, 8, 128, 8)
    qi = c.q_indptr.numpy()
    assert (np.diff(qi) == 512).all() and (c.q_real.numpy() == 512).all()
    ctx = c.kv_lens.numpy() - 512
    assert ((ctx >= 2048) & (ctx <= 16384)).all()
    assert c.mask == "causal"
    _check_common(c)


def test_shared_prefix():
    c = wl.shared_prefix()
    e = c.extra
    G, n = e["groups"], e["samples"]
    assert (G, n) == (16, 8) and c.batch == G * n
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim) == (32, 8, 128)
    assert (e["prefix_lens"].numpy() == 4096).all() and tuple(e["prefix_table"].shape) == (G, 128)
    tails = e["tail_lens"].numpy()
    assert ((tails >= 1) & (tails <= 1024)).all()
    assert (c.kv_lens.numpy() == 4096 + tails).all()
    table, pt, tt = c.block_table.numpy(), e["prefix_table"].numpy(), e["tail_table"].numpy()
    for r in range(c.batch):
        # the full row is the group's prefix pages then the sample's own tail pages
        assert (table[r, :128] == pt[r // n]).all()
        tp = (int(tails[r]) + P - 1) // P
        assert (table[r, 128:128 + tp] == tt[r, :tp]).all()
    # each prefix page belongs to one group; no tail page is a prefix page
    assert len(np.unique(pt)) == pt.size
    tail_pages = np.concatenate([tt[r, :(int(tails[r]) + P - 1) // P] for r in range(c.batch)])
    assert len(np.unique(tail_pages)) == len(tail_pages) and not (set(tail_pages) & set(pt.ravel()))
    # the prefix is referenced once per group, not once per sample
    assert pt.size == G * 128
    slots = c.slots.numpy()
    for r in range(c.batch):
        pos = int(c.kv_lens[r]) - 1
        assert slots[r] == table[r, pos // P] * P + pos % P


def test_block_causal_video():
    c = wl.block_causal_video()
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.batch) == (40, 40, 128, 1)
    assert c.kv_lens.tolist() == [7800] and c.q.shape[0] == 1568 and c.q_real.tolist() == [1560]
    assert c.mask == "block_causal" and c.causal_block == 1560
    pages = c.block_table.numpy()[0, :(7800 + P - 1) // P]
    assert (pages == np.arange(len(pages))).all()            # identity page range
    _check_common(c, permuted=False)
