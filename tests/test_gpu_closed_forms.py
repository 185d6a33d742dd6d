"""GPU checks of paged_attention against closed forms, and at long contexts.

With q = 0 every visible key scores 0, so each visible key gets the same
weight: LSE = ln(n) for n visible keys and O = the mean of the visible V rows.
With V row j one-hot at column j mod D, O[d] = (number of visible j with
j mod D = d) / n, which names the visible set: the causal, block-causal and
padding boundaries of each kernel are pinned without the oracle (the
visibility rules of "Paged causal K/V cache and cached attention for
VisualGen", Description, Attention; the q = 0 / one-hot V check is the one its
test notes describe).  The long-context cases run one sequence of 131,072+
keys through the decode kernel (about a hundred fused split partials) and the
tile kernel (key splits), compared with the oracle on sampled rows."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl
from pkv_testutil import assert_attention_close, gpu_step, oracle_step

pytestmark = pytest.mark.gpu
P = 32


def visible_count(i, q_real, kv_len, mask, cb):
    """Keys visible to query row i (row i sits at position kv_len - q_real + i)."""
    if i >= q_real:
        return 0
    first = kv_len - q_real
    if mask == "none":
        return kv_len
    if mask == "causal":
        return first + i + 1
    return first + min(q_real, (i // cb + 1) * cb)


def one_hot_case(seed, kv_lens, q_rows, q_real, Hq, Hkv, D, mask, cb=0):
    """A pool case with q = 0 and V row j of every sequence one-hot at j mod D
    (every head), all keys already in the pool (no scatter)."""
    c = wl.build_pool_case(f"onehot_{seed}", seed, kv_lens, q_rows, q_real, Hq, Hkv, D,
                           mask=mask, causal_block=cb)
    c.q.zero_()
    v = c.v_pool.view(-1, Hkv, D)
    table = c.block_table.numpy()
    for b, L in enumerate(kv_lens):
        j = np.arange(L)
        slots = torch.from_numpy(table[b, j // P].astype(np.int64) * P + j % P)
        rows = torch.zeros((L, Hkv, D), dtype=torch.bfloat16)
        rows[torch.arange(L), :, torch.from_numpy(j % D)] = 1.0
        v[slots] = rows
    return c


def expected(c, mask, cb):
    """(O, LSE, real) from the closed form."""
    D, Hq = c.head_dim, c.num_q_heads
    qi, qr, kl = c.q_indptr.numpy(), c.q_real.numpy(), c.kv_lens.numpy()
    rows = c.q.shape[0]
    O = np.zeros((rows, Hq, D))
    L = np.full((rows, Hq), -np.inf)
    for b in range(c.batch):
        for i in range(qi[b + 1] - qi[b]):
            n = visible_count(i, int(qr[b]), int(kl[b]), mask, cb)
            if n == 0:
                continue
            counts = np.full(D, n // D, dtype=np.float64)
            counts[: n % D] += 1
            O[qi[b] + i] = counts / n
            L[qi[b] + i] = math.log(n)
    return O, L


def check(out, lse, O, L):
    got = out.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)
    pad = np.isneginf(L[:, 0])
    assert (got[pad] == 0).all(), "padding rows must be zero"
    assert np.isneginf(gl[pad]).all()
    # bf16 output: within one bf16 ulp (2^-8 relative) of the exact ratio
    err = np.abs(got[~pad] - O[~pad])
    assert (err <= np.abs(O[~pad]) * 2.0 ** -8 + 1e-6).all(), f"max err {err.max():.3e}"
    assert np.abs(gl[~pad] - L[~pad]).max() <= 1e-4


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 4, 64), (6, 6, 128)])
@pytest.mark.parametrize("num_splits", [0, 1, 4])
def test_q_zero_decode(Hq, Hkv, D, num_splits):
    rng = np.random.default_rng(3 + D + num_splits)
    kv = rng.integers(1, 1500, size=9)
    kv[0], kv[1] = 1, 32       # a single key; exactly one page
    q_real = np.ones(9, dtype=np.int64)
    q_real[4] = 0              # a padding row
    c = one_hot_case(11, kv, np.ones(9), q_real, Hq, Hkv, D, "causal")
    out, lse, *_, err = gpu_step(c, scatter=False, num_splits=num_splits)
    assert err == 0
    check(out, lse, *expected(c, "causal", 0))


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 37), ("block_causal", 128),
                                     ("none", 0)])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8)])
@pytest.mark.parametrize("num_splits", [0, 2])
def test_q_zero_tile_kernel(mask, cb, Hq, Hkv, num_splits):
    """Several rows per sequence (one- and two-tile CTAs, ragged last tiles,
    padding rows) through the tensor-core tile kernel."""
    rng = np.random.default_rng(5 + Hq + cb + num_splits)
    B = 5
    q_real = rng.integers(2, 300, size=B)
    q_real[0] = 1 if Hq == Hkv else 2
    pad = rng.integers(0, 9, size=B)
    kv = q_real + rng.integers(0, 1300, size=B)
    c = one_hot_case(13, kv, q_real + pad, q_real, Hq, Hkv, 128, mask, cb)
    out, lse, *_, err = gpu_step(c, scatter=False, num_splits=num_splits)
    assert err == 0
    check(out, lse, *expected(c, mask, cb))


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 20), ("none", 0)])
def test_q_zero_simt_kernel(mask, cb):
    """The generic kernel (head_dim 64 with several rows)."""
    rng = np.random.default_rng(17 + cb)
    q_real = rng.integers(1, 60, size=4)
    kv = q_real + rng.integers(0, 400, size=4)
    c = one_hot_case(19, kv, q_real + 3, q_real, 8, 2, 64, mask, cb)
    out, lse, *_, err = gpu_step(c, scatter=False, flags=pkv.PKV_FLAG_SIMT_ONLY)
    assert err == 0
    check(out, lse, *expected(c, mask, cb))


def test_decode_long_context_many_splits():
    """Two sequences of 131,073 and 70,001 keys, one decode row each: the
    automatic split gives on the order of a hundred partial states per (row,
    head), merged by the last split to finish."""
    c = wl.build_pool_case("long_decode", 23, [131073, 70001], [1, 1], [1, 1], 8, 2, 128,
                           mask="causal")
    out, lse, *_, err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


def test_tile_kernel_long_context_sampled():
    """200 new query tokens over a 131,272-key context (causal, 8/2 heads):
    the tile kernel with key splits, sampled rows against the oracle."""
    c = wl.build_pool_case("long_prefill", 29, [131272], [208], [200], 8, 2, 128, mask="causal")
    out, lse, *_, err = gpu_step(c)
    rows = [0, 1, 31, 32, 99, 150, 199, 200, 207]
    O, L, *_ = oracle_step(c, rows=rows)
    assert err == 0
    assert_attention_close(out, lse, O, L, c, rows=rows)
