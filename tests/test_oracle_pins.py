"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one oracle function to an independent anchor: a library routine
computing the same quantity from a different formulation (torch's
scaled-dot-product attention on contiguous K/V with a mask built from block
membership, numpy fancy indexing, numpy.roll), a closed form, a hand-derived
fixture (tests/golden/visible_keys.txt) or an invariant the pages fix (page
permutation, merge of prefix and tail equals full attention, padding rows).
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t):
    return orc.bf16_bits(t)


def f64(t):
    return orc.bf16_to_f64(orc.bf16_bits(t))


def bf16_from_f64(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def build_pool(kv_per_seq, perm_seed, page=32, extra_pages=3):
    """Lay contiguous per-sequence K (or V) ``[L, H, D]`` bf16 tensors into a
    pool whose pages are a random permutation; return (pool, table)."""
    rng = np.random.default_rng(perm_seed)
    n_pages = [(x.shape[0] + page - 1) // page for x in kv_per_seq]
    total = sum(n_pages) + extra_pages
    H, D = kv_per_seq[0].shape[1:]
    pool = torch.zeros(total, page, H, D, dtype=torch.bfloat16)
    perm = rng.permutation(total)
    table = np.full((len(kv_per_seq), max(n_pages)), -1, dtype=np.int32)
    at = 0
    for b, x in enumerate(kv_per_seq):
        for j in range(n_pages[b]):
            phys = int(perm[at]); at += 1
            table[b, j] = phys
            chunk = x[j * page:(j + 1) * page]
            pool[phys, :chunk.shape[0]] = chunk
    return pool, table


def mask_by_block_membership(n_rows, q_real, kv_len, mask, cb):
    """Visibility written from block membership (a different formulation from
    the oracle's count of leading keys): key j is either cached (before this
    step's tokens) or new token number j - first_new; a new key is visible to
    real row i if it is not later than i (causal) or not in a later block than
    i (block-causal)."""
    first_new = kv_len - q_real
    m = np.zeros((n_rows, kv_len), dtype=bool)
    for i in range(min(n_rows, q_real)):
        for j in range(kv_len):
            if j < first_new or mask == "none":
                m[i, j] = True
            elif mask == "causal":
                m[i, j] = (j - first_new) <= i
            else:
                m[i, j] = (j - first_new) // cb <= i // cb
    return m


# ----------------------------------------------------------------------------
# attention vs torch SDPA (library routine) on contiguous K/V
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 3), ("block_causal", 5),
                                     ("none", 0)])
@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 16), (6, 6, 8), (8, 2, 32)])
def test_attention_matches_sdpa(mask, cb, Hq, Hkv, D):
    gen = torch.Generator().manual_seed(11)
    rng = np.random.default_rng(12)
    B = 3
    kv_lens = [int(x) for x in rng.integers(1, 90, size=B)]
    q_real = [int(rng.integers(1, min(L, 12) + 1)) for L in kv_lens]
    q_rows = [qr + int(rng.integers(0, 3)) for qr in q_real]
    Ks = [wl.randn_bf16((L, Hkv, D), gen) for L in kv_lens]
    Vs = [wl.randn_bf16((L, Hkv, D), gen) for L in kv_lens]
    q = wl.randn_bf16((sum(q_rows), Hq, D), gen, scale=2.0)
    k_pool, table = build_pool(Ks, 5)
    v_pool, table_v = build_pool(Vs, 5)
    assert (table == table_v).all()
    indptr = np.concatenate([[0], np.cumsum(q_rows)]).astype(np.int32)
    O, L = orc.paged_attention(q, k_pool, v_pool, table, kv_lens, indptr, q_real,
                               mask=mask, causal_block=cb)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        r0, r1 = indptr[b], indptr[b + 1]
        Qt = torch.from_numpy(f64(q[r0:r1])).permute(1, 0, 2)          # [Hq, n, D]
        Kt = torch.from_numpy(f64(Ks[b])).permute(1, 0, 2)             # [Hkv, L, D]
        Vt = torch.from_numpy(f64(Vs[b])).permute(1, 0, 2)
        vis = mask_by_block_membership(r1 - r0, q_real[b], kv_lens[b], mask, cb)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Qt, Kt, Vt, attn_mask=torch.from_numpy(vis), scale=scale, enable_gqa=True)
        ref = ref.permute(1, 0, 2).numpy()
        real = slice(0, q_real[b])
        np.testing.assert_allclose(O[r0:r1][real], ref[real], rtol=1e-11, atol=1e-12)
        # LSE against scipy's logsumexp of the masked scores
        from scipy.special import logsumexp
        G = Hq // Hkv
        s = np.einsum("nhd,hld->hnl", f64(q[r0:r1]),
                      np.repeat(f64(Ks[b]).transpose(1, 0, 2), G, axis=0)) * scale
        s = np.where(vis[None], s, -np.inf)
        lse_ref = logsumexp(s, axis=-1).T                             # [n, Hq]
        np.testing.assert_allclose(L[r0:r1][real], lse_ref[real], rtol=1e-12, atol=1e-12)
        # padding rows: zero output, -inf LSE
        assert (O[r0:r1][q_real[b]:] == 0).all()
        assert np.isneginf(L[r0:r1][q_real[b]:]).all()


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 2), ("block_causal", 4), ("none", 0)])
def test_more_new_tokens_than_keys_matches_sdpa(mask, cb):
    """Rows positioned before key 0 (q_real > kv_len): the oracle against SDPA
    with the block-membership mask, where new token j - first_new with
    first_new < 0 is key j.  Rows the mask leaves empty come back zero with
    LSE -inf (SDPA has no value for them)."""
    gen = torch.Generator().manual_seed(21)
    Hq, Hkv, D = 4, 2, 16
    cases = [(3, 7), (1, 5), (6, 9)]                 # (kv_len, q_real)
    Ks = [wl.randn_bf16((L, Hkv, D), gen) for L, _ in cases]
    Vs = [wl.randn_bf16((L, Hkv, D), gen) for L, _ in cases]
    q_real = [qr for _, qr in cases]
    q = wl.randn_bf16((sum(q_real), Hq, D), gen, scale=2.0)
    k_pool, table = build_pool(Ks, 7)
    v_pool, _ = build_pool(Vs, 7)
    indptr = np.concatenate([[0], np.cumsum(q_real)]).astype(np.int32)
    kv_lens = [L for L, _ in cases]
    O, L = orc.paged_attention(q, k_pool, v_pool, table, kv_lens, indptr, q_real, mask=mask, causal_block=cb)
    scale = 1.0 / math.sqrt(D)
    empty_seen = 0
    for b, (kv, qr) in enumerate(cases):
        r0, r1 = indptr[b], indptr[b + 1]
        vis = mask_by_block_membership(qr, qr, kv, mask, cb)
        some = vis.any(axis=1)
        Qt = torch.from_numpy(f64(q[r0:r1])).permute(1, 0, 2)
        Kt = torch.from_numpy(f64(Ks[b])).permute(1, 0, 2)
        Vt = torch.from_numpy(f64(Vs[b])).permute(1, 0, 2)
        if some.any():
            ref = torch.nn.functional.scaled_dot_product_attention(
                Qt[:, some], Kt, Vt, attn_mask=torch.from_numpy(vis[some]), scale=scale,
                enable_gqa=True).permute(1, 0, 2).numpy()
            np.testing.assert_allclose(O[r0:r1][some], ref, rtol=1e-11, atol=1e-12)
        assert (O[r0:r1][~some] == 0).all() and np.isneginf(L[r0:r1][~some]).all()
        empty_seen += int((~some).sum())
        for i in range(qr):
            assert orc.visible_keys(i, qr, kv, mask, max(cb, 1)) == int(vis[i].sum())
    if mask != "none":
        assert empty_seen > 0


# ----------------------------------------------------------------------------
# visible-key sets against the hand-derived golden fixture
# ----------------------------------------------------------------------------

def load_visible_cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "visible_keys.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case"):
            _, mask, kv, qr, rows, cb = line.split()
            cur = dict(mask=mask, kv=int(kv), q_real=int(qr), rows=int(rows), cb=int(cb), vis={})
            cases.append(cur)
            continue
        row, keys = line.split(":")
        keys = keys.strip()
        s = set()
        if keys != "-":
            for part in keys.split(","):
                a, _, b = part.partition("-")
                s.update(range(int(a), int(b or a) + 1))
        cur["vis"][int(row)] = s
    return cases


@pytest.mark.parametrize("case", load_visible_cases(),
                         ids=lambda c: f"{c['mask']}-{c['kv']}-{c['q_real']}-{c['rows']}-{c['cb']}")
def test_visible_key_sets_one_hot(case):
    """q = 0 makes the weights uniform; V row j = e_j reads the set back."""
    kv, rows = case["kv"], case["rows"]
    D = 16
    assert kv <= D
    V = torch.zeros(kv, 1, D, dtype=torch.bfloat16)
    for j in range(kv):
        V[j, 0, j] = 1.0
    K = wl.randn_bf16((kv, 1, D), torch.Generator().manual_seed(3))
    k_pool, table = build_pool([K], 1)
    v_pool, _ = build_pool([V], 1)
    q = torch.zeros(rows, 1, D, dtype=torch.bfloat16)
    O, L = orc.paged_attention(q, k_pool, v_pool, table, [kv], [0, rows], [case["q_real"]],
                               mask=case["mask"], causal_block=case["cb"])
    for i in range(rows):
        expect = case["vis"][i]
        got = {d for d in range(D) if O[i, 0, d] != 0}
        assert got == expect, (i, got, expect)
        if expect:
            np.testing.assert_allclose(O[i, 0, sorted(expect)], 1.0 / len(expect), rtol=1e-15)
            assert L[i, 0] == pytest.approx(math.log(len(expect)), abs=1e-15)
        else:
            assert np.isneginf(L[i, 0])
        assert orc.visible_keys(i, case["q_real"], kv, case["mask"], case["cb"]) == len(expect)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

def _single_seq(K, V, q, mask="causal"):
    k_pool, table = build_pool([K], 2)
    v_pool, _ = build_pool([V], 2)
    n = q.shape[0]
    return orc.paged_attention(q, k_pool, v_pool, table, [K.shape[0]], [0, n], [n], mask=mask)


def test_single_key_closed_form():
    """One key: O = V_0 and LSE = scale * q . k_0."""
    D = 8
    K = bf16_from_f64(np.arange(D).reshape(1, 1, D) * 0.25)
    V = bf16_from_f64(np.linspace(-1, 1, D).reshape(1, 1, D))
    q = bf16_from_f64(np.ones((1, 1, D)) * 0.5)
    O, L = _single_seq(K, V, q)
    np.testing.assert_array_equal(O[0, 0], f64(V)[0, 0])
    assert L[0, 0] == pytest.approx(0.5 * 0.25 * sum(range(D)) / math.sqrt(D), rel=1e-15)


def test_two_keys_closed_form():
    """Two keys: weights are a logistic pair; LSE = s0 + ln(1 + e^(s1 - s0))."""
    D = 4
    K = bf16_from_f64([[[2.0, 0, 0, 0]], [[0, 1.0, 0, 0]]])
    V = bf16_from_f64([[[1.0, 0, 3.0, 0]], [[0, 1.0, 0, -2.0]]])
    q = bf16_from_f64([[[1.0, 0.5, 0, 0]]])
    O, L = _single_seq(K, V, q)
    scale = 1 / math.sqrt(D)
    s0, s1 = 2.0 * scale, 0.5 * scale
    w0 = 1 / (1 + math.exp(s1 - s0))
    w1 = 1 - w0
    np.testing.assert_allclose(O[0, 0], [w0, w1, 3 * w0, -2 * w1], rtol=1e-14)
    assert L[0, 0] == pytest.approx(s0 + math.log1p(math.exp(s1 - s0)), rel=1e-15)


def test_identical_keys_give_mean_and_log_count():
    """All keys equal: uniform weights; LSE = s + ln n."""
    n, D = 37, 8
    K = bf16_from_f64(np.tile(np.array([0.5, -1, 0, 2, 0, 0, 1, 0]), (n, 1, 1)))
    V = wl.randn_bf16((n, 1, D), torch.Generator().manual_seed(4))
    q = bf16_from_f64(np.array([[[1.0, 1, 1, 1, 1, 1, 1, 1]]]))
    O, L = _single_seq(K, V, q)
    np.testing.assert_allclose(O[0, 0], f64(V).mean(axis=0)[0], rtol=1e-13, atol=1e-15)
    s = (0.5 - 1 + 2 + 1) / math.sqrt(D)
    assert L[0, 0] == pytest.approx(s + math.log(n), rel=1e-14)


def test_peaked_scores_select_one_value():
    """One key far above the rest: O equals that key's value to fp64 precision."""
    n, D = 50, 8
    K = torch.zeros(n, 1, D, dtype=torch.bfloat16)
    K[17, 0, 0] = 64.0
    V = wl.randn_bf16((n, 1, D), torch.Generator().manual_seed(5))
    q = torch.zeros(1, 1, D, dtype=torch.bfloat16)
    q[0, 0, 0] = 64.0
    O, L = _single_seq(K, V, q)
    np.testing.assert_allclose(O[0, 0], f64(V)[17, 0], rtol=1e-12, atol=1e-300)


# ----------------------------------------------------------------------------
# invariants the pages fix
# ----------------------------------------------------------------------------

def _permute_pages(case, seed):
    """Move every physical page to a new index and rewrite the table."""
    rng = np.random.default_rng(seed)
    P = case.num_pages
    perm = rng.permutation(P)          # new index of old page p is perm[p]
    k_new = torch.empty_like(case.k_pool)
    v_new = torch.empty_like(case.v_pool)
    k_new[torch.from_numpy(perm)] = case.k_pool
    v_new[torch.from_numpy(perm)] = case.v_pool
    t = case.block_table.numpy().copy()
    t[t >= 0] = perm[t[t >= 0]]
    return k_new, v_new, t


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 4), ("none", 0)])
def test_page_permutation_invariance(mask, cb):
    c = wl.random_case(21, batch=3, Hq=4, Hkv=2, D=16, kv_range=(5, 140), q_range=(1, 9),
                       pad_range=(0, 2), mask=mask, causal_block=cb)
    O1, L1 = orc.paged_attention(c.q, c.k_pool, c.v_pool, c.block_table, c.kv_lens,
                                 c.q_indptr, c.q_real, mask=mask, causal_block=cb)
    k2, v2, t2 = _permute_pages(c, 7)
    O2, L2 = orc.paged_attention(c.q, k2, v2, t2, c.kv_lens, c.q_indptr, c.q_real,
                                 mask=mask, causal_block=cb)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_merge_of_prefix_and_tail_equals_full_attention():
    """[SP]: prefix attention (all samples, no mask) + private-tail attention,
    merged by LSE, equals attention over the whole row."""
    c = wl.shared_prefix(seed=31, groups=2, samples=3, prefix=64, tail_lo=1, tail_hi=70,
                         Hq=4, Hkv=2, D=16)
    e = c.extra
    O_full, L_full = orc.paged_attention(c.q, c.k_pool, c.v_pool, c.block_table, c.kv_lens,
                                         c.q_indptr, c.q_real, mask="causal")
    O_p, L_p = orc.paged_attention(c.q, c.k_pool, c.v_pool, e["prefix_table"],
                                   e["prefix_lens"], e["prefix_q_indptr"], e["prefix_q_real"],
                                   mask="none")
    O_t, L_t = orc.paged_attention(c.q, c.k_pool, c.v_pool, e["tail_table"], e["tail_lens"],
                                   c.q_indptr, c.q_real, mask="causal")
    O_m, L_m = orc.merge_attn_states(O_p, L_p, O_t, L_t)
    np.testing.assert_allclose(O_m, O_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L_m, L_full, rtol=1e-13, atol=1e-13)


def test_gqa_equals_repeated_kv_heads():
    """Grouped-query heads: Hq/Hkv query heads per K/V head equals MHA with
    each K/V head repeated for its group (torch.repeat_interleave)."""
    c = wl.random_case(41, batch=2, Hq=8, Hkv=2, D=16, kv_range=(3, 80), q_range=(1, 4))
    O1, L1 = orc.paged_attention(c.q, c.k_pool, c.v_pool, c.block_table, c.kv_lens,
                                 c.q_indptr, c.q_real)
    kr = c.k_pool.repeat_interleave(4, dim=2)
    vr = c.v_pool.repeat_interleave(4, dim=2)
    O2, L2 = orc.paged_attention(c.q, kr, vr, c.block_table, c.kv_lens, c.q_indptr, c.q_real)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_split_kv_merge_order_independent():
    """Split the keys of a row into chunks, attend each, merge in two orders."""
    gen = torch.Generator().manual_seed(9)
    n, D = 200, 16
    K = wl.randn_bf16((n, 1, D), gen)
    V = wl.randn_bf16((n, 1, D), gen)
    q = wl.randn_bf16((1, 1, D), gen)
    O_full, L_full = _single_seq(K, V, q)
    cuts = [0, 33, 64, 65, 150, 200]
    parts = [_single_seq(K[a:b], V[a:b], q, mask="none") for a, b in zip(cuts, cuts[1:])]
    Os = [p[0] for p in parts]
    Ls = [p[1] for p in parts]
    O1, L1 = orc.merge_many(Os, Ls)
    O2, L2 = orc.merge_many(Os[::-1], Ls[::-1])
    np.testing.assert_allclose(O1, O_full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(O2, O_full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L1, L_full, rtol=1e-14)
    np.testing.assert_allclose(L2, L_full, rtol=1e-14)


def test_merge_special_cases():
    oa = np.array([[1.0, 2.0]]); ob = np.array([[3.0, -4.0]])
    # equal LSE: plain average, LSE + ln 2
    o, l = orc.merge_attn_states(oa, np.array([0.7]), ob, np.array([0.7]))
    np.testing.assert_allclose(o, [[2.0, -1.0]]); assert l[0] == pytest.approx(0.7 + math.log(2))
    # empty second state: first state unchanged
    o, l = orc.merge_attn_states(oa, np.array([1.5]), ob, np.array([-np.inf]))
    np.testing.assert_array_equal(o, oa); assert l[0] == 1.5
    # both empty: zero output, -inf, never NaN
    o, l = orc.merge_attn_states(oa, np.array([-np.inf]), ob, np.array([-np.inf]))
    np.testing.assert_array_equal(o, [[0.0, 0.0]]); assert np.isneginf(l[0])
    # large LSE gap stays finite
    o, l = orc.merge_attn_states(oa, np.array([1000.0]), ob, np.array([-1000.0]))
    np.testing.assert_allclose(o, oa); assert l[0] == pytest.approx(1000.0)


# ----------------------------------------------------------------------------
# scatter and rotate (exact) against numpy routines
# ----------------------------------------------------------------------------

def test_scatter_matches_fancy_index_assignment():
    gen = torch.Generator().manual_seed(1)
    rng = np.random.default_rng(2)
    pages, P, H, D, T = 9, 32, 3, 8, 40
    k_pool = wl.randn_bf16((pages, P, H, D), gen)
    v_pool = wl.randn_bf16((pages, P, H, D), gen)
    src_k = wl.randn_bf16((T + 5, H, D), gen)
    src_v = wl.randn_bf16((T + 5, H, D), gen)
    slots = rng.choice(pages * P, size=2 * T, replace=False).astype(np.int64)
    s1, s2 = slots[:T].copy(), slots[T:].copy()
    s1[::7] = -1
    s2[1::3] = -1
    src_idx = rng.integers(0, T + 5, size=T).astype(np.int64)
    k_o, v_o, rej = orc.kv_scatter_slots(bits(src_k), bits(src_v), s1, bits(k_pool),
                                         bits(v_pool), slots2=s2, src_idx=src_idx)
    assert rej == 0
    for pool, src, out in ((k_pool, src_k, k_o), (v_pool, src_v, v_o)):
        ref = bits(pool).reshape(pages * P, H, D).copy()
        for dest in (s1, s2):
            ok = dest >= 0
            ref[dest[ok]] = bits(src)[src_idx[ok]]
        np.testing.assert_array_equal(out.reshape(pages * P, H, D), ref)


def test_scatter_checked_mode_rejects_out_of_range():
    pages, P, H, D = 2, 32, 1, 4
    pool = np.zeros((pages, P, H, D), dtype=np.uint16)
    src = np.arange(3 * H * D, dtype=np.uint16).reshape(3, H, D) + 1
    slots = np.array([5, 64, 70], dtype=np.int64)       # 64, 70 are past the pool
    k_o, _, rej = orc.kv_scatter_slots(src, src, slots, pool, pool, num_slots=pages * P)
    assert rej == 2
    assert (k_o.reshape(-1, H, D)[5] == src[0]).all()
    assert k_o.reshape(-1, H, D)[np.arange(64) != 5].sum() == 0


@pytest.mark.parametrize("elem", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("rows,cols,shift", [(3, 17, 5), (1, 12, 0), (2, 9, -4), (4, 7, 7),
                                             (2, 10, 23), (0, 5, 1), (3, 1, 1)])
def test_rotate_matches_numpy_roll(elem, rows, cols, shift):
    rng = np.random.default_rng(elem * 100 + cols)
    x = rng.integers(0, 256, size=(rows, cols, elem), dtype=np.uint8)
    out = orc.rotate_rows(x, shift)
    np.testing.assert_array_equal(out, np.roll(x, -shift, axis=1))


def test_rotate_three_reversal_identity():
    """Left rotation by s equals reversing the first s and the remaining
    elements, then reversing the whole row."""
    rng = np.random.default_rng(0)
    x = rng.integers(0, 256, size=(2, 23, 2), dtype=np.uint8)
    s = 9
    y = np.concatenate([x[:, :s][:, ::-1], x[:, s:][:, ::-1]], axis=1)[:, ::-1]
    np.testing.assert_array_equal(orc.rotate_rows(x, s), y)


# ----------------------------------------------------------------------------
# rotary embedding + paged write, slot copy
# ----------------------------------------------------------------------------

def _cos_sin_table(max_pos, D, base=10000.0):
    """cos/sin of angle pos * base^(-2i/D) for the D/2 pairs (the usual RoPE
    frequencies), as the caller-supplied table the kernel reads."""
    i = np.arange(D // 2)
    ang = np.arange(max_pos)[:, None] * base ** (-2.0 * i / D)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1), ang


def test_rope_matches_complex_multiplication():
    """Each pair (x_i, x_{i+D/2}) is the complex number x_i + j x_{i+D/2}
    multiplied by e^{j angle}: numpy complex arithmetic, a different
    formulation."""
    rng = np.random.default_rng(0)
    D = 16
    x = rng.standard_normal((5, 3, D))
    table, ang = _cos_sin_table(50, D)
    pos = np.array([0, 1, 7, 31, 49])
    out = orc.rope_rotate(x, table[pos, :D // 2][:, None], table[pos, D // 2:][:, None])
    z = (x[..., :D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * ang[pos])[:, None, :]
    np.testing.assert_allclose(out, np.concatenate([z.real, z.imag], axis=-1), rtol=1e-13, atol=1e-13)


def test_rope_identity_norm_and_composition():
    rng = np.random.default_rng(1)
    D = 8
    x = rng.standard_normal((4, D))
    table, ang = _cos_sin_table(20, D)
    h = D // 2
    # position 0: the identity
    np.testing.assert_allclose(orc.rope_rotate(x, table[0, :h], table[0, h:]), x, rtol=0, atol=1e-15)
    # every pair keeps its length
    y = orc.rope_rotate(x, table[13, :h], table[13, h:])
    np.testing.assert_allclose(x[:, :h] ** 2 + x[:, h:] ** 2, y[:, :h] ** 2 + y[:, h:] ** 2, rtol=1e-13)
    # rotating by 5 then by 8 equals rotating by 13
    z = orc.rope_rotate(orc.rope_rotate(x, table[5, :h], table[5, h:]), table[8, :h], table[8, h:])
    np.testing.assert_allclose(z, y, rtol=1e-12, atol=1e-13)


def test_rope_write_kv_paged_writes_v_exactly_and_skips_sentinels():
    gen = torch.Generator().manual_seed(2)
    T, Hq, Hkv, D, pages = 6, 4, 2, 16, 3
    q = wl.randn_bf16((T, Hq, D), gen)
    k = wl.randn_bf16((T, Hkv, D), gen)
    v = wl.randn_bf16((T, Hkv, D), gen)
    kp = wl.randn_bf16((pages, 32, Hkv, D), gen)
    vp = wl.randn_bf16((pages, 32, Hkv, D), gen)
    table, ang = _cos_sin_table(64, D)
    pos = np.array([3, 0, 63, 10, 11, 12])
    slots = np.array([5, 40, -1, 70, 2, 33], dtype=np.int64)
    q_rot, k_rot, k_out, v_out, written = orc.rope_write_kv_paged(q, k, v, pos, table, slots, kp, vp)
    ref_v = bits(vp).reshape(-1, Hkv, D).copy()
    ok = slots >= 0
    ref_v[slots[ok]] = bits(v)[ok]
    np.testing.assert_array_equal(v_out.reshape(-1, Hkv, D), ref_v)
    # token 1 sits at position 0: unrotated
    np.testing.assert_array_equal(q_rot[1], f64(q)[1])
    np.testing.assert_array_equal(k_rot[1], f64(k)[1])
    # the K pool: numpy fancy-index assignment of the rotated rows, each rotated
    # as complex numbers (a different formulation), every other slot unchanged
    z = (f64(k)[..., :D // 2] + 1j * f64(k)[..., D // 2:]) * np.exp(1j * ang[pos])[:, None, :]
    ref_k = f64(kp).reshape(-1, Hkv, D).copy()
    ref_k[slots[ok]] = np.concatenate([z.real, z.imag], axis=-1)[ok]
    np.testing.assert_allclose(k_out.reshape(-1, Hkv, D), ref_k, rtol=1e-13, atol=1e-13)
    ref_w = np.zeros(pages * 32, dtype=bool)
    ref_w[slots[ok]] = True
    np.testing.assert_array_equal(written.reshape(-1), ref_w)
    np.testing.assert_array_equal(k_out.reshape(-1, Hkv, D)[~ref_w], f64(kp).reshape(-1, Hkv, D)[~ref_w])


def test_rope_write_kv_paged_slot_placement_is_pinned():
    """Planted placement mistakes (the K row written at the previous slot, or
    the sentinel token written at slot 0) change the oracle's K pool: a
    distinct random row lands in every written slot, so the pool alone names
    where each rotated row went."""
    gen = torch.Generator().manual_seed(4)
    T, Hkv, D, pages = 5, 1, 8, 1
    k = wl.randn_bf16((T, Hkv, D), gen)
    kp = wl.randn_bf16((pages, 32, Hkv, D), gen)
    table, _ = _cos_sin_table(8, D)
    pos = np.zeros(T, dtype=np.int64)          # identity rotation: K rows copied exactly
    slots = np.array([7, -1, 3, 30, 12], dtype=np.int64)
    _, _, k_out, _, written = orc.rope_write_kv_paged(k.repeat(1, 2, 1), k, k, pos, table, slots, kp, kp)
    flat = k_out.reshape(-1, Hkv, D)
    for t, s_ in enumerate(slots):
        if s_ >= 0:
            np.testing.assert_array_equal(flat[s_], f64(k)[t])
            assert not np.array_equal(flat[s_ - 1], f64(k)[t])
    assert written.sum() == 4 and not written.reshape(-1)[0]
    np.testing.assert_array_equal(flat[0], f64(kp).reshape(-1, Hkv, D)[0])


def test_copy_kv_slots_matches_fancy_indexing_across_layers():
    gen = torch.Generator().manual_seed(3)
    layers, pages, H, D = 3, 4, 2, 8
    k = bits(wl.randn_bf16((layers, pages, 32, H, D), gen))
    v = bits(wl.randn_bf16((layers, pages, 32, H, D), gen))
    src = np.array([1, 5, -1, 40, 77, 9], dtype=np.int64)
    dst = np.array([100, 64, 3, -1, 90, 120], dtype=np.int64)
    k_o, v_o = orc.copy_kv_slots(k, v, src, dst)
    ok = (src >= 0) & (dst >= 0)
    for pool, out in ((k, k_o), (v, v_o)):
        ref = pool.reshape(layers, -1, H, D).copy()
        ref[:, dst[ok]] = pool.reshape(layers, -1, H, D)[:, src[ok]]
        np.testing.assert_array_equal(out.reshape(layers, -1, H, D), ref)
