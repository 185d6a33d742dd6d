"""Pins of the oracle's exact-window layout (CPU only).

* the hand-derived fixture tests/golden/causal_layout_small.txt (layout fields
  and visible sets of two small geometries);
* structural properties on random geometries, checked from the layout's
  outputs alone: each row reads exactly its block's visible set, no key
  twice, the block's own tokens last and in order;
* attention through the layout (commit copies, the forward's two scatters, one
  unmasked ragged attention over all blocks) equals dense attention over the
  exact window computed directly from the logical sequence, and the pages'
  own check: q = 0 with one-hot V returns 1/|visible| exactly on the visible
  keys.
"""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "causal_layout_small.txt")


def _ranges(tokens):
    out = []
    for t in tokens:
        a, _, b = t.partition("-")
        out.extend(range(int(a), int(b or a) + 1))
    return out


def load_golden():
    cases = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, _, rest = line.partition(" ")
        if key == "geometry":
            g = dict(kv.split("=") for kv in rest.split())
            cases.append(dict(geom={k: int(v) for k, v in g.items()}, private={}, visible={},
                              rows={}, committed=[], current=[]))
            continue
        c = cases[-1]
        if key in ("private", "visible", "row"):
            k, _, vals = rest.partition(":")
            vals = vals.split()
            target = {"private": c["private"], "visible": c["visible"], "row": c["rows"]}[key]
            target[int(k)] = _ranges(vals) if key == "visible" else [int(v) for v in vals]
        elif key in ("committed", "current"):
            c[key] = [tuple(int(x) for x in e.split(":")) for e in rest.split()]
        else:
            c[key] = [int(v) for v in rest.split()]
    return cases


@pytest.mark.parametrize("ci", [0, 1])
def test_causal_layout_golden(ci):
    c = load_golden()[ci]
    g = c["geom"]
    nb = len(c["private"])
    for k in range(nb):
        assert orc.exact_window_keys(g["pin"], g["committed"], g["window"], g["staged"], g["block"], k) \
            == c["visible"][k]
    L = orc.causal_layout(c["table"], g["pin"], g["committed"], g["window"], g["staged"], g["block"],
                          [c["private"][k] for k in range(nb)], page_size=g["page"])
    assert L["rows"] == [c["rows"][k] for k in range(nb)]
    assert L["kv_lens"] == c["kv_lens"]
    assert L["q_indptr"] == c["q_indptr"]
    assert L["staged_slots"] == c["staged_slots"]
    assert L["staged_slots2"] == c["staged_slots2"]
    assert L["committed"] == c["committed"]
    assert L["current"] == c["current"]


def random_geometry(rng, page):
    pin = int(rng.integers(0, 4 * page))
    committed = int(rng.integers(0, 12 * page))
    window = int(rng.integers(0, 10 * page))
    staged = int(rng.integers(1, 6 * page))
    block = int(rng.integers(1, staged + 1))
    total = pin + committed + staged
    n_log = (total + page - 1) // page
    nb = len(orc.causal_blocks(staged, block))
    cap = (3 * (page - 1) + block + page - 1) // page + 1
    n_phys = n_log + nb * cap + 5
    perm = rng.permutation(n_phys)
    table = perm[:n_log].tolist()
    private = perm[n_log:n_log + nb * cap].reshape(nb, cap).tolist()
    return dict(pin=pin, committed=committed, window=window, staged=staged, block=block,
                table=table, private=private, n_phys=n_phys)


def row_positions(L, g, k, page):
    """Logical position behind every key of row k, from the layout's outputs:
    sequence slots map back through the table, private slots through whichever
    copy or write fills them."""
    base = g["pin"] + g["committed"]
    seq_slot = {}
    for lp, phys in enumerate(g["table"]):
        for o in range(page):
            seq_slot[phys * page + o] = lp * page + o
    filled = {}
    for src, dst in L["committed"]:
        assert dst not in filled
        filled[dst] = seq_slot[src]
    for t_idx, dst in L["current"]:
        assert dst not in filled
        filled[dst] = base + t_idx
    for t_idx, dst in enumerate(L["staged_slots2"]):
        if dst >= 0:
            assert dst not in filled
            filled[dst] = base + t_idx
    out = []
    for j in range(L["kv_lens"][k]):
        s = L["rows"][k][j // page] * page + j % page
        out.append(filled[s] if s in filled else seq_slot[s])
    return out


@pytest.mark.parametrize("page", [4, 8, 32])
@pytest.mark.parametrize("seed", range(6))
def test_causal_layout_reads_exactly_the_window(page, seed):
    rng = np.random.default_rng(1000 * page + seed)
    g = random_geometry(rng, page)
    L = orc.causal_layout(g["table"], g["pin"], g["committed"], g["window"], g["staged"], g["block"],
                          g["private"], page_size=page)
    base = g["pin"] + g["committed"]
    blocks = orc.causal_blocks(g["staged"], g["block"])
    assert L["staged_slots"] == [g["table"][(base + t) // page] * page + (base + t) % page
                                 for t in range(g["staged"])]
    for k, (first, n) in enumerate(blocks):
        pos = row_positions(L, g, k, page)
        vis = orc.exact_window_keys(g["pin"], g["committed"], g["window"], g["staged"], g["block"], k)
        assert len(pos) == len(set(pos))                  # no key twice
        assert sorted(pos) == sorted(vis)                  # exactly the window
        assert pos[-n:] == list(range(base + first, base + first + n))  # own tokens last
        # closed form of the window's size
        s = base + first
        assert len(vis) == g["pin"] + min(g["window"], s - g["pin"]) + n
    # every staged token has its private copy in its own block's row
    assert all(x >= 0 for x in L["staged_slots2"])


def _bits(x):
    return orc.bf16_bits(torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16))


@pytest.mark.parametrize("seed", range(3))
def test_attention_through_layout_equals_exact_window(seed):
    rng = np.random.default_rng(77 + seed)
    page = 32
    g = random_geometry(rng, page)
    H, D, Hq = 2, 64, 4
    total = g["pin"] + g["committed"] + g["staged"]
    base = g["pin"] + g["committed"]
    K = _bits(rng.standard_normal((total, H, D)))
    V = _bits(rng.standard_normal((total, H, D)))
    q = _bits(rng.standard_normal((g["staged"], Hq, D)))
    L = orc.causal_layout(g["table"], g["pin"], g["committed"], g["window"], g["staged"], g["block"],
                          g["private"], page_size=page)
    k_pool = np.zeros((g["n_phys"], page, H, D), np.uint16)
    v_pool = np.zeros_like(k_pool)
    for p in range(base):  # the committed sequence already sits in its slots
        s = g["table"][p // page] * page + p % page
        k_pool[s // page, s % page] = K[p]
        v_pool[s // page, s % page] = V[p]
    # commit: committed private copies
    src = [a for a, _ in L["committed"]]
    dst = [b for _, b in L["committed"]]
    k5, v5 = orc.copy_kv_slots(k_pool[None], v_pool[None], src, dst)
    k_pool, v_pool = k5[0], v5[0]
    # forward: staged rows to their own slots and own private slots, then the
    # earlier blocks' tokens to the later blocks' private pages
    k_pool, v_pool, _ = orc.kv_scatter_slots(K[base:], V[base:], L["staged_slots"], k_pool, v_pool,
                                          slots2=L["staged_slots2"])
    if L["current"]:
        k_pool, v_pool, _ = orc.kv_scatter_slots(K[base:], V[base:], [d for _, d in L["current"]], k_pool,
                                              v_pool, src_idx=[t for t, _ in L["current"]])
    nb = len(L["rows"])
    width = max(len(r) for r in L["rows"])
    table = np.full((nb, width), -1, np.int64)
    for k, r in enumerate(L["rows"]):
        table[k, :len(r)] = r
    O, LSE = orc.paged_attention(q, k_pool, v_pool, table, np.array(L["kv_lens"]),
                                 np.array(L["q_indptr"]), mask=orc.MASK_NONE)
    # dense attention over the exact window, straight from the logical sequence
    Kf, Vf, qf = orc.bf16_to_f64(K), orc.bf16_to_f64(V), orc.bf16_to_f64(q)
    scale = 1.0 / np.sqrt(D)
    for k, (first, n) in enumerate(orc.causal_blocks(g["staged"], g["block"])):
        vis = np.array(orc.exact_window_keys(g["pin"], g["committed"], g["window"], g["staged"],
                                             g["block"], k))
        for t in range(first, first + n):
            for h in range(Hq):
                s = scale * Kf[vis, h // (Hq // H)] @ qf[t, h]
                m = s.max()
                w = np.exp(s - m)
                np.testing.assert_allclose(O[t, h], w @ Vf[vis, h // (Hq // H)] / w.sum(), rtol=1e-12,
                                           atol=1e-12)
                np.testing.assert_allclose(LSE[t, h], m + np.log(w.sum()), rtol=1e-12, atol=1e-12)


def test_zero_query_one_hot_values_through_layout():
    """q = 0 gives uniform weights; V row of logical position p is e_p, so
    O[p] = 1/|window| exactly on the visible positions (the pages' visible-key
    check, with the window full and filling)."""
    page = 32
    for committed, window in ((20, 100), (150, 64)):
        pin, staged, block = 40, 50, 17
        total = pin + committed + staged
        base = pin + committed
        n_log = (total + page - 1) // page
        nb = len(orc.causal_blocks(staged, block))
        table = list(range(n_log))
        private = [[n_log + 4 * k + j for j in range(4)] for k in range(nb)]
        D = total if total % 2 == 0 else total + 1
        K = np.zeros((total, 1, D), np.uint16)
        V = _bits(np.eye(total, D)[:, None, :])
        q = np.zeros((staged, 1, D), np.uint16)
        L = orc.causal_layout(table, pin, committed, window, staged, block, private, page_size=page)
        k_pool = np.zeros((n_log + 4 * nb, page, 1, D), np.uint16)
        v_pool = np.zeros_like(k_pool)
        for p in range(base):
            v_pool[p // page, p % page] = V[p]
        k5, v5 = orc.copy_kv_slots(k_pool[None], v_pool[None], [a for a, _ in L["committed"]],
                                   [b for _, b in L["committed"]])
        k_pool, v_pool, _ = orc.kv_scatter_slots(K[base:], V[base:], L["staged_slots"], k5[0], v5[0],
                                              slots2=L["staged_slots2"])
        if L["current"]:
            k_pool, v_pool, _ = orc.kv_scatter_slots(K[base:], V[base:], [d for _, d in L["current"]], k_pool,
                                                  v_pool, src_idx=[t for t, _ in L["current"]])
        width = max(len(r) for r in L["rows"])
        table2 = np.full((nb, width), -1, np.int64)
        for k, r in enumerate(L["rows"]):
            table2[k, :len(r)] = r
        O, LSE = orc.paged_attention(q, k_pool, v_pool, table2, np.array(L["kv_lens"]),
                                     np.array(L["q_indptr"]), mask=orc.MASK_NONE)
        for k, (first, n) in enumerate(orc.causal_blocks(staged, block)):
            s = base + first
            vis = set(range(pin)) | set(range(max(pin, s - window), s + n))
            want = np.zeros(D)
            want[sorted(vis)] = 1.0 / len(vis)
            for t in range(first, first + n):
                np.testing.assert_allclose(O[t, 0], want, atol=1e-15)
                assert abs(LSE[t, 0] - np.log(len(vis))) < 1e-12


def test_exact_window_equals_block_causal_when_window_cuts_nothing():
    """With a window reaching back to the fixed region for every block, the
    exact window is the block-causal visible set over the whole sequence, so
    the direct definition must equal the paged oracle with the block-causal
    mask (itself pinned to torch SDPA)."""
    rng = np.random.default_rng(5)
    pin, committed, staged, block, H, Hq, D = 37, 90, 70, 24, 2, 4, 64
    total = pin + committed + staged
    window = committed + staged
    K = _bits(rng.standard_normal((total, H, D)))
    V = _bits(rng.standard_normal((total, H, D)))
    q = _bits(rng.standard_normal((staged, Hq, D)))
    O1, L1 = orc.exact_window_attention(q, K, V, pin, committed, window, staged, block)
    P = 32
    n_pages = (total + P - 1) // P
    kp = np.zeros((n_pages, P, H, D), np.uint16)
    vp = np.zeros_like(kp)
    for p in range(total):
        kp[p // P, p % P] = K[p]
        vp[p // P, p % P] = V[p]
    O2, L2 = orc.paged_attention(q, kp, vp, np.arange(n_pages)[None], np.array([total]),
                                 np.array([0, staged]), q_real=np.array([staged]),
                                 mask=orc.MASK_BLOCK_CAUSAL, causal_block=block)
    np.testing.assert_allclose(O1, O2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=1e-12, atol=1e-12)
