"""CUDA-graph capture and replay of the entry points beside paged_attention:
kv_scatter_slots, rotate_rows, merge_attn_states, rope_write_kv_paged and
copy_kv_slots.  Each call is captured once, its device inputs are rewritten in
place, and the replay must compute on the new contents ([VG] Description,
Cache, "CUDA-graph safe" bullet: every kernel input lives in caller-owned
device memory and the host never reads the GPU back), checked against the fp64
oracle: bit-exact for the copies and the rotation, the merge within the bf16
rounding bound, the rotary write within the rotation bound."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)                      # first call outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    torch.cuda.synchronize()
    return g


def test_scatter_graph_replay_reads_new_slots_and_rows():
    gen = torch.Generator().manual_seed(40)
    rng = np.random.default_rng(40)
    pages, H, D, T = 12, 8, 128, 50
    k_pool = wl.randn_bf16((pages, 32, H, D), gen)
    v_pool = wl.randn_bf16((pages, 32, H, D), gen)
    kp, vp = k_pool.to(DEV), v_pool.to(DEV)
    ks, vs = torch.zeros(T, H, D, dtype=torch.bfloat16, device=DEV), torch.zeros(T, H, D, dtype=torch.bfloat16,
                                                                                  device=DEV)
    slots = torch.full((T,), -1, dtype=torch.int64, device=DEV)
    g = _capture(lambda s: pkv.kv_scatter_slots(ks, vs, slots, kp, vp, stream=s))
    kb, vb = orc.bf16_bits(k_pool), orc.bf16_bits(v_pool)
    for it in range(2):
        nk, nv = wl.randn_bf16((T, H, D), gen), wl.randn_bf16((T, H, D), gen)
        sl = rng.choice(pages * 32, size=T, replace=False).astype(np.int64)
        sl[it::5] = -1
        ks.copy_(nk)
        vs.copy_(nv)
        slots.copy_(torch.from_numpy(sl))
        g.replay()
        torch.cuda.synchronize()
        kb, vb, _ = orc.kv_scatter_slots(orc.bf16_bits(nk), orc.bf16_bits(nv), sl, kb, vb)
        np.testing.assert_array_equal(orc.bf16_bits(kp.cpu()), kb)
        np.testing.assert_array_equal(orc.bf16_bits(vp.cpu()), vb)


def test_rotate_graph_replay_rotates_current_contents():
    rows, cols, shift = 3, 1000, 123
    x = torch.zeros(rows, cols, dtype=torch.int32, device=DEV)
    g = _capture(lambda s: pkv.rotate_rows(x, shift, stream=s))
    rng = np.random.default_rng(41)
    for _ in range(2):
        data = rng.integers(-2 ** 31, 2 ** 31 - 1, size=(rows, cols), dtype=np.int64).astype(np.int32)
        x.copy_(torch.from_numpy(data))
        g.replay()
        torch.cuda.synchronize()
        want = orc.rotate_rows(data.view(np.uint8).reshape(rows, cols, 4), shift)
        np.testing.assert_array_equal(x.cpu().numpy().view(np.uint8).reshape(rows, cols, 4), want)


def test_merge_graph_replay_merges_new_states():
    rows, H, D = 40, 8, 128
    oa, ob = torch.zeros(rows, H, D, device=DEV), torch.zeros(rows, H, D, device=DEV)
    la, lb = torch.zeros(rows, H, device=DEV), torch.zeros(rows, H, device=DEV)
    out = torch.zeros(rows, H, D, dtype=torch.bfloat16, device=DEV)
    lo = torch.zeros(rows, H, device=DEV)
    g = _capture(lambda s: pkv.merge_attn_states(oa, la, ob, lb, out, lo, stream=s))
    gen = torch.Generator().manual_seed(42)
    for _ in range(2):
        a, b = torch.randn(rows, H, D, generator=gen), torch.randn(rows, H, D, generator=gen)
        a_l, b_l = 5 * torch.randn(rows, H, generator=gen), 5 * torch.randn(rows, H, generator=gen)
        a_l[0] = -float("inf")
        for t, v in ((oa, a), (ob, b), (la, a_l), (lb, b_l)):
            t.copy_(v)
        g.replay()
        torch.cuda.synchronize()
        O, L = orc.merge_attn_states(a.double().numpy(), a_l.double().numpy(), b.double().numpy(),
                                     b_l.double().numpy())
        got = out.double().cpu().numpy()
        assert (np.abs(got - O) <= 2.0 ** -8 * np.abs(O) + 1e-5).all()
        assert np.abs(lo.double().cpu().numpy() - L).max() <= 1e-5


def test_rope_write_graph_replay_uses_new_positions_and_slots():
    gen = torch.Generator().manual_seed(43)
    rng = np.random.default_rng(43)
    T, Hq, Hkv, D, pages, max_pos = 24, 16, 4, 128, 6, 4096
    i = np.arange(D // 2)
    ang = np.arange(max_pos)[:, None] * 10000.0 ** (-2.0 * i / D)[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    k_pool = wl.randn_bf16((pages, 32, Hkv, D), gen)
    v_pool = wl.randn_bf16((pages, 32, Hkv, D), gen)
    kp, vp = k_pool.to(DEV), v_pool.to(DEV)
    q = torch.zeros(T, Hq, D, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(T, Hkv, D, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(T, Hkv, D, dtype=torch.bfloat16, device=DEV)
    pos = torch.zeros(T, dtype=torch.int64, device=DEV)
    slots = torch.full((T,), -1, dtype=torch.int64, device=DEV)
    tab = torch.from_numpy(table).to(DEV)
    g = _capture(lambda s: pkv.rope_write_kv_paged(q, k, v, pos, tab, slots, kp, vp, stream=s))
    kpool_now, vpool_now = kp.cpu().clone(), vp.cpu().clone()
    for _ in range(2):
        nq, nk, nv = (wl.randn_bf16((T, Hq, D), gen), wl.randn_bf16((T, Hkv, D), gen),
                      wl.randn_bf16((T, Hkv, D), gen))
        p_ = rng.integers(0, max_pos, size=T).astype(np.int64)
        sl = rng.choice(pages * 32, size=T, replace=False).astype(np.int64)
        sl[::6] = -1
        for t, val in ((q, nq), (k, nk), (v, nv), (pos, torch.from_numpy(p_)), (slots, torch.from_numpy(sl))):
            t.copy_(val)
        g.replay()
        torch.cuda.synchronize()
        q_rot, _, k_ref, v_ref, written = orc.rope_write_kv_paged(nq, nk, nv, p_, table, sl, kpool_now, vpool_now)
        rq = q_rot
        h = D // 2
        bound_q = 2.0 ** -8 * np.sqrt(2.0) * np.concatenate(
            [np.hypot(rq[..., :h], rq[..., h:])] * 2, axis=-1) + 1e-30
        assert (np.abs(q.double().cpu().numpy() - q_rot) <= bound_q * (1 + 1e-12)).all()
        rk = k_ref[written]
        bound_k = 2.0 ** -8 * np.sqrt(2.0) * np.concatenate([np.hypot(rk[..., :h], rk[..., h:])] * 2, axis=-1)
        assert (np.abs(kp.double().cpu().numpy()[written] - rk) <= bound_k * (1 + 1e-12) + 1e-30).all()
        np.testing.assert_array_equal(orc.bf16_bits(vp.cpu()), v_ref)
        kpool_now, vpool_now = kp.cpu().clone(), vp.cpu().clone()


def test_copy_slots_graph_replay_copies_new_lists():
    gen = torch.Generator().manual_seed(44)
    rng = np.random.default_rng(44)
    layers, pages, H, D, n = 3, 8, 8, 128, 40
    k = wl.randn_bf16((layers, pages, 32, H, D), gen)
    v = wl.randn_bf16((layers, pages, 32, H, D), gen)
    kg, vg = k.to(DEV), v.to(DEV)
    src = torch.full((n,), -1, dtype=torch.int64, device=DEV)
    dst = torch.full((n,), -1, dtype=torch.int64, device=DEV)
    g = _capture(lambda s: pkv.copy_kv_slots(kg, vg, src, dst, stream=s))
    kb, vb = orc.bf16_bits(k), orc.bf16_bits(v)
    for it in range(2):
        perm = rng.permutation(pages * 32)
        s_, d_ = perm[:n].astype(np.int64), perm[n:2 * n].astype(np.int64)
        s_[it::7] = -1
        src.copy_(torch.from_numpy(s_))
        dst.copy_(torch.from_numpy(d_))
        g.replay()
        torch.cuda.synchronize()
        kb, vb = orc.copy_kv_slots(kb, vb, s_, d_)
        np.testing.assert_array_equal(orc.bf16_bits(kg.cpu()), kb)
        np.testing.assert_array_equal(orc.bf16_bits(vg.cpu()), vb)
