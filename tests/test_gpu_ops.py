"""GPU parity of the exact ops (scatter, rotate) and of the LSE merge, called
through the C-ABI, against the fp64 oracle: bit-exact for scatter / rotate,
within the attention tolerances for the merge."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t):
    return orc.bf16_bits(t.cpu()) if t.dtype == torch.bfloat16 else t.cpu().numpy()


# ------------------------------------------------------------------ scatter
@pytest.mark.parametrize("H,D,T,with2,with_idx", [(2, 64, 2, False, False), (8, 128, 64, False, False),
                                                  (8, 128, 300, True, True), (40, 128, 1568, False, False),
                                                  (3, 24, 17, True, False)])
def test_scatter_bit_exact(H, D, T, with2, with_idx):
    gen = torch.Generator().manual_seed(T + H)
    rng = np.random.default_rng(T)
    pages = (2 * T) // 32 + 4
    k_pool = wl.randn_bf16((pages, 32, H, D), gen)
    v_pool = wl.randn_bf16((pages, 32, H, D), gen)
    src_rows = T + 3
    k_src = wl.randn_bf16((src_rows, H, D), gen)
    v_src = wl.randn_bf16((src_rows, H, D), gen)
    slots_all = rng.choice(pages * 32, size=2 * T, replace=False).astype(np.int64)
    s1 = slots_all[:T].copy()
    s1[::5] = -1
    s2 = slots_all[T:].copy() if with2 else None
    idx = rng.integers(0, src_rows, size=T).astype(np.int64) if with_idx else None
    kg, vg = k_pool.to(DEV), v_pool.to(DEV)
    pkv.kv_scatter_slots(k_src.to(DEV), v_src.to(DEV), torch.from_numpy(s1).to(DEV), kg, vg,
                         slots2=None if s2 is None else torch.from_numpy(s2).to(DEV),
                         src_idx=None if idx is None else torch.from_numpy(idx).to(DEV))
    ko, vo, _ = orc.kv_scatter_slots(bits(k_src), bits(v_src), s1, bits(k_pool), bits(v_pool),
                                     slots2=s2, src_idx=idx)
    np.testing.assert_array_equal(bits(kg), ko)
    np.testing.assert_array_equal(bits(vg), vo)


def test_scatter_strided_source_from_fused_qkv():
    """K/V sliced out of a fused QKV tensor [T, Hq + 2 Hkv, D] without a copy."""
    gen = torch.Generator().manual_seed(3)
    T, Hq, Hkv, D = 50, 8, 2, 128
    qkv = wl.randn_bf16((T, Hq + 2 * Hkv, D), gen).to(DEV)
    k_src, v_src = qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    pages = 4
    k_pool = torch.zeros(pages, 32, Hkv, D, dtype=torch.bfloat16, device=DEV)
    v_pool = torch.zeros_like(k_pool)
    slots = torch.randperm(pages * 32, generator=gen)[:T].to(torch.int64)
    pkv.kv_scatter_slots(k_src, v_src, slots.to(DEV), k_pool, v_pool)
    ko, vo, _ = orc.kv_scatter_slots(bits(k_src.contiguous()), bits(v_src.contiguous()),
                                     slots.numpy(), bits(torch.zeros(pages, 32, Hkv, D, dtype=torch.bfloat16)),
                                     bits(torch.zeros(pages, 32, Hkv, D, dtype=torch.bfloat16)))
    np.testing.assert_array_equal(bits(k_pool), ko)
    np.testing.assert_array_equal(bits(v_pool), vo)


def test_scatter_interleaved_kv_pool_page_stride():
    """K and V pages interleaved in one allocation: page stride = 2 pages."""
    gen = torch.Generator().manual_seed(4)
    pages, H, D, T = 6, 4, 64, 40
    both = torch.zeros(pages, 2, 32, H, D, dtype=torch.bfloat16, device=DEV)
    k_pool, v_pool = both[:, 0], both[:, 1]
    k_src = wl.randn_bf16((T, H, D), gen)
    v_src = wl.randn_bf16((T, H, D), gen)
    slots = torch.randperm(pages * 32, generator=gen)[:T].to(torch.int64)
    pkv.kv_scatter_slots(k_src.to(DEV), v_src.to(DEV), slots.to(DEV), k_pool, v_pool)
    z = bits(torch.zeros(pages, 32, H, D, dtype=torch.bfloat16))
    ko, vo, _ = orc.kv_scatter_slots(bits(k_src), bits(v_src), slots.numpy(), z, z)
    np.testing.assert_array_equal(bits(k_pool.contiguous()), ko)
    np.testing.assert_array_equal(bits(v_pool.contiguous()), vo)


def test_scatter_checked_mode_flags_out_of_range():
    pages, H, D = 2, 1, 64
    k_pool = torch.zeros(pages, 32, H, D, dtype=torch.bfloat16, device=DEV)
    v_pool = torch.zeros_like(k_pool)
    src = torch.ones(3, H, D, dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([5, 64, 1 << 40], dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.kv_scatter_slots(src, src, slots, k_pool, v_pool, checked=True, err=err)
    assert err.item() & pkv.PKV_ERRBIT_SLOT
    assert k_pool.view(-1, H, D)[5].float().sum().item() == D
    assert k_pool.float().sum().item() == D


def test_scatter_empty_is_noop():
    k_pool = torch.zeros(1, 32, 1, 64, dtype=torch.bfloat16, device=DEV)
    src = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device=DEV)
    pkv.kv_scatter_slots(src, src, torch.zeros(0, dtype=torch.int64, device=DEV), k_pool, k_pool)


# ------------------------------------------------------------------ rotate
@pytest.mark.parametrize("dtype,rows,cols,shift", [
    (torch.uint8, 3, 1001, 17), (torch.int16, 5, 999, -300), (torch.int32, 2, 4096, 1024),
    (torch.int64, 7, 513, 512), (torch.int16, 1, 100000, 33333), (torch.int32, 3, 65536, 1),
    (torch.int16, 2, 12, 12), (torch.uint8, 4, 1, 3), (torch.int32, 1, 3993600, 998400),
    (torch.int64, 300, 640, 160)])
def test_rotate_bit_exact(dtype, rows, cols, shift):
    g = torch.Generator().manual_seed(cols)
    x = torch.randint(-100, 100, (rows, cols + 5), generator=g).to(dtype)
    xg = x.to(DEV)
    pkv.rotate_rows(xg, shift, rows=rows, cols=cols, row_stride=cols + 5, elem_size=x.element_size())
    e = x.element_size()
    view = x.numpy().view(np.uint8).reshape(rows, cols + 5, e)
    ref = view.copy()
    ref[:, :cols] = orc.rotate_rows(view[:, :cols], shift)
    np.testing.assert_array_equal(xg.cpu().numpy().view(np.uint8).reshape(rows, cols + 5, e), ref)


def test_rotate_16_byte_elements_and_video_region():
    """The video workload's rolling region: 4 blocks of 1560 tokens x 40 heads
    x 128 bf16, rotated left by one block, in 16-byte elements."""
    block = 1560 * 40 * 128
    g = torch.Generator().manual_seed(5)
    x = wl.randn_bf16((4 * block,), g)
    xg = x.to(DEV)
    pkv.rotate_rows(xg.view(torch.uint8), block * 2 // 16, rows=1, cols=4 * block * 2 // 16,
                    row_stride=4 * block * 2 // 16, elem_size=16)
    ref = torch.cat([x[block:], x[:block]])
    assert torch.equal(xg.cpu(), ref)


# ------------------------------------------------------------------ merge
@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.float32, torch.bfloat16),
                                                (torch.float32, torch.float32),
                                                (torch.bfloat16, torch.bfloat16)])
def test_merge_matches_oracle(in_dtype, out_dtype):
    g = torch.Generator().manual_seed(8)
    rows, H, D = 37, 8, 128
    oa = torch.randn(rows, H, D, generator=g).to(in_dtype)
    ob = torch.randn(rows, H, D, generator=g).to(in_dtype)
    la = torch.randn(rows, H, generator=g) * 4
    lb = torch.randn(rows, H, generator=g) * 4
    la[0, :3] = -math.inf
    lb[0, 1:4] = -math.inf
    lb[1] = la[1] + 200.0
    out = torch.empty(rows, H, D, dtype=out_dtype, device=DEV)
    lout = torch.empty(rows, H, device=DEV)
    pkv.merge_attn_states(oa.to(DEV), la.to(DEV), ob.to(DEV), lb.to(DEV), out, lout)
    O, L = orc.merge_attn_states(oa.double().numpy(), la.double().numpy(), ob.double().numpy(),
                                 lb.double().numpy())
    got = out.double().cpu().numpy()
    # bf16 rounding of the output: half an ulp is 2^-9 relative; f32: 1e-5
    rel = 2.0 ** -8 if out_dtype == torch.bfloat16 else 1e-6
    assert (np.abs(got - O) <= rel * np.abs(O) + 1e-5).all()
    gl = lout.double().cpu().numpy()
    fin = np.isfinite(L)
    assert np.abs(gl[fin] - L[fin]).max() <= 1e-5
    assert np.isneginf(gl[~fin]).all()
    assert (got[~fin] == 0).all()


def test_merge_in_place_into_first_state():
    g = torch.Generator().manual_seed(9)
    rows, H, D = 5, 4, 64
    oa = torch.randn(rows, H, D, generator=g)
    ob = torch.randn(rows, H, D, generator=g)
    la = torch.randn(rows, H, generator=g)
    lb = torch.randn(rows, H, generator=g)
    O, L = orc.merge_attn_states(oa.double().numpy(), la.double().numpy(), ob.double().numpy(),
                                 lb.double().numpy())
    oag, lag = oa.to(DEV), la.to(DEV)
    pkv.merge_attn_states(oag, lag, ob.to(DEV), lb.to(DEV), oag, lag)
    assert np.abs(oag.double().cpu().numpy() - O).max() < 1e-5
    assert np.abs(lag.double().cpu().numpy() - L).max() < 1e-5
