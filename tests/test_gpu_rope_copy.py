"""GPU parity of rope_write_kv_paged (rotary embedding of Q in place, rotated
K and V written to pool slots) and copy_kv_slots (slot rows copied across
layers), through the C-ABI, against the fp64 oracle.

Rotation tolerance: the device rotates in fp32 and rounds to bf16, so each
output may differ from the exact rotation by half a bf16 ulp of the result
plus the fp32 error of the two products: |got - exact| <= 2^-8 * (|x1 cos| +
|x2 sin|) + 1e-30.  V rows, untouched pool rows and the slot copy: bit-exact."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def cos_sin_table(max_pos, D, base=10000.0):
    i = np.arange(D // 2)
    ang = np.arange(max_pos)[:, None] * base ** (-2.0 * i / D)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def rot_bound(x, table, pos):
    """Per-element error bound of the rotated values (see the module docstring)."""
    D = x.shape[-1]
    h = D // 2
    c = table[pos, :h].astype(np.float64)[:, None, :]
    s = table[pos, h:].astype(np.float64)[:, None, :]
    x1, x2 = x[..., :h], x[..., h:]
    mag = np.concatenate([np.abs(x1 * c) + np.abs(x2 * s), np.abs(x2 * c) + np.abs(x1 * s)], axis=-1)
    return 2.0 ** -8 * mag + 1e-30


def pair_bound(rot):
    """Error bound of rotated values from the exact rotation itself: each pair
    keeps its length r, and |x1 cos| + |x2 sin| <= sqrt(2) r, so the module
    docstring's bound is at most 2^-8 sqrt(2) r for both members of a pair."""
    h = rot.shape[-1] // 2
    r = np.sqrt(rot[..., :h] ** 2 + rot[..., h:] ** 2)
    return 2.0 ** -8 * np.sqrt(2.0) * np.concatenate([r, r], axis=-1) * (1 + 1e-12) + 1e-30


def bf16_bits_of_f64(x):
    """bf16 bit patterns of float64 values that are exactly bf16."""
    b = np.asarray(x).astype(np.float32).view(np.uint32)
    assert (b & 0xFFFF == 0).all()
    return (b >> 16).astype(np.uint16)


@pytest.mark.parametrize("T,Hq,Hkv,D", [(37, 32, 8, 128), (5, 4, 2, 64), (200, 40, 40, 128),
                                        (64, 16, 2, 128)])
def test_rope_write_kv_paged(T, Hq, Hkv, D):
    gen = torch.Generator().manual_seed(T)
    rng = np.random.default_rng(T)
    pages = (2 * T) // 32 + 3
    max_pos = 20000
    q = wl.randn_bf16((T, Hq, D), gen)
    # K / V sliced from a fused QKV tensor, as the pages' callers do
    qkv = wl.randn_bf16((T, Hq + 2 * Hkv, D), gen)
    k_src, v_src = qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    k_pool = wl.randn_bf16((pages, 32, Hkv, D), gen)
    v_pool = wl.randn_bf16((pages, 32, Hkv, D), gen)
    pos = rng.integers(0, max_pos, size=T).astype(np.int64)
    pos[0] = 0
    pos[-1] = max_pos - 1
    slots = rng.choice(pages * 32, size=T, replace=False).astype(np.int64)
    slots[1::7] = -1
    table = cos_sin_table(max_pos, D)
    qg, kp, vp = q.to(DEV), k_pool.to(DEV), v_pool.to(DEV)
    qkvg = qkv.to(DEV)
    pkv.rope_write_kv_paged(qg, qkvg[:, Hq:Hq + Hkv], qkvg[:, Hq + Hkv:], torch.from_numpy(pos).to(DEV),
                            torch.from_numpy(table).to(DEV), torch.from_numpy(slots).to(DEV), kp, vp)
    torch.cuda.synchronize()
    q_rot, _, k_ref, v_ref, written = orc.rope_write_kv_paged(q, k_src.contiguous(), v_src.contiguous(),
                                                              pos, table, slots, k_pool, v_pool)
    got_q = qg.double().cpu().numpy()
    assert (np.abs(got_q - q_rot) <= rot_bound(orc.bf16_to_f64(orc.bf16_bits(q)), table, pos)).all()
    # the whole K pool against the oracle's: slots the oracle wrote within the
    # rotation bound, every other slot bit-exact
    got_k = kp.double().cpu().numpy()
    assert (np.abs(got_k[written] - k_ref[written]) <= pair_bound(k_ref[written])).all()
    np.testing.assert_array_equal(orc.bf16_bits(kp.cpu())[~written], bf16_bits_of_f64(k_ref[~written]))
    np.testing.assert_array_equal(orc.bf16_bits(vp.cpu()), v_ref)
    # the fused QKV source is not modified
    assert torch.equal(qkvg.cpu(), qkv)


def test_rope_position_zero_is_exact_copy():
    """At position 0 (cos 1, sin 0) the rotation is the identity, bit for bit."""
    gen = torch.Generator().manual_seed(1)
    T, Hq, Hkv, D = 9, 8, 2, 128
    q = wl.randn_bf16((T, Hq, D), gen)
    k = wl.randn_bf16((T, Hkv, D), gen)
    v = wl.randn_bf16((T, Hkv, D), gen)
    pools = [torch.zeros(2, 32, Hkv, D, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    table = torch.from_numpy(cos_sin_table(4, D)).to(DEV)
    slots = torch.arange(T, dtype=torch.int64, device=DEV) * 3
    qg = q.to(DEV)
    pkv.rope_write_kv_paged(qg, k.to(DEV), v.to(DEV), torch.zeros(T, dtype=torch.int64, device=DEV),
                            table, slots, pools[0], pools[1])
    assert torch.equal(qg.cpu(), q)
    assert torch.equal(pools[0].view(-1, Hkv, D)[slots.cpu()].cpu(), k)
    assert torch.equal(pools[1].view(-1, Hkv, D)[slots.cpu()].cpu(), v)


def test_rope_checked_mode_flags_bad_position_and_slot():
    D = 64
    q = torch.zeros(2, 2, D, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(2, 1, D, dtype=torch.bfloat16, device=DEV)
    pools = [torch.zeros(1, 32, 1, D, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    table = torch.from_numpy(cos_sin_table(8, D)).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.rope_write_kv_paged(q, k, k, torch.tensor([3, 99], dtype=torch.int64, device=DEV), table,
                            torch.tensor([1, 500], dtype=torch.int64, device=DEV), pools[0], pools[1],
                            checked=True, err=err)
    e = int(err.item())
    assert e & pkv.PKV_ERRBIT_LEN and e & pkv.PKV_ERRBIT_SLOT


@pytest.mark.parametrize("layers,H,D", [(1, 8, 128), (4, 2, 64), (3, 40, 128)])
def test_copy_kv_slots_across_layers(layers, H, D):
    gen = torch.Generator().manual_seed(layers * H)
    rng = np.random.default_rng(layers)
    pages = 6
    k = wl.randn_bf16((layers, pages, 32, H, D), gen)
    v = wl.randn_bf16((layers, pages, 32, H, D), gen)
    perm = rng.permutation(pages * 32)
    n = 50
    src, dst = perm[:n].astype(np.int64), perm[n:2 * n].astype(np.int64)
    src[::9] = -1
    dst[4::11] = -1
    kg, vg = k.to(DEV), v.to(DEV)
    pkv.copy_kv_slots(kg, vg, torch.from_numpy(src).to(DEV), torch.from_numpy(dst).to(DEV))
    torch.cuda.synchronize()
    ko, vo = orc.copy_kv_slots(orc.bf16_bits(k), orc.bf16_bits(v), src, dst)
    np.testing.assert_array_equal(orc.bf16_bits(kg.cpu()), ko)
    np.testing.assert_array_equal(orc.bf16_bits(vg.cpu()), vo)


def test_copy_kv_slots_checked_mode():
    k = torch.zeros(1, 2, 32, 1, 64, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.copy_kv_slots(k, k.clone(), torch.tensor([3, 1000], dtype=torch.int64, device=DEV),
                      torch.tensor([4, 5], dtype=torch.int64, device=DEV), checked=True, err=err)
    assert int(err.item()) & pkv.PKV_ERRBIT_SLOT
