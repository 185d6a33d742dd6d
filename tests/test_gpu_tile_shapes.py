"""Tensor-core tiles for head_dim 64 and for head groups beyond powers of two.

The tile kernels take head_dim 64 or 128 and any head group G = Hq / Hkv up to
64 ([VG] Description, Attention: grouped-query heads over 32-token pages): a
128-row tile packs floor(128 / G) tokens x G heads and leaves the remaining
lanes empty.  Checked against the fp64 oracle (max-abs 1e-2, mean-abs 1e-3 on
bf16 outputs, LSE 1e-3; padding rows zero) through every path the plan picks:
the two-tile kernel (rows beyond one tile), the one-tile kernel with rows held
four times (rows x G <= 32) or once, key splits and their merge, single-row
decode with groups the decode kernel does not take, the one-launch grouped
shared-prefix path, and the stream-K schedule.  Peaked queries guard the
visibility boundaries; their outputs come back in f32, since a peaked row's
output approaches one V value (|v| up to ~4), where half a bf16 ulp alone is
above the 1e-2 bound."""
import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl

from pkv_testutil import assert_attention_close, gpu_step, oracle_step
from test_gpu_plan import fused_step

pytestmark = pytest.mark.gpu


def _run(case, kernel=pkv.PKV_KERNEL_TILE, **kw):
    plan = pkv.plan_attention(case.batch, case.max_q_rows, case.num_q_heads, case.num_kv_heads,
                              case.head_dim, case.max_kv_len, kw.get("num_splits", 0), kw.get("flags", 0))
    assert plan["kernel"] == kernel, plan
    out, lse, *_, err = gpu_step(case, **kw)
    assert err == 0
    O, L, *_ = oracle_step(case)
    assert_attention_close(out, lse, O, L, case)
    return plan


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 77), ("none", 0)])
@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (8, 8), (32, 2)])
def test_head_dim_64_two_tile(mask, cb, Hq, Hkv):
    case = wl.random_case(80 + Hq, batch=4, Hq=Hq, Hkv=Hkv, D=64, kv_range=(300, 2500), q_range=(40, 400),
                          pad_range=(0, 7), mask=mask, causal_block=cb)
    _run(case)


@pytest.mark.parametrize("q_range", [(1, 3), (5, 12)])
def test_head_dim_64_one_tile(q_range):
    # rows x G <= 32 holds the rows four times; more rows, once
    case = wl.random_case(90 + q_range[0], batch=9, Hq=32, Hkv=4, D=64, kv_range=(1, 1800), q_range=q_range,
                          pad_range=(0, 1), mask="causal", q_scale=4.0)
    _run(case, out_dtype=torch.float32)


def test_head_dim_64_key_splits_and_f32():
    case = wl.random_case(95, batch=2, Hq=16, Hkv=2, D=64, kv_range=(2000, 5000), q_range=(100, 300),
                          mask="causal")
    p = _run(case, num_splits=3, out_dtype=torch.float32)
    assert p["splits"] == 3


@pytest.mark.parametrize("Hq,Hkv", [(24, 8), (40, 8), (48, 8), (56, 8), (96, 8), (40, 1), (64, 1)])
def test_odd_head_groups_prefill(Hq, Hkv):
    # floor(128 / G) tokens per tile; the last 128 mod G lanes stay empty
    case = wl.random_case(100 + Hq + Hkv, batch=3, Hq=Hq, Hkv=Hkv, D=128, kv_range=(200, 2200),
                          q_range=(30, 260), pad_range=(0, 3), mask="causal", q_scale=3.0)
    _run(case, out_dtype=torch.float32)


@pytest.mark.parametrize("Hq,Hkv,D", [(24, 8, 128), (40, 8, 128), (96, 8, 128), (48, 8, 64), (64, 1, 64)])
def test_odd_head_groups_decode(Hq, Hkv, D):
    # one query row per sequence with a group the decode kernel does not take
    case = wl.random_case(120 + Hq, batch=20, Hq=Hq, Hkv=Hkv, D=D, kv_range=(1, 3000), mask="causal",
                          q_scale=3.0)
    _run(case, out_dtype=torch.float32)


@pytest.mark.parametrize("q_len", [1, 4])
@pytest.mark.parametrize("heads,D", [((24, 8), 128), ((16, 4), 64), ((8, 8), 64)])
def test_grouped_shared_prefix_new_shapes(q_len, heads, D):
    case = wl.shared_prefix(seed=130 + q_len, groups=3, samples=5, prefix=256, tail_lo=1, tail_hi=200,
                            Hq=heads[0], Hkv=heads[1], D=D, q_len=q_len)
    out, lse, plan = fused_step(case)
    O, L, *_ = oracle_step(case)
    assert_attention_close(out, lse, O, L, case)


@pytest.mark.parametrize("Hq,Hkv,D", [(24, 8, 128), (16, 4, 64)])
def test_stream_k_new_shapes(Hq, Hkv, D):
    case = wl.random_case(140 + Hq, batch=5, Hq=Hq, Hkv=Hkv, D=D, kv_range=(500, 3000), q_range=(100, 300),
                          pad_range=(0, 5), mask="block_causal", causal_block=61)
    _run(case, kernel=pkv.PKV_KERNEL_TILE_STREAM_K, flags=pkv.PKV_FLAG_STREAM_K)


def test_head_dim_64_page_permutation_bit_identical():
    """Results do not depend on where pages sit in the pool: bit-identical."""
    case = wl.random_case(150, batch=3, Hq=16, Hkv=4, D=64, kv_range=(500, 1500), q_range=(50, 200),
                          mask="causal")
    out1, lse1, *_ = gpu_step(case)
    rng = np.random.default_rng(150)
    perm = rng.permutation(case.num_pages)
    inv = np.argsort(perm)
    kp = case.k_pool[torch.from_numpy(inv)]
    vp = case.v_pool[torch.from_numpy(inv)]
    bt = case.block_table.numpy().copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    slots = case.slots.numpy().copy()
    ok = slots >= 0
    slots[ok] = perm[slots[ok] // 32] * 32 + slots[ok] % 32
    c2 = wl.PagedCase(name="perm", num_q_heads=16, num_kv_heads=4, head_dim=64, page_size=32, k_pool=kp,
                      v_pool=vp, block_table=torch.from_numpy(bt), kv_lens=case.kv_lens, q=case.q,
                      q_indptr=case.q_indptr, q_real=case.q_real, new_k=case.new_k, new_v=case.new_v,
                      slots=torch.from_numpy(slots), mask="causal")
    out2, lse2, *_ = gpu_step(c2)
    assert torch.equal(out1.cpu(), out2.cpu())
    assert torch.equal(lse1.cpu(), lse2.cpu())


def test_head_dim_64_two_tile_after_grouped_launches():
    """Kernels run before a tile call leave their data in shared and tensor
    memory.  A reducing tensor-memory load once let rows of a warp that also held
    padding rows come out as zero with LSE -inf after the shared-prefix planner and
    grouped launches had run (the suite's file order exposed it).  The same
    sequence in one test: those launches, then every head-dim-64 two-tile case."""
    import itertools
    import test_gpu_plan as tp
    for seed in range(6):
        tp.test_plan_matches_oracle_random(seed)
    tp.test_plan_matches_oracle_edge_cases()
    for q_len, heads in itertools.product([1, 4, 16], [(32, 8), (8, 8), (16, 1)]):
        tp.test_fused_shared_prefix_small(q_len, heads)
    tp.test_fused_nan_in_unused_slots_and_random_batches()
    for q_len in (1, 4):
        tp.test_fused_shared_prefix_full_size(q_len)
    tp.test_fused_shared_prefix_graph_replay()
    for (mask, cb), (hq, hkv) in itertools.product([("causal", 0), ("block_causal", 77), ("none", 0)],
                                                   [(16, 4), (8, 8), (32, 2)]):
        test_head_dim_64_two_tile(mask, cb, hq, hkv)
