"""The stream-K schedule of the two-tile tensor-core kernel: one persistent
CTA per SM runs one whole tile pair of the first wave (when the pairs fill
one) and then a contiguous share of the remaining pairs' 128-key tiles; pairs
split between CTAs leave partial states that a reduce merges by LSE.  Taken
on request (PKV_FLAG_STREAM_K), as every case here does.

Checked against the fp64 oracle (attention tolerances) and against the
one-CTA-per-tile grid (PKV_FLAG_TILE_GRID), on the schedule's edge cases: a
single tile pair spread over every CTA (a long chain of partial states, CTAs
with an empty share), pairs whose rows fill only one tile (lighter weight),
pairs of padding rows only and sequences without keys (zeroed by the
persistent CTAs), ragged causal and block-causal batches, f32 output."""
import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl

from pkv_testutil import assert_attention_close, gpu_step, oracle_step

pytestmark = pytest.mark.gpu


SK = pkv.PKV_FLAG_STREAM_K


def _check(case, **kw):
    plan = pkv.plan_attention(case.batch, case.max_q_rows, case.num_q_heads, case.num_kv_heads,
                              case.head_dim, case.max_kv_len, flags=SK)
    assert plan["kernel"] == pkv.PKV_KERNEL_TILE_STREAM_K
    out, lse, *_, err = gpu_step(case, flags=SK, **kw)
    assert err == 0
    O, L, *_ = oracle_step(case)
    assert_attention_close(out, lse, O, L, case)
    ref, ref_lse, *_ = gpu_step(case, flags=pkv.PKV_FLAG_TILE_GRID, **kw)
    d = np.abs(out.double().cpu().numpy() - ref.double().cpu().numpy())
    assert d.max() <= 1e-2 and d.mean() <= 1e-3
    return out, lse


def test_one_pair_over_every_cta():
    # one sequence, one K/V head, 200 rows (one pair, tile B partly filled) over
    # 3000 keys: 24 key tiles spread over all CTAs, most shares empty
    case = wl.build_pool_case("sk_one", 70, [3000], [200], [200], 1, 1, 128, mask="none")
    _check(case)


def test_light_pairs_and_zero_pairs():
    # causal chunks whose last pair fills one tile, a sequence of padding rows
    # only, and a sequence without keys
    kv = np.array([900, 2500, 700, 400, 1800])
    rows = np.array([300, 200, 150, 280, 40])
    real = np.array([300, 0, 150, 280, 40])
    case = wl.build_pool_case("sk_edges", 71, np.maximum(kv, real), rows, real, 16, 2, 128, mask="causal")
    _check(case)


def test_block_causal_ragged_and_f32_out():
    case = wl.random_case(72, batch=6, Hq=8, Hkv=8, D=128, kv_range=(200, 4000), q_range=(130, 600),
                          pad_range=(0, 9), mask="block_causal", causal_block=97)
    _check(case, out_dtype=torch.float32)


def test_grouped_heads_many_waves():
    # 7 sequences x 8 K/V heads x 3 pairs = 168 pairs (just over one wave)
    case = wl.random_case(73, batch=7, Hq=32, Hkv=8, D=128, kv_range=(1000, 9000), q_range=(150, 192),
                          mask="causal")
    _check(case)


def test_video_geometry():
    # the block-causal video step's shape: 7 pairs x 40 heads = 280 pairs
    # (1.84 waves: 152 whole first-wave pairs, 128 shared), shorter keys
    case = wl.build_pool_case("sk_video", 75, [2600], [1568], [1560], 40, 40, 128, mask="block_causal",
                              causal_block=1560, free_frac=0.0, identity_pages=True)
    _check(case)


def test_stream_k_graph_replay_follows_device_lengths():
    """The planner reads the lengths on the device every call: a captured call
    replays correctly after the lengths (within the host bounds) change."""
    case = wl.random_case(74, batch=4, Hq=16, Hkv=4, D=128, kv_range=(2000, 6000), q_range=(300, 300),
                          mask="causal")
    dev = "cuda"
    k_pool, v_pool = case.k_pool.to(dev), case.v_pool.to(dev)
    pkv.kv_scatter_slots(case.new_k.to(dev), case.new_v.to(dev), case.slots.to(dev), k_pool, v_pool)
    q, bt = case.q.to(dev), case.block_table.to(dev)
    kl, qi, qr = case.kv_lens.to(dev), case.q_indptr.to(dev), case.q_real.to(dev)
    out = torch.zeros(case.q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(case.q.shape[:2], dtype=torch.float32, device=dev)
    ws = torch.empty(pkv.paged_attention_workspace_size(4, 300, 16, 4, 128, case.max_kv_len, flags=SK),
                     dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    call = lambda: pkv.paged_attention(q, k_pool, v_pool, bt, kl, qi, out, q_real=qr, lse=lse, max_q_rows=300,
                                       max_kv_len=case.max_kv_len, workspace=ws, flags=SK, stream=s)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    # fewer real rows and shorter rows: the last 100 rows become padding
    qr2 = case.q_real.clone()
    qr2[:] = 200
    kl2 = case.kv_lens.clone() - 100
    qr.copy_(qr2)
    kl.copy_(kl2)
    g.replay()
    torch.cuda.synchronize()
    c2 = wl.PagedCase(name="replay", num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=32,
                      k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table, kv_lens=kl2,
                      q=case.q, q_indptr=case.q_indptr, q_real=qr2, new_k=case.new_k, new_v=case.new_v,
                      slots=case.slots, mask="causal")
    O, L, *_ = oracle_step(c2)
    assert_attention_close(out, lse, O, L, c2)
