"""GPU parity of the exact-window layout and of a forward over it.

* causal_layout on the device equals the oracle's layout bit for bit (rows,
  key counts, query ranges, both staged slots, both copy lists once their -1
  sentinels are dropped) over edge-case geometries and the full video one;
* the forward through the C ABI -- commit copies (copy_kv_slots), the staged
  K/V to their two slots and the earlier blocks' tokens to the later blocks'
  private pages (kv_scatter_slots, the second time with source indices), one
  unmasked ragged attention over all blocks -- equals the oracle's dense
  attention over each block's exact window (max-abs 1e-2, mean-abs 1e-3, LSE
  1e-3), at small size on every row and at the video geometry on sampled rows;
* the forward captured once in a CUDA graph replays correctly after a commit
  that only device kernels performed (layout + copies).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
P = 32


def gpu_layout(case, committed=None, table=None):
    committed = case.committed if committed is None else committed
    table = case.table if table is None else table
    bufs = pkv.causal_layout_buffers(case.staged, case.block, case.row_stride, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.causal_layout(table.to(DEV), torch.tensor([committed], dtype=torch.int64, device=DEV), case.pin,
                      case.window, case.staged, case.block, case.private_pages.to(DEV), bufs, err=err)
    torch.cuda.synchronize()
    return bufs, int(err.item())


def oracle_layout(case):
    return orc.causal_layout(case.table.numpy(), case.pin, case.committed, case.window, case.staged,
                             case.block, case.private_pages.numpy())


GEOMS = [
    # pin, committed, window, staged, block
    (37, 90, 40, 70, 24),        # generic
    (0, 0, 0, 50, 7),            # no fixed region, no history, no window
    (64, 100, 1000, 33, 1),      # one-token blocks, window reaching the fixed region
    (5, 300, 31, 100, 100),      # one block, window shorter than a page
    (33, 64, 10, 96, 20),        # later blocks' windows start inside this forward
    (512, 96 * 394, 95 * 394, 4 * 394, 394),   # the video clean pass
    (512, 96 * 394, 95 * 394, 4 * 394, 1576),  # the video denoising forward
]


@pytest.mark.parametrize("geom", GEOMS)
def test_causal_layout_matches_oracle(geom):
    pin, committed, window, staged, block = geom
    case = wl.exact_window(11, pin, committed, window, staged, block, Hq=4, Hkv=2, D=64)
    bufs, err = gpu_layout(case)
    assert err == 0
    L = oracle_layout(case)
    rows = bufs["rows"].cpu().numpy()
    for k, r in enumerate(L["rows"]):
        np.testing.assert_array_equal(rows[k, :len(r)], r)
        assert (rows[k, len(r):] == -1).all()
    np.testing.assert_array_equal(bufs["kv_lens"].cpu().numpy(), L["kv_lens"])
    np.testing.assert_array_equal(bufs["q_indptr"].cpu().numpy(), L["q_indptr"])
    np.testing.assert_array_equal(bufs["staged_slots"].cpu().numpy(), L["staged_slots"])
    np.testing.assert_array_equal(bufs["staged_slots2"].cpu().numpy(), L["staged_slots2"])
    cs, cd = bufs["committed_src"].cpu().numpy(), bufs["committed_dst"].cpu().numpy()
    assert ((cs < 0) == (cd < 0)).all()
    assert [(int(a), int(b)) for a, b in zip(cs, cd) if a >= 0] == L["committed"]
    us, ud = bufs["current_src_idx"].cpu().numpy(), bufs["current_dst"].cpu().numpy()
    assert ((us < 0) == (ud < 0)).all()
    assert [(int(a), int(b)) for a, b in zip(us, ud) if a >= 0] == L["current"]


def test_causal_layout_reports_small_capacities():
    case = wl.exact_window(12, 37, 90, 40, 70, 24, Hq=4, Hkv=2, D=64)
    case.private_pages = case.private_pages[:, :1].contiguous()  # too few private pages
    _, err = gpu_layout(case)
    assert err & pkv.PKV_ERRBIT_LEN


def logical_sequence(case, committed, k_pool, v_pool, new_k, new_v, table):
    """K/V of the long sequence by logical position: committed tokens from the
    pool through the table, staged ones from the forward's rows."""
    base = case.pin + committed
    pos = np.arange(base)
    slots = table[pos // P].astype(np.int64) * P + pos % P
    kb = orc.bf16_bits(k_pool.cpu()).reshape(-1, case.num_kv_heads, case.head_dim)
    vb = orc.bf16_bits(v_pool.cpu()).reshape(-1, case.num_kv_heads, case.head_dim)
    k_seq = np.concatenate([kb[slots], orc.bf16_bits(new_k)])
    v_seq = np.concatenate([vb[slots], orc.bf16_bits(new_v)])
    return k_seq, v_seq


def forward(case, bufs, k_pool, v_pool, new_k, new_v, q, out, lse, ws, stream=None):
    """One forward over the layout: the staged K/V to both slots, the earlier
    blocks' tokens to the later blocks' private pages, attention."""
    pkv.kv_scatter_slots(new_k, new_v, bufs["staged_slots"], k_pool, v_pool,
                         slots2=bufs["staged_slots2"], stream=stream)
    pkv.kv_scatter_slots(new_k, new_v, bufs["current_dst"], k_pool, v_pool,
                         src_idx=bufs["current_src_idx"], stream=stream)
    pkv.paged_attention(q, k_pool, v_pool, bufs["rows"], bufs["kv_lens"], bufs["q_indptr"], out, lse=lse,
                        max_q_rows=case.block, max_kv_len=case.max_kv_len, mask="none", workspace=ws,
                        stream=stream)


def commit_copies(bufs, k_pool, v_pool, stream=None):
    pkv.copy_kv_slots(k_pool, v_pool, bufs["committed_src"], bufs["committed_dst"], stream=stream)


def run_case(case, rows=None):
    k_pool, v_pool = case.k_pool.to(DEV), case.v_pool.to(DEV)
    table_np = case.table.numpy()
    k_seq, v_seq = logical_sequence(case, case.committed, case.k_pool, case.v_pool, case.new_k,
                                    case.new_v, table_np)
    bufs, err = gpu_layout(case)
    assert err == 0
    commit_copies(bufs, k_pool, v_pool)
    n, Hq, D = case.q.shape
    out = torch.empty(n, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(n, Hq, device=DEV)
    ws = torch.empty(max(1, pkv.paged_attention_workspace_size(case.num_blocks, case.block, Hq,
                                                              case.num_kv_heads, D, case.max_kv_len)),
                     dtype=torch.uint8, device=DEV)
    forward(case, bufs, k_pool, v_pool, case.new_k.to(DEV), case.new_v.to(DEV), case.q.to(DEV), out, lse, ws)
    torch.cuda.synchronize()
    O, L = orc.exact_window_attention(orc.bf16_bits(case.q), k_seq, v_seq, case.pin, case.committed,
                                      case.window, case.staged, case.block, rows=rows)
    return out, lse, O, L


def check(out, lse, O, L, rows):
    o = out.float().cpu().numpy()[rows]
    err = np.abs(o - O[rows])
    assert err.max() <= 1e-2, err.max()
    assert err.mean() <= 1e-3, err.mean()
    assert np.abs(lse.cpu().numpy()[rows] - L[rows]).max() <= 1e-3


@pytest.mark.parametrize("geom", GEOMS[:5])
@pytest.mark.parametrize("heads", [(8, 2), (4, 4)])
def test_exact_window_forward_small(geom, heads):
    pin, committed, window, staged, block = geom
    case = wl.exact_window(21, pin, committed, window, staged, block, Hq=heads[0], Hkv=heads[1], D=128)
    out, lse, O, L = run_case(case)
    check(out, lse, O, L, np.arange(case.staged))


@pytest.mark.parametrize("blocks", [4, 1])
def test_exact_window_video_full_size_sampled(blocks):
    case = wl.exact_window_video(blocks_per_chunk=blocks)
    rng = np.random.default_rng(3)
    rows = sorted(r for r in set(rng.integers(0, case.staged, 48).tolist()) |
                  {0, case.block - 1, case.block, case.staged - 1} if r < case.staged)
    out, lse, O, L = run_case(case, rows=rows)
    check(out, lse, O, L, np.array(rows))


def test_forward_graph_replays_across_a_device_side_commit():
    """Capture the forward once; commit (the committed count advances on the
    device, the layout and the commit copies rerun); write the next forward's
    inputs into the same buffers and replay: the result is the next forward's
    exact-window attention."""
    pin, window, staged, block = 40, 150, 64, 16
    c0 = 100
    case = wl.exact_window(31, pin, c0, window, 2 * staged, block, Hq=8, Hkv=2, D=128)
    # the table covers both forwards; the first forward uses its first `staged` tokens
    first = wl.ExactWindowCase(**{**case.__dict__, "staged": staged})
    new_k2 = wl.randn_bf16((staged, 2, 128), torch.Generator().manual_seed(9))
    new_v2 = wl.randn_bf16((staged, 2, 128), torch.Generator().manual_seed(10))
    q2 = wl.randn_bf16((staged, 8, 128), torch.Generator().manual_seed(11))
    k_pool, v_pool = case.k_pool.to(DEV), case.v_pool.to(DEV)
    table = case.table.to(DEV)
    priv = case.private_pages[:first.num_blocks].contiguous().to(DEV)
    committed = torch.tensor([c0], dtype=torch.int64, device=DEV)
    bufs = pkv.causal_layout_buffers(staged, block, first.row_stride, DEV)
    new_k, new_v, q = first.new_k[:staged].to(DEV), first.new_v[:staged].to(DEV), first.q[:staged].to(DEV)
    out = torch.empty(staged, 8, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(staged, 8, device=DEV)
    ws = torch.empty(max(1, pkv.paged_attention_workspace_size(first.num_blocks, block, 8, 2, 128,
                                                              first.max_kv_len)),
                     dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.causal_layout(table, committed, pin, window, staged, block, priv, bufs, stream=s)
        commit_copies(bufs, k_pool, v_pool, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        forward(first, bufs, k_pool, v_pool, new_k, new_v, q, out, lse, ws, stream=s)
    # forward 1 (replay) against the oracle
    k_seq, v_seq = logical_sequence(first, c0, case.k_pool, case.v_pool, first.new_k[:staged],
                                    first.new_v[:staged], case.table.numpy())
    g.replay()
    torch.cuda.synchronize()
    O, L = orc.exact_window_attention(orc.bf16_bits(first.q[:staged]), k_seq, v_seq, pin, c0, window,
                                      staged, block)
    check(out, lse, O, L, np.arange(staged))
    # commit on the device: the staged tokens (already at their own slots) become history
    with torch.cuda.stream(s):
        committed.add_(staged)
        pkv.causal_layout(table, committed, pin, window, staged, block, priv, bufs, stream=s)
        commit_copies(bufs, k_pool, v_pool, stream=s)
    s.synchronize()
    pool_k_after, pool_v_after = k_pool.cpu(), v_pool.cpu()
    new_k.copy_(new_k2.to(DEV))
    new_v.copy_(new_v2.to(DEV))
    q.copy_(q2.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    c1 = c0 + staged
    k_seq, v_seq = logical_sequence(first, c1, pool_k_after, pool_v_after, new_k2, new_v2,
                                    case.table.numpy())
    O, L = orc.exact_window_attention(orc.bf16_bits(q2), k_seq, v_seq, pin, c1, window, staged, block)
    check(out, lse, O, L, np.arange(staged))
