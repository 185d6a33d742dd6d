"""GPU parity of the shared-prefix planner and of the one-launch grouped
attention, through the C ABI.

* plan_shared_prefix on the device equals the oracle's plan bit for bit:
  group count, members in order, shared runs, group rows, tail starts and
  lengths, over random n-sample batches (groups interleaved, groups whose
  members share the page with their new tokens, rows sharing nothing), the
  hand-derived batch, a single row, and 1024 rows;
* shared_prefix_attention (plan + one launch) equals the oracle's causal
  attention over every row's full block table (max-abs 1e-2, mean-abs 1e-3,
  LSE 1e-3), for 1, 4 and 16 query tokens per row, with NaN in every pool slot
  no row uses, at the full n-sample geometry (16 groups x 8 samples over a
  4096-token prefix) and captured in a CUDA graph.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl
from pkv_testutil import assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"
P = 32


def run_plan(table, kv, ql, stride=None):
    B = len(kv)
    qi = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    ref = orc.plan_shared_prefix(table, kv, ql)
    if stride is None:
        stride = max(len(r) for r in ref["group_rows"]) + 5
    plan = pkv.plan_buffers(B, stride, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.plan_shared_prefix(torch.from_numpy(np.ascontiguousarray(table, np.int32)).to(DEV),
                           torch.from_numpy(np.asarray(kv, np.int32)).to(DEV), torch.from_numpy(qi).to(DEV),
                           plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return plan, ref


def check_plan(plan, ref, B):
    ng = int(plan["num_groups"].item())
    assert ng == len(ref["groups"])
    gi = plan["group_indptr"].cpu().numpy()
    perm = plan["perm"].cpu().numpy()
    runs = plan["run_lens"].cpu().numpy()
    rows = plan["group_rows"].cpu().numpy()
    for g, members in enumerate(ref["groups"]):
        assert perm[gi[g]:gi[g + 1]].tolist() == members
        assert runs[g] == P * ref["run_pages"][g]
        row = ref["group_rows"][g]
        assert rows[g, :len(row)].tolist() == row
        assert (rows[g, len(row):] == -1).all()
    assert (gi[ng:] == B).all() and gi[0] == 0
    assert (runs[ng:] == 0).all() and (rows[ng:] == -1).all()
    for k in ("tail_start", "tail_lens", "group_of"):
        assert plan[k].cpu().numpy().tolist() == ref[k], k
    assert perm.tolist() == ref["perm"]


@pytest.mark.parametrize("seed", range(6))
def test_plan_matches_oracle_random(seed):
    table, kv, ql, _ = wl.nsample_tables(np.random.default_rng(seed))
    plan, ref = run_plan(table, kv, ql)
    check_plan(plan, ref, len(kv))


def test_plan_matches_oracle_edge_cases():
    # one row; every row alone; the hand-derived batch; 1024 rows
    for table, kv, ql in [
        (np.array([[3, 4]], np.int32), [40], [1]),
        (np.arange(8, dtype=np.int32).reshape(8, 1), [30] * 8, [1] * 8),
        (np.array([[5, 6, 7, 20, -1], [5, 6, 7, 21, 22], [9, 1, 2, -1, -1], [5, 6, 8, 23, -1],
                   [9, 1, 3, -1, -1], [4, -1, -1, -1, -1], [30, 31, -1, -1, -1], [30, 31, -1, -1, -1]],
                  np.int32), [120, 150, 70, 100, 90, 10, 40, 45], [1, 1, 1, 1, 4, 1, 1, 1]),
    ]:
        plan, ref = run_plan(table, np.array(kv), np.array(ql))
        check_plan(plan, ref, len(kv))
    table, kv, ql, _ = wl.nsample_tables(np.random.default_rng(99), n_groups=150, loners=300, width=16)
    table, kv, ql = table[:1024], kv[:1024], ql[:1024]
    plan, ref = run_plan(table, kv, ql)
    check_plan(plan, ref, len(kv))


def fused_step(case, dev=DEV, graph=False):
    """Scatter, plan and one grouped attention launch on the GPU."""
    k_pool, v_pool = case.k_pool.to(dev), case.v_pool.to(dev)
    pkv.kv_scatter_slots(case.new_k.to(dev), case.new_v.to(dev), case.slots.to(dev), k_pool, v_pool)
    table, kv, qi = case.block_table.to(dev), case.kv_lens.to(dev), case.q_indptr.to(dev)
    B = case.batch
    ql = case.q_indptr[1:] - case.q_indptr[:-1]
    max_q = int(ql.max())
    width = table.shape[1]
    max_group = B  # no bound known: every row could be in one group
    stride = width * max_group
    max_keys = stride * P
    plan = pkv.plan_buffers(B, stride, dev)
    n, Hq, D = case.q.shape
    q = case.q.to(dev)
    out = torch.full((n, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((n, Hq), float("nan"), device=dev)
    mgt = int(ql.sum())
    ws_b = pkv.shared_prefix_attention_workspace_size(B, max_q, mgt, max_keys, Hq, case.num_kv_heads, D)
    ws = torch.empty(max(ws_b, 1), dtype=torch.uint8, device=dev)

    def step(stream=None):
        pkv.plan_shared_prefix(table, kv, qi, plan, stream=stream)
        pkv.shared_prefix_attention(q, k_pool, v_pool, plan, qi, out, lse=lse, max_q_len=max_q,
                                    max_group_tokens=mgt, max_group_keys=max_keys, workspace=ws,
                                    stream=stream)
    if graph:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            step(s)
            s.synchronize()
            out.fill_(float("nan"))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step(s)
        g.replay()
    else:
        step()
    torch.cuda.synchronize()
    return out, lse, plan


@pytest.mark.parametrize("q_len", [1, 4, 16])
@pytest.mark.parametrize("heads", [(32, 8), (8, 8), (16, 1)])
def test_fused_shared_prefix_small(q_len, heads):
    case = wl.shared_prefix(seed=7 + q_len, groups=3, samples=5, prefix=256, tail_lo=1, tail_hi=200,
                            Hq=heads[0], Hkv=heads[1], q_len=q_len)
    out, lse, plan = fused_step(case)
    assert int(plan["num_groups"].item()) == 3
    O, L, *_ = oracle_step(case)
    assert_attention_close(out, lse, O, L, case)


def test_fused_nan_in_unused_slots_and_random_batches():
    """Random n-sample batches (groups sharing the page with their new tokens,
    loners); every pool slot no row reads holds NaN."""
    rng = np.random.default_rng(5)
    table, kv, ql, _ = wl.nsample_tables(rng, n_groups=6, loners=5, width=24)
    Hq, Hkv, D = 16, 4, 128
    B = len(kv)
    n_pages = int(table.max()) + 2
    gen = torch.Generator().manual_seed(5)
    k_pool = wl.randn_bf16((n_pages, P, Hkv, D), gen)
    v_pool = wl.randn_bf16((n_pages, P, Hkv, D), gen)
    used = np.zeros((n_pages, P), bool)
    for r in range(B):
        for p in range(kv[r]):
            used[table[r][p // P], p % P] = True
    k_pool[torch.from_numpy(~used)] = float("nan")
    v_pool[torch.from_numpy(~used)] = float("nan")
    qi = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    case = wl.PagedCase(name="nsample_random", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                        k_pool=k_pool, v_pool=v_pool, block_table=torch.from_numpy(table),
                        kv_lens=torch.from_numpy(kv.astype(np.int32)), q=wl.randn_bf16((int(qi[-1]), Hq, D), gen),
                        q_indptr=torch.from_numpy(qi), q_real=torch.from_numpy(ql.astype(np.int32)),
                        new_k=wl.randn_bf16((0, Hkv, D), gen), new_v=wl.randn_bf16((0, Hkv, D), gen),
                        slots=torch.zeros(0, dtype=torch.int64), mask="causal")
    out, lse, _ = fused_step(case)
    O, L, *_ = oracle_step(case, scatter=False)
    assert_attention_close(out, lse, O, L, case)


@pytest.mark.parametrize("q_len", [1, 4])
def test_fused_shared_prefix_full_size(q_len):
    case = wl.shared_prefix(q_len=q_len)
    out, lse, plan = fused_step(case)
    assert int(plan["num_groups"].item()) == 16
    assert plan["run_lens"][:16].tolist() == [4096] * 16
    O, L, *_ = oracle_step(case)
    assert_attention_close(out, lse, O, L, case)


def test_fused_shared_prefix_graph_replay():
    case = wl.shared_prefix(seed=21, groups=4, samples=4, prefix=512, tail_lo=1, tail_hi=300, q_len=2)
    out, lse, _ = fused_step(case, graph=True)
    O, L, *_ = oracle_step(case)
    assert_attention_close(out, lse, O, L, case)
