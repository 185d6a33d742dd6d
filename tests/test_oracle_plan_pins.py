"""Pins of the oracle's shared-prefix planner (CPU only).

* the hand-derived plan in tests/golden/shared_prefix_plan_small.txt;
* on random n-sample batches (groups of rows built to share leading pages,
  private tails, unrelated rows): every row's keys are exactly its group's
  shared run followed by its tail, slot for slot; the built groups and shared
  runs are recovered; no member's new token lies in the run;
* attention over the full row equals the exact merge of attention over the
  group's shared run (every query sees all of it) and over the row's tail
  (causal), for every row.
"""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300.workloads import nsample_tables as nsample_batch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "shared_prefix_plan_small.txt")
P = 32


def load_golden():
    g = {"table": {}, "group_row": {}}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, _, rest = line.partition(" ")
        if key in ("table", "group_row"):
            k, _, vals = rest.partition(":")
            g[key][int(k)] = [int(v) for v in vals.split()]
        elif key == "groups":
            g[key] = [[int(x) for x in grp.split(",")] for grp in rest.split()]
        else:
            g[key] = [int(v) for v in rest.split()]
    return g


def test_plan_golden():
    g = load_golden()
    B = len(g["kv_lens"])
    width = max(len(v) for v in g["table"].values())
    table = np.full((B, width), -1, np.int32)
    for r, v in g["table"].items():
        table[r, :len(v)] = v
    plan = orc.plan_shared_prefix(table, g["kv_lens"], g["q_lens"])
    assert plan["groups"] == g["groups"]
    assert plan["run_pages"] == g["run_pages"]
    assert plan["group_rows"] == [g["group_row"][i] for i in range(len(g["groups"]))]
    for k in ("tail_start", "tail_lens", "group_of", "perm"):
        assert plan[k] == g[k], k


@pytest.mark.parametrize("seed", range(8))
def test_plan_rows_are_run_plus_tail(seed):
    rng = np.random.default_rng(seed)
    table, kv, ql, truth = nsample_batch(rng)
    plan = orc.plan_shared_prefix(table, kv, ql)
    B = len(kv)
    for r in range(B):
        gi = plan["group_of"][r]
        run = plan["run_pages"][gi]
        grow = plan["group_rows"][gi]
        slots_full = [table[r][p // P] * P + p % P for p in range(kv[r])]
        slots_run = [grow[p // P] * P + p % P for p in range(run * P)]
        ts = plan["tail_start"][r]
        slots_tail = [grow[ts + p // P] * P + p % P for p in range(plan["tail_lens"][r])]
        assert slots_run + slots_tail == slots_full
        assert run * P <= kv[r] - ql[r]
    got = {tuple(m) for m in plan["groups"] if len(m) > 1}
    assert got == {tuple(m) for m, _ in truth}
    for members, run in truth:
        gi = plan["group_of"][members[0]]
        cap = min((kv[m] - ql[m]) // P for m in members)
        assert plan["run_pages"][gi] == min(run, cap)
    assert sorted(plan["perm"]) == list(range(B))


def _bits(x):
    return orc.bf16_bits(torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16))


def test_plan_split_attention_equals_full_attention():
    rng = np.random.default_rng(42)
    table, kv, ql, _ = nsample_batch(rng, n_groups=3, loners=2, width=24)
    H, Hq, D = 2, 4, 64
    n_pages = int(table.max()) + 1
    kp = _bits(rng.standard_normal((n_pages, P, H, D)))
    vp = _bits(rng.standard_normal((n_pages, P, H, D)))
    qi = np.concatenate([[0], np.cumsum(ql)])
    q = _bits(rng.standard_normal((int(qi[-1]), Hq, D)))
    O, L = orc.paged_attention(q, kp, vp, np.maximum(table, 0), kv, qi, mask=orc.MASK_CAUSAL)
    plan = orc.plan_shared_prefix(table, kv, ql)
    B = len(kv)
    run_tab = np.zeros((B, 24), np.int64)
    tail_tab = np.zeros((B, 24), np.int64)
    run_len = np.zeros(B, np.int64)
    for r in range(B):
        gi = plan["group_of"][r]
        run = plan["run_pages"][gi]
        grow = plan["group_rows"][gi]
        run_tab[r, :run] = grow[:run]
        run_len[r] = run * P
        ts = plan["tail_start"][r]
        tp = (plan["tail_lens"][r] + P - 1) // P
        tail_tab[r, :tp] = grow[ts:ts + tp]
    Op, Lp = orc.paged_attention(q, kp, vp, run_tab, run_len, qi, mask=orc.MASK_NONE)
    Ot, Lt = orc.paged_attention(q, kp, vp, tail_tab, np.array(plan["tail_lens"]), qi,
                                 mask=orc.MASK_CAUSAL)
    Om, Lm = orc.merge_attn_states(Op, Lp, Ot, Lt)
    np.testing.assert_allclose(Om, O, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Lm, L, rtol=1e-12, atol=1e-12)
