"""paged_attention_no_alloc: the entry point for callers that cannot allocate
(graph capture, fixed-memory servers, pointer-only plugin hosts).  Its scratch
is a fixed device array inside the library, so it takes no workspace.

Checked here, through the C ABI, against paged_attention with a caller
workspace and against the fp64 oracle, on two calls in a row (the second call
finds the first call's leftovers in the shared scratch), with the attention
tolerances used by every parity test (max-abs 1e-2, mean-abs 1e-3 on bf16
outputs, LSE 1e-3).  Two paths keep split partial states in the scratch: the
persistent decode kernel (single-row decode, head group 4) and the
tensor-core tile kernel (several causal rows per sequence, and single-row
decode with head group 8), each with key splits.  This file sorts last so
that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl

from pkv_testutil import assert_attention_close, oracle_step, real_row_mask

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(case, no_alloc, num_splits=0):
    k_pool, v_pool = case.k_pool.to(DEV), case.v_pool.to(DEV)
    pkv.kv_scatter_slots(case.new_k.to(DEV), case.new_v.to(DEV), case.slots.to(DEV), k_pool, v_pool)
    rows, Hq, D = case.q.shape
    out = torch.full((rows, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((rows, Hq), float("nan"), dtype=torch.float32, device=DEV)
    args = (case.q.to(DEV), k_pool, v_pool, case.block_table.to(DEV), case.kv_lens.to(DEV),
            case.q_indptr.to(DEV), out)
    kw = dict(q_real=case.q_real.to(DEV), lse=lse, max_q_rows=case.max_q_rows,
              max_kv_len=case.max_kv_len, mask=case.mask, num_splits=num_splits)
    if no_alloc:
        pkv.paged_attention_no_alloc(*args, **kw)
    else:
        ws_bytes = pkv.paged_attention_workspace_size(case.batch, case.max_q_rows, Hq, case.num_kv_heads,
                                                      D, case.max_kv_len, num_splits)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
        pkv.paged_attention(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    return out, lse


def _check_pair(case, num_splits=0):
    need = pkv.paged_attention_workspace_size(case.batch, case.max_q_rows, case.num_q_heads,
                                              case.num_kv_heads, case.head_dim, case.max_kv_len,
                                              num_splits)
    assert 0 < need <= pkv.NO_ALLOC_SCRATCH_BYTES
    ref_o, ref_l = _run(case, no_alloc=False, num_splits=num_splits)
    got_o, got_l = _run(case, no_alloc=True, num_splits=num_splits)
    g, r = got_o.double().cpu().numpy(), ref_o.double().cpu().numpy()
    assert np.isfinite(g).all()
    diff = np.abs(g - r)
    assert diff.max() <= 1e-2 and diff.mean() <= 1e-3
    real = real_row_mask(case)
    gl, rl = got_l.double().cpu().numpy(), ref_l.double().cpu().numpy()
    assert np.abs(gl[real] - rl[real]).max() <= 1e-3
    assert np.isneginf(gl[~real]).all() and np.isneginf(rl[~real]).all()   # padding rows
    O, L, _, _ = oracle_step(case)
    assert_attention_close(got_o, got_l, O, L, case)


def test_no_alloc_matches_paged_attention_on_two_calls():
    for seed in (31, 32):
        # several 512-key splits per row, so the scratch holds partial states
        case = wl.random_case(seed, batch=16, Hq=32, Hkv=8, D=128, kv_range=(1, 3000))
        _check_pair(case)


def test_no_alloc_tile_path_with_split_partials_on_two_calls():
    """The tensor-core tile kernel's key splits also keep their partial
    states in the scratch: several causal rows per sequence (one tile per
    sequence and K/V head), then single-row decode with 8 query heads per K/V
    head, each with 3 forced key splits; the second call of each pair reads
    the scratch the first one left."""
    cases = [wl.random_case(34, batch=3, Hq=16, Hkv=2, D=128, kv_range=(300, 1500), q_range=(5, 40),
                            pad_range=(0, 3)),
             wl.random_case(35, batch=6, Hq=64, Hkv=8, D=128, kv_range=(200, 1600))]
    for case in cases:
        for _ in range(2):
            _check_pair(case, num_splits=3)


def test_no_alloc_rejects_calls_beyond_its_scratch():
    case = wl.random_case(33, batch=2, Hq=32, Hkv=8, D=128, kv_range=(10, 40))
    out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device=DEV)
    # 64 sequences x 32 heads x 64 key splits of partial states: far more than the
    # scratch holds
    big, splits = 1 << 20, 64
    assert pkv.paged_attention_workspace_size(64, 1, 32, 8, 128, big, splits) > pkv.NO_ALLOC_SCRATCH_BYTES
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_no_alloc(case.q.to(DEV), case.k_pool.to(DEV), case.v_pool.to(DEV),
                                     case.block_table.to(DEV), case.kv_lens.to(DEV),
                                     case.q_indptr.to(DEV), out, batch=64, max_q_rows=1,
                                     max_kv_len=big, num_splits=splits)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE
    assert "scratch" in str(e.value)
