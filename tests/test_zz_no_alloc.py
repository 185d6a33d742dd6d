"""paged_attention_no_alloc: the entry point for callers that cannot allocate
(graph capture, fixed-memory servers, pointer-only plugin hosts).  Its scratch
is a fixed device array inside the library, so it takes no workspace.

Checked here, through the C ABI, against paged_attention with a caller
workspace, on two calls in a row (the second call finds the first call's
leftovers in the shared scratch), with the attention tolerances used by every
parity test (max-abs 1e-2, mean-abs 1e-3 on bf16 outputs, LSE 1e-3).  This
file sorts last so that a run stopping at the first failure has already run
every other test."""
import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(case, no_alloc):
    k_pool, v_pool = case.k_pool.to(DEV), case.v_pool.to(DEV)
    pkv.kv_scatter_slots(case.new_k.to(DEV), case.new_v.to(DEV), case.slots.to(DEV), k_pool, v_pool)
    rows, Hq, D = case.q.shape
    out = torch.full((rows, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((rows, Hq), float("nan"), dtype=torch.float32, device=DEV)
    args = (case.q.to(DEV), k_pool, v_pool, case.block_table.to(DEV), case.kv_lens.to(DEV),
            case.q_indptr.to(DEV), out)
    kw = dict(q_real=case.q_real.to(DEV), lse=lse, max_q_rows=1, max_kv_len=case.max_kv_len)
    if no_alloc:
        pkv.paged_attention_no_alloc(*args, **kw)
    else:
        ws_bytes = pkv.paged_attention_workspace_size(case.batch, 1, Hq, case.num_kv_heads, D,
                                                      case.max_kv_len)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
        pkv.paged_attention(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def test_no_alloc_matches_paged_attention_on_two_calls():
    for seed in (31, 32):
        # several 512-key splits per row, so the scratch holds partial states
        case = wl.random_case(seed, batch=16, Hq=32, Hkv=8, D=128, kv_range=(1, 3000))
        need = pkv.paged_attention_workspace_size(case.batch, 1, 32, 8, 128, case.max_kv_len)
        assert 0 < need <= pkv.NO_ALLOC_SCRATCH_BYTES
        ref_o, ref_l = _run(case, no_alloc=False)
        got_o, got_l = _run(case, no_alloc=True)
        assert np.isfinite(got_o).all()
        diff = np.abs(got_o - ref_o)
        assert diff.max() <= 1e-2 and diff.mean() <= 1e-3
        assert np.abs(got_l - ref_l).max() <= 1e-3


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
