"""The bounded-wait failure path on the GPU, made to run without a fault.

Every device wait in the TMA-fed kernels gives up after a bounded time, sets
PKV_ERRBIT_TIMEOUT in the caller's error word and winds down: the waiting warps
leave together and the producer waits for every copy it issued before its CTA
exits, so the context stays usable.  PKV_FLAG_TEST_WAIT_TIMEOUT makes the
decode kernel's consumer warps wait on a barrier that nothing completes (a
flag nothing sets), with a ~20 us limit, so this path runs deterministically.
Checked: the call returns promptly, the error bit is set, and the same
context then computes a normal call correctly."""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl

from pkv_testutil import assert_attention_close, gpu_step, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("batch,kv_range", [(4, (40, 300)), (64, (600, 3000))])
def test_decode_wait_timeout_sets_error_and_returns(batch, kv_range):
    case = wl.random_case(50 + batch, batch=batch, Hq=32, Hkv=8, D=128, kv_range=kv_range)
    plan = pkv.plan_attention(case.batch, 1, 32, 8, 128, case.max_kv_len)
    assert plan["kernel"] == pkv.PKV_KERNEL_DECODE
    k_pool, v_pool = case.k_pool.to(DEV), case.v_pool.to(DEV)
    out = torch.zeros(case.q.shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(case.q.shape[:2], dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(plan["workspace_bytes"], 256), dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pkv.paged_attention(case.q.to(DEV), k_pool, v_pool, case.block_table.to(DEV), case.kv_lens.to(DEV),
                        case.q_indptr.to(DEV), out, q_real=case.q_real.to(DEV), lse=lse, max_q_rows=1,
                        max_kv_len=case.max_kv_len, workspace=ws, flags=pkv.PKV_FLAG_TEST_WAIT_TIMEOUT,
                        err=err)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) & pkv.PKV_ERRBIT_TIMEOUT
    assert dt < 1.0, f"the wind-down took {dt:.3f} s"
    # the context is intact: a normal call right after is correct
    got, got_lse, *_ = gpu_step(case)
    O, L, *_ = oracle_step(case)
    assert_attention_close(got, got_lse, O, L, case)


def test_wait_test_flag_is_refused_off_the_decode_kernel():
    case = wl.random_case(60, batch=2, Hq=16, Hkv=2, D=128, kv_range=(200, 400), q_range=(8, 8))
    out = torch.zeros(case.q.shape, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention(case.q.to(DEV), case.k_pool.to(DEV), case.v_pool.to(DEV), case.block_table.to(DEV),
                            case.kv_lens.to(DEV), case.q_indptr.to(DEV), out, max_q_rows=8,
                            max_kv_len=case.max_kv_len, flags=pkv.PKV_FLAG_TEST_WAIT_TIMEOUT, err=err)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    assert int(err.item()) == 0
