"""Degenerate sequences through every attention path the plan picks.

One batch holds, side by side, sequences with no keys (all rows padding, or
real rows that see nothing), more new tokens than keys (the first rows sit
before key 0 and see nothing), one key, exactly one key tile, one key past a
tile, a ragged last page over several tiles, an ordinary sequence with padding
rows, and keys without rows.  [VG] Description, Attention (a real-token count
separate from the key count; padding rows neither attend nor are attended and
come back zero) and Cache ("Exact window" bullet: the new tokens are the last
keys of their row, so row i sits at kv_len - q_real + i).  Rows with an empty
visible set return O = 0 and LSE = -inf.  Checked against the fp64 oracle with
the usual bounds (max-abs 1e-2, mean-abs 1e-3, LSE 1e-3) with the output in
f32: a row that sees one to three keys returns nearly one V value (|v| up to
~4), where half a bf16 ulp alone is above 1e-2.  A second run with bf16 output
checks the empty rows (exactly zero, LSE -inf) and the LSE on the bf16 store
path.  The output buffer starts as NaN, so a row no kernel wrote fails."""
import numpy as np
import pytest
import torch

from paged_kv_cache_189_gb300 import pkv, workloads as wl

from pkv_testutil import assert_attention_close, gpu_step, oracle_step

pytestmark = pytest.mark.gpu


def degenerate_case(seed, q_len, Hq, Hkv, D, mask, cb):
    # (keys, rows, real rows) per sequence
    spec = [
        (0, q_len, 0),
        (0, q_len, q_len),
        (3, q_len, q_len),
        (1, q_len, 1),
        (128, q_len, q_len),
        (129, q_len, q_len),
        (32 * 40 + 31, q_len, q_len),
        (700, q_len, max(q_len - 2, 1)),
        (50, 0, 0),
    ]
    kv = np.array([s[0] for s in spec], dtype=np.int64)
    rows = np.array([s[1] for s in spec], dtype=np.int64)
    real = np.array([s[2] for s in spec], dtype=np.int64)
    # The generator places the real rows as the last keys of their sequence, so
    # its pools are built for at least that many keys; the key counts are then
    # cut to the degenerate values (the pools are read, never scattered into).
    c = wl.build_pool_case("degenerate", seed, np.maximum(kv, np.maximum(real, 1)), rows, real,
                           Hq, Hkv, D, mask=mask, causal_block=cb)
    c.kv_lens.copy_(torch.from_numpy(kv.astype(np.int32)))
    return c


# (q_len, Hq, Hkv, D, flags, num_splits, kernel the plan must pick)
PATHS = {
    "one_tile_rows_x4": (4, 32, 8, 128, 0, 1, pkv.PKV_KERNEL_TILE),
    "one_tile_rows_x4_splits": (4, 32, 8, 128, 0, 0, pkv.PKV_KERNEL_TILE),
    "one_tile": (20, 32, 8, 128, 0, 1, pkv.PKV_KERNEL_TILE),
    "one_tile_d64_splits": (20, 16, 4, 64, 0, 3, pkv.PKV_KERNEL_TILE),
    "two_tile": (70, 32, 8, 128, 0, 1, pkv.PKV_KERNEL_TILE),
    "two_tile_g1_splits": (200, 8, 8, 128, 0, 0, pkv.PKV_KERNEL_TILE),
    "two_tile_d64": (70, 32, 8, 64, 0, 1, pkv.PKV_KERNEL_TILE),
    "two_tile_stream_k": (70, 32, 8, 128, pkv.PKV_FLAG_STREAM_K, 0, pkv.PKV_KERNEL_TILE_STREAM_K),
    "two_tile_d64_stream_k": (200, 8, 8, 64, pkv.PKV_FLAG_STREAM_K, 0, pkv.PKV_KERNEL_TILE_STREAM_K),
    "single_row_group_8": (1, 64, 8, 128, 0, 0, pkv.PKV_KERNEL_TILE),
    "simt": (6, 8, 2, 128, pkv.PKV_FLAG_SIMT_ONLY, 0, pkv.PKV_KERNEL_SIMT),
}


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 3), ("none", 0)])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_degenerate_sequences(path, mask, cb):
    q_len, Hq, Hkv, D, flags, num_splits, kernel = PATHS[path]
    c = degenerate_case(900 + q_len, q_len, Hq, Hkv, D, mask, cb)
    plan = pkv.plan_attention(c.batch, c.max_q_rows, Hq, Hkv, D, c.max_kv_len, num_splits, flags)
    assert plan["kernel"] == kernel, plan
    if num_splits == 0 and flags == 0:
        assert plan["splits"] > 1, plan          # the split path and its merge
    O, L, *_ = oracle_step(c, scatter=False)
    empty = np.isneginf(L[:, 0])
    assert empty.any()
    out, lse, *_, err = gpu_step(c, scatter=False, flags=flags, num_splits=num_splits,
                                 out_dtype=torch.float32)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)
    out16, lse16, *_, err = gpu_step(c, scatter=False, flags=flags, num_splits=num_splits)
    assert err == 0
    got, gl = out16.float().cpu().numpy(), lse16.cpu().numpy()
    # rows with nothing visible: exactly zero with LSE -inf; the rest finite
    assert (got[empty] == 0).all() and np.isneginf(gl[empty]).all()
    assert np.isfinite(got[~empty]).all()
    np.testing.assert_allclose(gl[~empty], L[~empty], rtol=0, atol=1e-3)
