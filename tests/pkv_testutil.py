"""Shared helpers for the parity tests: run a synthetic step through the CUDA
library (via the C-ABI binding) and through the fp64 oracle, and compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv

# Tolerances for bf16 attention outputs against the fp64 oracle: max-abs 1e-2,
# mean-abs 1e-3 on the output, LSE within 1e-3 (absolute).
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def oracle_step(case, scatter=True, rows=None):
    """Scatter the case's new rows into its pools, then attend (oracle)."""
    kb, vb = orc.bf16_bits(case.k_pool), orc.bf16_bits(case.v_pool)
    if scatter:
        kb, vb, _ = orc.kv_scatter_slots(orc.bf16_bits(case.new_k), orc.bf16_bits(case.new_v),
                                         case.slots.numpy(), kb, vb)
    O, L = orc.paged_attention(orc.bf16_bits(case.q), kb, vb, case.block_table.numpy(),
                               case.kv_lens.numpy(), case.q_indptr.numpy(), case.q_real.numpy(),
                               mask=case.mask, causal_block=case.causal_block, rows=rows)
    return O, L, kb, vb


def gpu_step(case, scatter=True, out_dtype=torch.bfloat16, flags=0, num_splits=0,
             with_lse=True, max_kv_len=None, max_q_rows=None, checked=False):
    dev = "cuda"
    k_pool = case.k_pool.to(dev)
    v_pool = case.v_pool.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if scatter:
        pkv.kv_scatter_slots(case.new_k.to(dev), case.new_v.to(dev), case.slots.to(dev), k_pool,
                             v_pool, checked=checked, err=err)
    rows = case.q.shape[0]
    Hq, D = case.num_q_heads, case.head_dim
    out = torch.full((rows, Hq, D), float("nan"), dtype=out_dtype, device=dev)
    lse = torch.full((rows, Hq), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    mq = max_q_rows or case.max_q_rows
    mk = max_kv_len or case.max_kv_len
    fl = flags | (pkv.PKV_FLAG_CHECKED if checked else 0)
    ws_bytes = pkv.paged_attention_workspace_size(case.batch, mq, Hq, case.num_kv_heads, D, mk,
                                                  num_splits, fl)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    pkv.paged_attention(case.q.to(dev), k_pool, v_pool, case.block_table.to(dev),
                        case.kv_lens.to(dev), case.q_indptr.to(dev), out,
                        q_real=case.q_real.to(dev), lse=lse, max_q_rows=mq, max_kv_len=mk,
                        mask=case.mask, causal_block=case.causal_block, workspace=ws,
                        num_splits=num_splits, flags=fl, err=err)
    torch.cuda.synchronize()
    return out, lse, k_pool, v_pool, int(err.item())


def real_row_mask(case):
    qi = case.q_indptr.numpy()
    qr = case.q_real.numpy()
    m = np.zeros(case.q.shape[0], dtype=bool)
    for b in range(case.batch):
        m[qi[b]:qi[b] + qr[b]] = True
    return m


def assert_attention_close(out, lse, O, L, case, rows=None):
    """out/lse: GPU tensors; O/L: oracle arrays.  Real rows within tolerance,
    padding rows exactly zero with LSE -inf."""
    got = out.float().cpu().numpy().astype(np.float64)
    real = real_row_mask(case)
    sel = np.arange(case.q.shape[0]) if rows is None else np.asarray(sorted(rows))
    r_sel = sel[real[sel]]
    p_sel = sel[~real[sel]]
    if len(r_sel):
        diff = np.abs(got[r_sel] - O[r_sel])
        assert np.isfinite(got[r_sel]).all(), "non-finite output"
        assert diff.max() <= O_MAX_ABS, f"max abs {diff.max():.3e}"
        assert diff.mean() <= O_MEAN_ABS, f"mean abs {diff.mean():.3e}"
        if lse is not None:
            gl = lse.cpu().numpy().astype(np.float64)
            # real rows with an empty visible set: exactly -inf (and zero output)
            none = np.isneginf(L[r_sel])
            assert np.isneginf(gl[r_sel][none]).all(), "empty visible set must give LSE -inf"
            assert (got[r_sel][none] == 0).all(), "empty visible set must give zero output"
            dl = np.abs(gl[r_sel][~none] - L[r_sel][~none])
            assert dl.size == 0 or dl.max() <= LSE_MAX_ABS, f"lse max abs {dl.max():.3e}"
    if len(p_sel):
        assert (got[p_sel] == 0).all(), "padding rows must be zero"
        if lse is not None:
            assert np.isneginf(lse.cpu().numpy()[p_sel]).all()
