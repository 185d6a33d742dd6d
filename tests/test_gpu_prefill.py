"""GPU parity of the tensor-core tile path of paged_attention (several query
rows per sequence: causal / block-causal prefill, shared-prefix tiles)
against the fp64 oracle, through the C-ABI.

Tolerances (bf16 output vs fp64): max-abs 1e-2, mean-abs 1e-3, LSE 1e-3.
Full-size workloads are checked on sampled rows (every row of the first and
last query tile of each sequence plus a seeded random sample), the oracle
computing those rows one by one."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl
from pkv_testutil import assert_attention_close, gpu_step, oracle_step, real_row_mask

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 7), ("block_causal", 64),
                                     ("none", 0)])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 2), (4, 2), (32, 2)])
def test_tile_kernel_random(mask, cb, Hq, Hkv):
    c = wl.random_case(300 + Hq + cb, batch=3, Hq=Hq, Hkv=Hkv, D=128, kv_range=(40, 700),
                       q_range=(2, 150), pad_range=(0, 9), mask=mask, causal_block=cb)
    out, lse, *_ , err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


def test_multi_token_decode_workload():
    """Speculative verification rows: 4 new tokens per sequence, causal."""
    c = wl.multi_token_decode(batch=16)
    out, lse, *_ , err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


@pytest.mark.parametrize("q_len", [2, 3, 9, 16])
def test_few_rows_per_sequence(q_len):
    c = wl.random_case(500 + q_len, batch=6, Hq=32, Hkv=8, D=128, kv_range=(q_len, 900),
                       q_range=(q_len, q_len), pad_range=(0, 1), mask="causal")
    out, lse, *_ = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)


def test_longest_first_dispatch_edge_cases():
    """Several rows per sequence over a batch whose CTAs span more than one
    wave, so each CTA takes its sequence in longest-first order: sequences
    without rows, padding rows, equal lengths (ties broken by index)."""
    rng = np.random.default_rng(41)
    B, q_len = 40, 4
    kv = rng.integers(q_len, 3000, size=B, endpoint=True)
    kv[5:9] = 1234                 # ties
    q_rows = np.full(B, q_len, dtype=np.int64)
    q_real = np.full(B, q_len, dtype=np.int64)
    q_rows[[3, 17]] = 0
    q_real[[3, 17]] = 0            # sequences without rows
    q_real[[7, 30]] = 2            # two real rows and two padding rows
    c = wl.build_pool_case("longest_first", 41, kv, q_rows, q_real, 32, 8, 128, mask="causal")
    out, lse, *_, err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


@pytest.mark.parametrize("num_splits", [2, 5])
def test_tile_kernel_key_splits(num_splits):
    c = wl.random_case(401, batch=2, Hq=32, Hkv=8, D=128, kv_range=(600, 1500), q_range=(20, 64),
                       pad_range=(0, 3), mask="causal")
    out, lse, *_ = gpu_step(c, num_splits=num_splits)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)


def test_tile_kernel_f32_output_and_peaked():
    c = wl.random_case(402, batch=2, Hq=32, Hkv=8, D=128, kv_range=(300, 900), q_range=(30, 90),
                       mask="block_causal", causal_block=16, q_scale=6.0)
    out, lse, *_ = gpu_step(c, out_dtype=torch.float32)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)


def test_tile_kernel_matches_simt_kernel():
    c = wl.random_case(403, batch=3, Hq=32, Hkv=8, D=128, kv_range=(100, 1200), q_range=(5, 100),
                       pad_range=(0, 4), mask="causal")
    o1, l1, *_ = gpu_step(c)
    o2, l2, *_ = gpu_step(c, flags=pkv.PKV_FLAG_SIMT_ONLY)
    real = torch.from_numpy(real_row_mask(c)).to(DEV)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1[real] - l2[real]).abs().max().item() <= 1e-3


def test_tile_kernel_page_permutation_bit_identical():
    c = wl.random_case(404, batch=2, Hq=32, Hkv=8, D=128, kv_range=(200, 800), q_range=(10, 70),
                       mask="causal")
    out1, lse1, *_ = gpu_step(c)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(c.num_pages))
    k2 = torch.empty_like(c.k_pool); k2[perm] = c.k_pool
    v2 = torch.empty_like(c.v_pool); v2[perm] = c.v_pool
    t = c.block_table.clone()
    t[t >= 0] = perm[t[t >= 0].long()].to(torch.int32)
    s = c.slots.clone()
    s[s >= 0] = perm[s[s >= 0] // 32] * 32 + s[s >= 0] % 32
    c.k_pool, c.v_pool, c.block_table, c.slots = k2, v2, t, s
    out2, lse2, *_ = gpu_step(c)
    assert torch.equal(out1, out2)
    assert torch.equal(torch.nan_to_num(lse1, neginf=-1e30), torch.nan_to_num(lse2, neginf=-1e30))


def test_tile_kernel_nan_in_unused_slots_does_not_leak():
    """Pool slots past a sequence's last key (inside its last page) hold NaN:
    the zero probabilities of those keys must not turn into NaN outputs."""
    c = wl.random_case(405, batch=2, Hq=32, Hkv=8, D=128, kv_range=(100, 300), q_range=(8, 40),
                       mask="causal")
    table = c.block_table.numpy()
    for b in range(c.batch):
        L = int(c.kv_lens[b])
        last = table[b, (L - 1) // 32]
        c.k_pool[last, (L % 32 or 32):] = float("nan")
        c.v_pool[last, (L % 32 or 32):] = float("nan")
    out, lse, *_ = gpu_step(c)
    O, L_, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L_, c)


def _sample_rows(case, n=256, seed=0):
    rng = np.random.default_rng(seed)
    qi = case.q_indptr.numpy()
    rows = set()
    for b in range(case.batch):
        r0, r1 = qi[b], qi[b + 1]
        rows.update(range(r0, min(r1, r0 + 32)))
        rows.update(range(max(r0, r1 - 32), r1))
    rows.update(rng.integers(0, qi[-1], size=n).tolist())
    return sorted(rows)


def test_chunked_prefill_full_size_sampled():
    """Chunked causal prefill at full size: 8 sequences x 512 new tokens over
    2k-16k cached keys, 32/8 heads; the chunk's K/V is scattered first."""
    c = wl.chunked_prefill()
    out, lse, kg, vg, err = gpu_step(c)
    assert err == 0
    rows = _sample_rows(c)
    O, L, kb, vb = oracle_step(c, rows=rows)
    # the scatter is exact: compare the touched pages
    touched = np.unique(c.slots.numpy()[c.slots.numpy() >= 0] // 32)
    np.testing.assert_array_equal(orc.bf16_bits(kg.cpu())[touched], kb[touched])
    np.testing.assert_array_equal(orc.bf16_bits(vg.cpu())[touched], vb[touched])
    assert_attention_close(out, lse, O, L, c, rows=rows)


def test_block_causal_video_full_size_step():
    """The video workload's step: scatter 1560 staged rows (8 padding rows
    skipped), block-causal attention over prefix + history + current block
    (1568 rows, 40 heads), then rotate the rolling region left by one block."""
    c = wl.block_causal_video()
    out, lse, kg, vg, err = gpu_step(c)
    assert err == 0
    rows = _sample_rows(c, n=192)
    O, L, kb, vb = oracle_step(c, rows=rows)
    assert_attention_close(out, lse, O, L, c, rows=rows)
    np.testing.assert_array_equal(orc.bf16_bits(kg.cpu()), kb)
    # rotation of the rolling region [prefix, end) of K and V, left by one block
    e = c.extra
    H, D = c.num_kv_heads, c.head_dim
    first, n, sh = e["rotate_first_token"], e["rotate_tokens"], e["rotate_shift_tokens"]
    unit = 16
    tok_bytes = H * D * 2
    for pool, bits in ((kg, kb), (vg, vb)):
        flat = pool.view(torch.uint8).view(-1)
        region = flat[first * tok_bytes:(first + n) * tok_bytes]
        pkv.rotate_rows(region, sh * tok_bytes // unit, rows=1, cols=n * tok_bytes // unit,
                        row_stride=n * tok_bytes // unit, elem_size=unit)
        torch.cuda.synchronize()
        ref = orc.rotate_rows(bits.reshape(-1).view(np.uint8)[first * tok_bytes:(first + n) * tok_bytes]
                              .reshape(1, -1, unit), sh * tok_bytes // unit)
        np.testing.assert_array_equal(region.cpu().numpy().reshape(1, -1, unit), ref)


def test_shared_prefix_step_full_size():
    """Shared-prefix n-sample decode: 16 groups x 8 samples, 4096-token prefix
    attended once per group (the group's 8 rows as one query sequence, no
    mask), each sample's private tail attended by decode, states merged by
    LSE; equals attention over prefix ++ tail (oracle)."""
    c = wl.shared_prefix()
    e = c.extra
    k_pool, v_pool = c.k_pool.to(DEV), c.v_pool.to(DEV)
    pkv.kv_scatter_slots(c.new_k.to(DEV), c.new_v.to(DEV), c.slots.to(DEV), k_pool, v_pool)
    n, Hq, D = c.q.shape
    q = c.q.to(DEV)
    o_p = torch.empty(n, Hq, D, device=DEV)
    l_p = torch.empty(n, Hq, device=DEV)
    o_t = torch.empty(n, Hq, D, device=DEV)
    l_t = torch.empty(n, Hq, device=DEV)
    G = e["groups"]
    ws_p = pkv.paged_attention_workspace_size(G, e["samples"], Hq, 8, D, 4096)
    ws_p = torch.empty(max(ws_p, 1), dtype=torch.uint8, device=DEV)
    pkv.paged_attention(q, k_pool, v_pool, e["prefix_table"].to(DEV), e["prefix_lens"].to(DEV),
                        e["prefix_q_indptr"].to(DEV), o_p, q_real=e["prefix_q_real"].to(DEV),
                        lse=l_p, max_q_rows=e["samples"], max_kv_len=4096, mask="none",
                        workspace=ws_p)
    mt = int(e["tail_lens"].max())
    ws_t = torch.empty(pkv.paged_attention_workspace_size(n, 1, Hq, 8, D, mt), dtype=torch.uint8,
                       device=DEV)
    pkv.paged_attention(q, k_pool, v_pool, e["tail_table"].to(DEV), e["tail_lens"].to(DEV),
                        c.q_indptr.to(DEV), o_t, q_real=c.q_real.to(DEV), lse=l_t, max_q_rows=1,
                        max_kv_len=mt, workspace=ws_t)
    out = torch.empty(n, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(n, Hq, device=DEV)
    pkv.merge_attn_states(o_p, l_p, o_t, l_t, out, lse)
    torch.cuda.synchronize()
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)
