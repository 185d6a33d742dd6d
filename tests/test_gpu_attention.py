"""GPU parity of paged_attention (through the C-ABI) against the fp64 oracle.

Tolerances (bf16 output vs fp64): max-abs 1e-2, mean-abs 1e-3, LSE 1e-3.
Covers the decode kernel (split-KV and single split), the generic SIMT
kernel, padding rows, empty sequences, page-permutation invariance (bit
identical GPU outputs), checked mode, and the full-size decode workload."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_cache_189_gb300 import pkv, workloads as wl
from pkv_testutil import assert_attention_close, gpu_step, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_tiny_decode_workload():
    c = wl.tiny_decode()
    out, lse, kg, vg, err = gpu_step(c)
    O, L, kb, vb = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)
    np.testing.assert_array_equal(orc.bf16_bits(kg.cpu()), kb)
    np.testing.assert_array_equal(orc.bf16_bits(vg.cpu()), vb)


def test_tiny_decode_scatter_into_free_slots():
    """The tiny workload's standalone scatter of two new rows into random free
    slots: bit exact, and attention over the untouched sequences unchanged."""
    c = wl.tiny_decode()
    free = c.extra["free_slots"]
    kg, vg = c.k_pool.to(DEV), c.v_pool.to(DEV)
    pkv.kv_scatter_slots(c.new_k.to(DEV), c.new_v.to(DEV), free.to(DEV), kg, vg)
    ko, vo, _ = orc.kv_scatter_slots(orc.bf16_bits(c.new_k), orc.bf16_bits(c.new_v), free.numpy(),
                                     orc.bf16_bits(c.k_pool), orc.bf16_bits(c.v_pool))
    np.testing.assert_array_equal(orc.bf16_bits(kg.cpu()), ko)
    np.testing.assert_array_equal(orc.bf16_bits(vg.cpu()), vo)


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 4, 128), (8, 8, 128), (4, 2, 64),
                                      (16, 4, 64), (6, 6, 64),
                                      # head groups of 8 and 16: the tile kernel
                                      (64, 8, 128), (32, 2, 128)])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_random(Hq, Hkv, D, num_splits):
    c = wl.random_case(100 + Hq + D + num_splits, batch=7, Hq=Hq, Hkv=Hkv, D=D,
                       kv_range=(1, 1500))
    out, lse, *_ , err = gpu_step(c, num_splits=num_splits)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


def test_decode_f32_output_and_padding_rows():
    """One-row sequences whose row is padding (q_real = 0) come back zero."""
    c = wl.random_case(7, batch=6, Hq=32, Hkv=8, D=128, kv_range=(30, 700))
    c.q_real[1] = 0
    c.q_real[4] = 0
    c.slots[1] = -1
    c.slots[4] = -1
    out, lse, *_ , err = gpu_step(c, out_dtype=torch.float32)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)
    assert (out[1] == 0).all() and (out[4] == 0).all()


def test_decode_peaked_queries():
    """Scaled-up queries concentrate the softmax, so a wrong visible set or a
    wrong page shows up beyond the tolerance even at long lengths."""
    c = wl.random_case(11, batch=5, Hq=32, Hkv=8, D=128, kv_range=(1000, 5000), q_scale=8.0)
    out, lse, *_ = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)


def test_decode_page_permutation_bit_identical():
    c = wl.random_case(12, batch=4, Hq=32, Hkv=8, D=128, kv_range=(100, 3000))
    out1, lse1, *_ = gpu_step(c)
    rng = np.random.default_rng(3)
    perm = torch.from_numpy(rng.permutation(c.num_pages))
    k2 = torch.empty_like(c.k_pool); k2[perm] = c.k_pool
    v2 = torch.empty_like(c.v_pool); v2[perm] = c.v_pool
    t = c.block_table.clone()
    t[t >= 0] = perm[t[t >= 0].long()].to(torch.int32)
    s = c.slots.clone()
    s[s >= 0] = perm[s[s >= 0] // 32] * 32 + s[s >= 0] % 32
    c.k_pool, c.v_pool, c.block_table, c.slots = k2, v2, t, s
    out2, lse2, *_ = gpu_step(c)
    assert torch.equal(out1, out2)
    assert torch.equal(lse1, lse2)


def test_decode_zero_length_and_empty_sequences():
    c = wl.random_case(13, batch=4, Hq=8, Hkv=2, D=128, kv_range=(5, 60))
    # sequence 2 has no keys at all (its only row is padding)
    c.kv_lens[2] = 0
    c.q_real[2] = 0
    c.slots[2] = -1
    out, lse, *_ = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)


def test_decode_group_8_full_size():
    """Single-row decode with 64 query / 8 K/V heads (head group 8) over the
    GQA decode lengths, through the tensor-core tile kernel, every row against
    the oracle."""
    c = wl.gqa_decode(Hq=64, Hkv=8)
    out, lse, kg, vg, err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


def test_decode_planned_order_edge_cases():
    """A batch whose decode units outnumber the persistent CTAs, so they are
    taken in the planned order (full splits first, partial splits longest
    first), with the planner's edge cases: rows that attend nothing (padding),
    sequences without rows, lengths ending exactly on a split boundary, a
    one-key row."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, D = 96, 32, 8, 128
    kv = rng.integers(1, 6000, size=B, endpoint=True)
    # the automatic split size for this batch on this device's SM count (~6
    # units per resident CTA, at least 512 keys)
    sk = pkv.plan_attention(B, 1, Hq, Hkv, D, int(kv.max()))["split_keys"]
    assert 3 * sk <= int(kv.max())
    kv[0:4] = [sk, 2 * sk, 3 * sk, 1]
    q_rows = np.ones(B, dtype=np.int64)
    q_real = np.ones(B, dtype=np.int64)
    q_rows[[10, 11]] = 0
    q_real[[10, 11]] = 0          # sequences without rows
    q_real[[20, 21, 22]] = 0      # padding rows: attend nothing, come back zero
    c = wl.build_pool_case("planned_edges", 31, kv, q_rows, q_real, Hq, Hkv, D, mask="causal")
    out, lse, *_, err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


def test_decode_checked_mode_bad_page_flags_error():
    c = wl.random_case(14, batch=3, Hq=8, Hkv=2, D=128, kv_range=(40, 90))
    c.block_table[1, 0] = c.num_pages + 5
    *_, err = gpu_step(c, scatter=False, checked=True)
    assert err & pkv.PKV_ERRBIT_PAGE


def test_decode_graph_capture_replay():
    """The call is capturable: a graph replays with new device contents."""
    c = wl.random_case(15, batch=8, Hq=32, Hkv=8, D=128, kv_range=(600, 2000))
    k_pool, v_pool = c.k_pool.to(DEV), c.v_pool.to(DEV)
    q = c.q.to(DEV)
    bt, kl, qi, qr = (c.block_table.to(DEV), c.kv_lens.to(DEV), c.q_indptr.to(DEV),
                      c.q_real.to(DEV))
    rows, Hq, D = q.shape
    out = torch.empty(rows, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(rows, Hq, device=DEV)
    mk = c.max_kv_len
    ws = torch.empty(pkv.paged_attention_workspace_size(c.batch, 1, Hq, 8, D, mk), dtype=torch.uint8,
                     device=DEV)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        pkv.paged_attention(q, k_pool, v_pool, bt, kl, qi, out, q_real=qr, lse=lse, max_q_rows=1,
                            max_kv_len=mk, workspace=ws)  # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            pkv.paged_attention(q, k_pool, v_pool, bt, kl, qi, out, q_real=qr, lse=lse,
                                max_q_rows=1, max_kv_len=mk, workspace=ws)
    q2 = wl.randn_bf16(tuple(q.shape), torch.Generator().manual_seed(99))
    q.copy_(q2.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    c.q = q2
    O, L, *_ = oracle_step(c, scatter=False)
    assert_attention_close(out, lse, O, L, c)


@pytest.mark.parametrize("mask,cb", [("causal", 0), ("block_causal", 5), ("none", 0)])
def test_simt_kernel_multi_row(mask, cb):
    c = wl.random_case(20, batch=4, Hq=8, Hkv=2, D=128, kv_range=(20, 400), q_range=(1, 40),
                       pad_range=(0, 5), mask=mask, causal_block=cb)
    out, lse, *_ = gpu_step(c, flags=pkv.PKV_FLAG_SIMT_ONLY)
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)


def test_simt_kernel_matches_decode_kernel():
    c = wl.random_case(21, batch=6, Hq=32, Hkv=8, D=128, kv_range=(50, 2500))
    o1, l1, *_ = gpu_step(c)
    o2, l2, *_ = gpu_step(c, flags=pkv.PKV_FLAG_SIMT_ONLY)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_gqa_decode_full_size():
    """The GQA decode workload at its full size (64 sequences of up to 8193
    keys, 32/8 heads): every output row against the oracle."""
    c = wl.gqa_decode()
    out, lse, kg, vg, err = gpu_step(c)
    O, L, *_ = oracle_step(c)
    assert err == 0
    assert_attention_close(out, lse, O, L, c)


def _planned_units(ws, B, Hkv):
    """The decode scheduling region at the start of the workspace: the unit
    count after the ticket and split counters, then the unit list of (split,
    sequence * Hkv + head) pairs after the sequence order."""
    a256 = lambda n: -(-n // 256) * 256
    raw = ws.cpu().numpy()
    off_total = a256((B * Hkv + 1) * 4)
    total = int(raw[off_total:off_total + 4].view(np.int32)[0])
    off_list = off_total + 256 + a256(B * 4)
    lst = raw[off_list:off_list + total * 8].view(np.int32).reshape(total, 2)
    return total, lst


@pytest.mark.parametrize("B", [96, 128, 200])
def test_decode_planned_unit_order(B):
    """The planned order itself, read back from the workspace: every unit once;
    the full splits first, split-major, sequences with more full splits first;
    then the partial last splits, longest first (exactly up to 128 sequences,
    by 1/1024-split buckets above); then the rows without keys.  Outputs
    against the oracle as well."""
    rng = np.random.default_rng(53 + B)
    Hq, Hkv, D = 32, 8, 128
    kv = rng.integers(1, 7000, size=B, endpoint=True)
    kv[5] = 7000                              # the longest row fixes the split size
    sk = pkv.plan_attention(B, 1, Hq, Hkv, D, 7000)["split_keys"]
    assert sk < 7000
    kv[0:5] = [sk, 7000 // sk * sk, 1, sk + 1, sk - 1]   # split boundaries, one key
    kv[40:43] = 1234                          # equal lengths
    q_rows = np.ones(B, dtype=np.int64)
    q_real = np.ones(B, dtype=np.int64)
    q_rows[[10, 11]] = 0
    q_real[[10, 11]] = 0                      # sequences without rows
    q_real[[20, 21, 22]] = 0                  # rows without keys
    c = wl.build_pool_case("unit_order", 53 + B, kv, q_rows, q_real, Hq, Hkv, D, mask="causal")
    plan = pkv.plan_attention(B, 1, Hq, Hkv, D, c.max_kv_len)
    assert plan["kernel"] == pkv.PKV_KERNEL_DECODE and plan["split_keys"] == sk
    k_pool, v_pool = c.k_pool.to(DEV), c.v_pool.to(DEV)
    pkv.kv_scatter_slots(c.new_k.to(DEV), c.new_v.to(DEV), c.slots.to(DEV), k_pool, v_pool)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, Hq), float("nan"), device=DEV)
    ws = torch.zeros(plan["workspace_bytes"], dtype=torch.uint8, device=DEV)
    pkv.paged_attention(c.q.to(DEV), k_pool, v_pool, c.block_table.to(DEV), c.kv_lens.to(DEV),
                        c.q_indptr.to(DEV), out, q_real=c.q_real.to(DEV), lse=lse, max_q_rows=1,
                        max_kv_len=c.max_kv_len, workspace=ws)
    torch.cuda.synchronize()
    O, L, *_ = oracle_step(c)
    assert_attention_close(out, lse, O, L, c)

    # the units of the call: keys per row (0 for a row without keys; none for a
    # sequence without rows), cut into splits of sk keys
    keys = {b: (int(kv[b]) if q_real[b] > 0 else 0) for b in range(B) if q_rows[b] > 0}
    expect = set()
    for b, n in keys.items():
        for h in range(Hkv):
            for s in range(max(1, -(-n // sk))):
                expect.add((s, b * Hkv + h))
    total, lst = _planned_units(ws, B, Hkv)
    got = [tuple(int(v) for v in e) for e in lst]
    assert total == len(expect) and len(set(got)) == total and set(got) == expect

    f = {b: n // sk for b, n in keys.items()}
    r = {b: n % sk for b, n in keys.items()}
    kind = []
    for s, bh in got:
        b = bh // Hkv
        kind.append(0 if s < f[b] else (1 if r[b] > 0 else 2))
    assert kind == sorted(kind)                       # full, then partial, then no keys
    full = [(s, bh // Hkv) for (s, bh), k in zip(got, kind) if k == 0]
    assert [s for s, _ in full] == sorted(s for s, _ in full)   # split-major
    for s in set(x for x, _ in full):
        fs = [f[b] for x, b in full if x == s]
        assert fs == sorted(fs, reverse=True)                   # more full splits first
    part = [r[bh // Hkv] for (s, bh), k in zip(got, kind) if k == 1]
    key = part if B <= 128 else [x * 1024 // sk for x in part]
    assert key == sorted(key, reverse=True)                     # longest partial first
