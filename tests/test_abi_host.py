"""CPU-only checks of the C ABI: the library builds for sm_103a, loads without
a GPU, exports every function include/pkv.h declares, and rejects bad
arguments on the host before touching CUDA (no compute calls here)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_189_gb300 import build as pkv_build
from paged_kv_cache_189_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first


@pytest.fixture(scope="module")
def L():
    pkv_build.build()
    return pkv.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"if", "sizeof", "defined", "extern"}
    return sorted({n for n in names if n not in keywords})


def test_exports_every_declared_function(L):
    decl = declared_functions()
    assert set(decl) == set(pkv.EXPORTED), decl
    for name in decl:
        assert hasattr(L, name), name


def test_status_strings(L):
    assert pkv.status_string(0) == "PKV_OK"
    assert pkv.status_string(pkv.PKV_ERR_UNSUPPORTED) == "PKV_ERR_UNSUPPORTED"


def _attn(L, **kw):
    a = dict(q=FAKE, qts=32 * 128, qhs=128, k=FAKE, v=FAKE, pages=10, ps=32, pstride=32 * 8 * 128,
             bt=FAKE, bts=4, kl=FAKE, qi=FAKE, qr=None, batch=2, mq=1, mk=100, hq=32, hkv=8,
             d=128, mask=1, cb=0, scale=0.0, out=FAKE, odt=0, lse=None, ws=None, wsb=0,
             splits=0, flags=0, err=None)
    a.update(kw)
    return L.paged_attention(a["q"], a["qts"], a["qhs"], a["k"], a["v"], a["pages"], a["ps"],
                             a["pstride"], a["bt"], a["bts"], a["kl"], a["qi"], a["qr"], a["batch"],
                             a["mq"], a["mk"], a["hq"], a["hkv"], a["d"], a["mask"], a["cb"],
                             a["scale"], a["out"], a["odt"], a["lse"], a["ws"], a["wsb"],
                             a["splits"], a["flags"], a["err"], None)


def test_attention_host_validation(L):
    assert _attn(L, ps=16) == pkv.PKV_ERR_UNSUPPORTED
    assert "page" in pkv.last_error()
    assert _attn(L, d=96) == pkv.PKV_ERR_UNSUPPORTED
    assert _attn(L, hq=30) == pkv.PKV_ERR_INVALID_ARG
    assert _attn(L, mask=2, cb=0) == pkv.PKV_ERR_INVALID_ARG
    assert _attn(L, mask=7) == pkv.PKV_ERR_INVALID_ARG
    assert _attn(L, bts=2, mk=100) == pkv.PKV_ERR_INVALID_ARG      # 100 keys need 4 pages
    assert _attn(L, pstride=100) == pkv.PKV_ERR_INVALID_ARG
    assert _attn(L, q=ctypes.c_void_p(0x1002)) == pkv.PKV_ERR_INVALID_ARG  # misaligned
    assert _attn(L, q=None) == pkv.PKV_ERR_INVALID_ARG
    assert _attn(L, flags=pkv.PKV_FLAG_CHECKED, err=None) == pkv.PKV_ERR_INVALID_ARG
    assert _attn(L, odt=pkv.PKV_F16) == pkv.PKV_ERR_UNSUPPORTED
    # the decode kernel needs a workspace (counters; partials past 512 keys)
    assert _attn(L, mk=3000, bts=94) == pkv.PKV_ERR_WORKSPACE
    assert _attn(L, mk=100) == pkv.PKV_ERR_WORKSPACE
    # empty problems return OK without touching the device
    assert _attn(L, batch=0) == pkv.PKV_OK
    assert _attn(L, mq=0) == pkv.PKV_OK


def test_workspace_size(L):
    # one split when everything fits in 512 keys: only the scheduling region
    # (counters and the planned unit order: one (split, row-head) pair per unit)
    small = pkv.paged_attention_workspace_size(64, 1, 32, 8, 128, 512)
    assert 64 * 8 * 4 + 64 * 8 * 8 < small <= 8192
    # the automatic split size aims at ~6 work units per resident CTA (3 per SM
    # on 152 SMs): 8193 keys x 512 (sequence, head) pairs / 2736 -> 1536 keys,
    # i.e. 6 splits
    ws = pkv.paged_attention_workspace_size(64, 1, 32, 8, 128, 8193)
    splits = 6
    states = 64 * 32 * splits
    assert ws >= states * 128 * 4 + states * 4 + 64 * 8 * 4
    # an explicit split count overrides it
    ws17 = pkv.paged_attention_workspace_size(64, 1, 32, 8, 128, 8193, num_splits=17)
    assert ws17 >= 64 * 32 * 17 * 129 * 4
    # the generic kernel (several query rows) needs none
    assert pkv.paged_attention_workspace_size(4, 16, 32, 8, 128, 8193,
                                              flags=pkv.PKV_FLAG_SIMT_ONLY) == 0
    assert pkv.paged_attention_workspace_size(0, 1, 32, 8, 128, 8193) == 0
    # one row per sequence with a head group of 8 or 16 (head_dim 128) takes the
    # tensor-core tile path: no decode scheduling region, and no split partials
    # for a grid of more than two waves (64 sequences x 8 heads = 512 CTAs)
    assert pkv.paged_attention_workspace_size(64, 1, 64, 8, 128, 8193) == 0
    assert pkv.paged_attention_workspace_size(64, 1, 128, 8, 128, 8193) == 0
    assert pkv.paged_attention_workspace_size(64, 1, 32, 8, 128, 8193) > 0   # group 4: decode kernel


def test_scatter_host_validation(L):
    def sc(**kw):
        a = dict(ks=FAKE, vs=FAKE, T=4, nsrc=4, h=2, d=64, ts=128, hs=64, sl=FAKE, sl2=None,
                 idx=None, kp=FAKE, vp=FAKE, pages=2, ps=32, pstride=32 * 128, dt=0, flags=0,
                 err=None)
        a.update(kw)
        return L.kv_scatter_slots(a["ks"], a["vs"], a["T"], a["nsrc"], a["h"], a["d"], a["ts"],
                                  a["hs"], a["sl"], a["sl2"], a["idx"], a["kp"], a["vp"],
                                  a["pages"], a["ps"], a["pstride"], a["dt"], a["flags"], a["err"],
                                  None)
    assert sc(T=0) == pkv.PKV_OK
    assert sc(sl=None) == pkv.PKV_ERR_INVALID_ARG
    assert sc(pstride=100) == pkv.PKV_ERR_INVALID_ARG
    assert sc(nsrc=2) == pkv.PKV_ERR_INVALID_ARG
    assert sc(dt=9) == pkv.PKV_ERR_INVALID_ARG
    assert sc(flags=pkv.PKV_FLAG_CHECKED) == pkv.PKV_ERR_INVALID_ARG
    assert sc(ks=ctypes.c_void_p(0x1001)) == pkv.PKV_ERR_INVALID_ARG


def test_rotate_and_merge_host_validation(L):
    assert L.rotate_rows(FAKE, 3, 10, 10, 3, 1, None) == pkv.PKV_ERR_UNSUPPORTED
    assert L.rotate_rows(FAKE, 0, 10, 10, 4, 1, None) == pkv.PKV_OK      # no rows: no launch
    assert L.rotate_rows(FAKE, 3, 1, 1, 4, 1, None) == pkv.PKV_OK        # one column: no launch
    assert L.rotate_rows(FAKE, 3, 10, 10, 4, 20, None) == pkv.PKV_OK     # shift = 0 mod cols
    assert L.rotate_rows(FAKE, 3, 10, 5, 4, 1, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.rotate_rows(None, 3, 10, 10, 4, 1, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.merge_attn_states(FAKE, FAKE, FAKE, FAKE, 0, 0, 4, 64, FAKE, 0, None, None) == pkv.PKV_OK
    assert L.merge_attn_states(FAKE, FAKE, FAKE, FAKE, 0, 3, 4, 66, FAKE, 0, None, None) == \
        pkv.PKV_ERR_UNSUPPORTED
    assert L.merge_attn_states(FAKE, None, FAKE, FAKE, 0, 3, 4, 64, FAKE, 0, None, None) == \
        pkv.PKV_ERR_INVALID_ARG


def test_causal_layout_host_validation(L):
    def lay(page=32, staged=100, block=30, com_cap=4 * 93, cur_cap=4 * 62, table=FAKE, row_stride=64,
            priv_stride=8, pin=0, window=0):
        return L.causal_layout(table, 10, FAKE, pin, window, staged, block, FAKE, priv_stride, page, FAKE,
                               row_stride, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, com_cap, FAKE, FAKE, cur_cap,
                               None, None)
    assert lay(page=16) == pkv.PKV_ERR_UNSUPPORTED
    assert lay(block=0) == pkv.PKV_ERR_INVALID_ARG
    assert lay(staged=0, table=None) == pkv.PKV_OK           # empty forward: nothing to do
    assert lay(table=None) == pkv.PKV_ERR_INVALID_ARG
    assert lay(com_cap=3 * 93) == pkv.PKV_ERR_INVALID_ARG    # 4 blocks need 4 x 93 entries
    assert lay(cur_cap=4 * 62 - 1) == pkv.PKV_ERR_INVALID_ARG
    assert lay(row_stride=0) == pkv.PKV_ERR_INVALID_ARG
    assert lay(pin=2 ** 31, window=1) == pkv.PKV_ERR_UNSUPPORTED


def test_plan_and_shared_prefix_host_validation(L):
    def plan(batch=8, max_pages=4, stride_bt=4, stride_out=16, table=FAKE):
        return L.plan_shared_prefix(table, stride_bt, FAKE, FAKE, batch, max_pages, FAKE, stride_out, FAKE,
                                    FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None)
    assert plan(batch=0, table=None) == pkv.PKV_OK
    assert plan(batch=1025) == pkv.PKV_ERR_UNSUPPORTED
    assert plan(table=None) == pkv.PKV_ERR_INVALID_ARG
    assert plan(stride_bt=3) == pkv.PKV_ERR_INVALID_ARG      # table narrower than max_pages
    assert plan(stride_out=0) == pkv.PKV_ERR_INVALID_ARG

    def spa(D=128, Hq=32, Hkv=8, page=32, out=FAKE, row_stride=64, max_keys=2048, ws=None, ws_bytes=0):
        return L.shared_prefix_attention(FAKE, 4096, 128, FAKE, FAKE, 100, page, 32 * Hkv * 128, FAKE, row_stride,
                                         FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 1, 8, max_keys, Hq, Hkv, D,
                                         0.0, out, pkv.PKV_BF16, None, ws, ws_bytes, 0, 0, None, None)
    assert spa(D=96) == pkv.PKV_ERR_UNSUPPORTED              # tensor-core tiles: head_dim 64 or 128
    assert spa(Hq=8 * 65) == pkv.PKV_ERR_UNSUPPORTED         # a group of 65 query heads
    assert spa(page=16) == pkv.PKV_ERR_UNSUPPORTED
    assert spa(out=None) == pkv.PKV_ERR_INVALID_ARG
    assert spa(row_stride=63) == pkv.PKV_ERR_INVALID_ARG     # row narrower than max_group_keys
    assert pkv.shared_prefix_attention_workspace_size(16, 1, 8, 2048, 32, 8, 128) >= 0


def test_plan_follows_the_sm_count(L):
    """The split planner sizes its choice by the GPU's SM count, so the same
    bounds plan differently on GPUs of different sizes; with no device to query
    (this host) the workspace size is the 152-SM plan's."""
    # exact-window denoising forward: 25 CTAs of two 32-token tiles x 8 K/V
    # heads = 200 CTAs.  On 152 SMs two waves, so 3 key splits (4 waves of
    # thirds, 1.39 against 2 unsplit); on 200 SMs one wave, no split; on 100
    # SMs exactly two waves that no split count shortens by 10 %
    # (with the one-CTA-per-tile grid; by default the stream-K schedule)
    grid = pkv.PKV_FLAG_TILE_GRID
    p152 = pkv.plan_attention(1, 1576, 32, 8, 128, 39518, flags=grid, num_sms=152)
    p200 = pkv.plan_attention(1, 1576, 32, 8, 128, 39518, flags=grid, num_sms=200)
    p100 = pkv.plan_attention(1, 1576, 32, 8, 128, 39518, flags=grid, num_sms=100)
    assert p152["kernel"] == p200["kernel"] == pkv.PKV_KERNEL_TILE
    assert (p152["splits"], p200["splits"], p100["splits"]) == (3, 1, 1)
    assert p152["workspace_bytes"] > 0 and p200["workspace_bytes"] == 0
    # stream-K only on request (one persistent CTA per SM, each with two
    # fragment slots of 256 rows x 128 f32 + LSE): the video step's 280 tile
    # pairs keep the grid by default
    v152 = pkv.plan_attention(1, 1568, 40, 40, 128, 7800, num_sms=152)
    assert v152["kernel"] == pkv.PKV_KERNEL_TILE and v152["splits"] == 1
    vsk = pkv.plan_attention(1, 1568, 40, 40, 128, 7800, flags=pkv.PKV_FLAG_STREAM_K, num_sms=152)
    assert vsk["kernel"] == pkv.PKV_KERNEL_TILE_STREAM_K
    assert vsk["splits"] == 1 and vsk["split_keys"] >= 7800
    # forced stream-K: the workspace follows the SM count
    sk = pkv.PKV_FLAG_STREAM_K
    s152 = pkv.plan_attention(1, 1576, 32, 8, 128, 39518, flags=sk, num_sms=152)
    s120 = pkv.plan_attention(1, 1576, 32, 8, 128, 39518, flags=sk, num_sms=120)
    assert s152["kernel"] == s120["kernel"] == pkv.PKV_KERNEL_TILE_STREAM_K
    frag = 2 * 256 * (128 + 1) * 4
    assert s152["workspace_bytes"] - s120["workspace_bytes"] >= 32 * frag
    # by default the exact-window forward keeps its 3 key splits
    assert pkv.plan_attention(1, 1576, 32, 8, 128, 39518, num_sms=152)["splits"] == 3
    # tensor-core tiles for head_dim 64 and for any head group up to 64; the
    # generic kernel past that
    assert pkv.plan_attention(4, 300, 32, 8, 64, 4000)["kernel"] == pkv.PKV_KERNEL_TILE
    for hq, hkv in ((24, 8), (40, 8), (48, 8), (56, 8), (96, 8), (64, 1)):
        assert pkv.plan_attention(4, 300, hq, hkv, 128, 4000)["kernel"] == pkv.PKV_KERNEL_TILE, (hq, hkv)
        assert pkv.plan_attention(4, 1, hq, hkv, 128, 4000)["kernel"] == pkv.PKV_KERNEL_TILE, (hq, hkv)
    assert pkv.plan_attention(4, 300, 65, 1, 128, 4000)["kernel"] == pkv.PKV_KERNEL_SIMT
    assert pkv.plan_attention(4, 1, 32, 8, 64, 4000)["kernel"] == pkv.PKV_KERNEL_DECODE
    # an explicit split count keeps the one-CTA-per-tile grid
    assert pkv.plan_attention(1, 1568, 40, 40, 128, 7800, num_splits=2,
                              flags=pkv.PKV_FLAG_STREAM_K)["kernel"] == pkv.PKV_KERNEL_TILE
    # decode: ~6 work units per resident CTA (3 per SM): 8193 keys x 512
    # (sequence, head) pairs / (6 x 456) -> 1536 keys per split on 152 SMs,
    # 3072 on 76
    d152 = pkv.plan_attention(64, 1, 32, 8, 128, 8193, num_sms=152)
    d76 = pkv.plan_attention(64, 1, 32, 8, 128, 8193, num_sms=76)
    assert d152["kernel"] == d76["kernel"] == pkv.PKV_KERNEL_DECODE
    assert (d152["split_keys"], d152["splits"]) == (1536, 6)
    assert (d76["split_keys"], d76["splits"]) == (3072, 3)
    assert d76["workspace_bytes"] < d152["workspace_bytes"]
    # workspace_size plans for the current device (here: none -> 152 SMs)
    assert pkv.paged_attention_workspace_size(64, 1, 32, 8, 128, 8193) == d152["workspace_bytes"]
    assert pkv.paged_attention_workspace_size(1, 1576, 32, 8, 128, 39518) == p152["workspace_bytes"]
    assert pkv.paged_attention_workspace_size(1, 1568, 40, 40, 128, 7800) == v152["workspace_bytes"]
    # bad arguments are refused on the host
    with pytest.raises(pkv.PkvError):
        pkv.plan_attention(4, 1, 30, 8, 128, 100)
