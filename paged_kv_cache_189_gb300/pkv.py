"""Python binding of the C ABI in ``include/pkv.h`` (ctypes).

Argument marshalling only: every function here turns torch tensors into the
pointers, sizes and strides the C entry point takes and raises on a non-OK
status.  All arithmetic runs in the CUDA kernels of ``libpkv.so``; if the
library has not been built this module raises instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA = range(5)
PKV_BF16, PKV_F16, PKV_F32 = range(3)
MASKS = {"none": 0, "causal": 1, "block_causal": 2}
PKV_FLAG_CHECKED = 0x1
PKV_FLAG_SIMT_ONLY = 0x2
PKV_FLAG_TEST_WAIT_TIMEOUT = 0x4
PKV_FLAG_TILE_GRID = 0x8
PKV_FLAG_STREAM_K = 0x10
PKV_ERRBIT_SLOT, PKV_ERRBIT_SRC, PKV_ERRBIT_PAGE, PKV_ERRBIT_LEN, PKV_ERRBIT_TIMEOUT = (
    0x1, 0x2, 0x4, 0x8, 0x10)

# every symbol include/pkv.h declares
EXPORTED = ("pkv_status_string", "pkv_last_error", "kv_scatter_slots",
            "paged_attention_workspace_size", "paged_attention", "merge_attn_states",
            "rotate_rows", "paged_attention_no_alloc", "rope_write_kv_paged", "copy_kv_slots",
            "causal_layout", "plan_shared_prefix", "shared_prefix_attention",
            "shared_prefix_attention_workspace_size", "pkv_plan_attention")
NO_ALLOC_SCRATCH_BYTES = 32 << 20

_vp, _i64, _i32, _u32, _f32, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_uint, ctypes.c_float, ctypes.c_size_t)
_SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_i32]),
    "pkv_last_error": (ctypes.c_char_p, []),
    "kv_scatter_slots": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _i64, _i64, _vp, _vp, _vp,
                                _vp, _vp, _i64, _i32, _i64, _i32, _u32, _vp, _vp]),
    "paged_attention_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _u32]),
    "pkv_plan_attention": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _u32, _i32, _vp, _vp, _vp,
                                  _vp]),
    "paged_attention": (_i32, [_vp, _i64, _i64, _vp, _vp, _i64, _i32, _i64, _vp, _i64, _vp, _vp,
                               _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp,
                               _i32, _vp, _vp, _sz, _i32, _u32, _vp, _vp]),
    "paged_attention_no_alloc": (_i32, [_vp, _i64, _i64, _vp, _vp, _i64, _i32, _i64, _vp, _i64,
                                        _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                        _i32, _f32, _vp, _i32, _vp, _i32, _u32, _vp, _vp]),
    "merge_attn_states": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _vp, _i32, _vp,
                                 _vp]),
    "rotate_rows": (_i32, [_vp, _i64, _i64, _i64, _i32, _i64, _vp]),
    "rope_write_kv_paged": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _i64, _i64, _i64, _i32, _i32,
                                   _vp, _vp, _i64, _vp, _vp, _vp, _i64, _i32, _i64, _u32, _vp,
                                   _vp]),
    "copy_kv_slots": (_i32, [_vp, _vp, _i32, _i64, _i64, _i32, _i64, _i32, _i32, _i32, _vp, _vp,
                             _i64, _u32, _vp, _vp]),
    "causal_layout": (_i32, [_vp, _i64, _vp, _i64, _i64, _i32, _i32, _vp, _i32, _i32, _vp, _i64,
                             _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp]),
    "plan_shared_prefix": (_i32, [_vp, _i64, _vp, _vp, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp]),
    "shared_prefix_attention_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "shared_prefix_attention": (_i32, [_vp, _i64, _i64, _vp, _vp, _i64, _i32, _i64, _vp, _i64, _vp, _vp,
                                       _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                       _i32, _f32, _vp, _i32, _vp, _vp, _sz, _i32, _u32, _vp, _vp]),
}

_lib = None


class PkvError(RuntimeError):
    def __init__(self, func, status, message):
        self.status = status
        super().__init__(f"{func}: {status_string(status)}: {message}")


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded library with its C signatures declared."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libpkv.so is not built ({p}); call __graft_entry__.build() or "
                           "paged_kv_cache_189_gb300.build.build() first")
    L = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = L
    return L


def status_string(status: int) -> str:
    return lib().pkv_status_string(status).decode()


def last_error() -> str:
    return lib().pkv_last_error().decode()


def _check(func, status):
    if status != PKV_OK:
        raise PkvError(func, status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(stream)


def _dtype(t):
    return {torch.bfloat16: PKV_BF16, torch.float16: PKV_F16, torch.float32: PKV_F32}[t.dtype]


def _pool_geometry(pool):
    """[num_pages, page_size, Hkv, D] with dense slots; page stride may be larger."""
    assert pool.dim() == 4, "pool must be [num_pages, page_size, num_kv_heads, head_dim]"
    n, P, H, D = pool.shape
    if pool.stride(3) != 1 or pool.stride(2) != D or pool.stride(1) != H * D:
        raise ValueError("pool slots must be dense [num_kv_heads, head_dim] rows")
    return n, P, H, D, pool.stride(0)


# ----------------------------------------------------------------------------
def kv_scatter_slots(k_src, v_src, slots, k_pool, v_pool, slots2=None, src_idx=None,
                     checked=False, err=None, stream=None):
    """Write rows of ``k_src``/``v_src`` ``[T, Hkv, D]`` (any token/head stride,
    unit dim stride) into pool slots ``slots`` (and ``slots2``) in place."""
    assert k_src.stride() == v_src.stride() and k_src.shape == v_src.shape
    assert k_src.stride(2) == 1
    n, P, H, D, page_stride = _pool_geometry(k_pool)
    assert v_pool.shape == k_pool.shape and v_pool.stride() == k_pool.stride()
    T = slots.numel()
    st = lib().kv_scatter_slots(
        _ptr(k_src), _ptr(v_src), T, k_src.shape[0], H, D, k_src.stride(0), k_src.stride(1),
        _ptr(slots), _ptr(slots2), _ptr(src_idx), _ptr(k_pool), _ptr(v_pool), n, P, page_stride,
        _dtype(k_pool), PKV_FLAG_CHECKED if checked else 0, _ptr(err), _stream(stream))
    _check("kv_scatter_slots", st)


def paged_attention_workspace_size(batch, max_q_rows, num_q_heads, num_kv_heads, head_dim,
                                   max_kv_len, num_splits=0, flags=0) -> int:
    return int(lib().paged_attention_workspace_size(batch, max_q_rows, num_q_heads, num_kv_heads,
                                                    head_dim, max_kv_len, num_splits, flags))


PKV_KERNEL_NONE, PKV_KERNEL_DECODE, PKV_KERNEL_TILE, PKV_KERNEL_SIMT, PKV_KERNEL_TILE_STREAM_K = range(5)


def plan_attention(batch, max_q_rows, num_q_heads, num_kv_heads, head_dim, max_kv_len,
                   num_splits=0, flags=0, num_sms=0) -> dict:
    """The launch plan of ``paged_attention`` for these host bounds on a GPU
    with ``num_sms`` SMs (0: the current device's): kernel, splits, keys per
    split and workspace bytes."""
    k, s, sk, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    st = lib().pkv_plan_attention(batch, max_q_rows, num_q_heads, num_kv_heads, head_dim, max_kv_len,
                                  num_splits, flags, num_sms, ctypes.byref(k), ctypes.byref(s),
                                  ctypes.byref(sk), ctypes.byref(ws))
    _check("pkv_plan_attention", st)
    return {"kernel": k.value, "splits": s.value, "split_keys": sk.value, "workspace_bytes": ws.value}


def paged_attention(q, k_pool, v_pool, block_table, kv_lens, q_indptr, out, *, q_real=None,
                    lse=None, batch=None, max_q_rows, max_kv_len, mask="causal",
                    causal_block=0, scale=0.0, workspace=None, num_splits=0, flags=0, err=None,
                    stream=None):
    """Paged attention of packed query rows ``q [rows, Hq, D]`` (bf16) into
    ``out [rows, Hq, D]`` (bf16 or f32) and ``lse [rows, Hq]`` (f32)."""
    n, P, H, D, page_stride = _pool_geometry(k_pool)
    assert v_pool.shape == k_pool.shape and v_pool.stride() == k_pool.stride()
    assert q.stride(2) == 1 and out.is_contiguous()
    if batch is None:
        batch = kv_lens.numel()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_attention(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k_pool), _ptr(v_pool), n, P, page_stride,
        _ptr(block_table), block_table.stride(0), _ptr(kv_lens), _ptr(q_indptr), _ptr(q_real),
        batch, max_q_rows, max_kv_len, q.shape[1], H, D, MASKS[mask], causal_block,
        float(scale), _ptr(out), _dtype(out), _ptr(lse), _ptr(workspace), ws_bytes, num_splits,
        flags, _ptr(err), _stream(stream))
    _check("paged_attention", st)


def paged_attention_no_alloc(q, k_pool, v_pool, block_table, kv_lens, q_indptr, out, *,
                             q_real=None, lse=None, batch=None, max_q_rows, max_kv_len,
                             mask="causal", causal_block=0, scale=0.0, num_splits=0, flags=0,
                             err=None, stream=None):
    """``paged_attention`` without a workspace argument, for callers that
    cannot allocate: the scratch is the library's fixed device array of
    ``NO_ALLOC_SCRATCH_BYTES`` (see include/pkv.h).  Calls on one device share
    it, so they must not overlap on the GPU."""
    n, P, H, D, page_stride = _pool_geometry(k_pool)
    assert v_pool.shape == k_pool.shape and v_pool.stride() == k_pool.stride()
    assert q.stride(2) == 1 and out.is_contiguous()
    if batch is None:
        batch = kv_lens.numel()
    st = lib().paged_attention_no_alloc(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k_pool), _ptr(v_pool), n, P, page_stride,
        _ptr(block_table), block_table.stride(0), _ptr(kv_lens), _ptr(q_indptr), _ptr(q_real),
        batch, max_q_rows, max_kv_len, q.shape[1], H, D, MASKS[mask], causal_block,
        float(scale), _ptr(out), _dtype(out), _ptr(lse), num_splits, flags, _ptr(err),
        _stream(stream))
    _check("paged_attention_no_alloc", st)


def merge_attn_states(o_a, lse_a, o_b, lse_b, o_out, lse_out=None, stream=None):
    """Exact LSE merge of two states ``[rows, heads, D]`` into ``o_out``."""
    rows, heads, D = o_a.shape
    assert o_b.shape == o_a.shape and o_out.shape == o_a.shape and o_a.dtype == o_b.dtype
    st = lib().merge_attn_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _dtype(o_a),
                                 rows, heads, D, _ptr(o_out), _dtype(o_out), _ptr(lse_out),
                                 _stream(stream))
    _check("merge_attn_states", st)


def rotate_rows(x, shift, rows=None, cols=None, row_stride=None, elem_size=None, stream=None):
    """Rotate every row of ``x`` left by ``shift`` elements in place.  By
    default ``x`` is viewed as ``[rows, cols]`` of its own element type."""
    if rows is None:
        if x.dim() == 1:
            rows, cols, row_stride = 1, x.shape[0], x.shape[0]
        else:
            assert x.dim() == 2 and x.stride(1) == 1
            rows, cols, row_stride = x.shape[0], x.shape[1], x.stride(0)
        elem_size = x.element_size()
    st = lib().rotate_rows(_ptr(x), rows, cols, row_stride, elem_size, shift, _stream(stream))
    _check("rotate_rows", st)


def rope_write_kv_paged(q, k_src, v_src, positions, cos_sin, slots, k_pool, v_pool,
                        checked=False, err=None, stream=None):
    """Rotate ``q [T, Hq, D]`` in place and write the rotated ``k_src`` and the
    ``v_src`` rows ``[T, Hkv, D]`` into pool slots ``slots`` (NeoX pairs,
    angles from the table ``cos_sin [max_position, D]``)."""
    assert q.stride(2) == 1 and k_src.stride(2) == 1 and k_src.stride() == v_src.stride()
    n, P, H, D, page_stride = _pool_geometry(k_pool)
    assert v_pool.shape == k_pool.shape and v_pool.stride() == k_pool.stride()
    assert cos_sin.dtype == torch.float32 and cos_sin.is_contiguous() and cos_sin.shape[1] == D
    st = lib().rope_write_kv_paged(
        _ptr(q), q.stride(0), q.stride(1), q.shape[1], _ptr(k_src), _ptr(v_src), k_src.stride(0),
        k_src.stride(1), q.shape[0], H, D, _ptr(positions), _ptr(cos_sin), cos_sin.shape[0],
        _ptr(slots), _ptr(k_pool), _ptr(v_pool), n, P, page_stride,
        PKV_FLAG_CHECKED if checked else 0, _ptr(err), _stream(stream))
    _check("rope_write_kv_paged", st)


def copy_kv_slots(k_pools, v_pools, src_slots, dst_slots, checked=False, err=None, stream=None):
    """Copy slot rows ``src -> dst`` in every layer of ``k_pools``/``v_pools``
    ``[layers, pages, P, Hkv, D]`` (a 4-D pool is one layer); negative entries
    are skipped."""
    if k_pools.dim() == 4:
        k_pools, v_pools = k_pools.unsqueeze(0), v_pools.unsqueeze(0)
    layers = k_pools.shape[0]
    n, P, H, D, page_stride = _pool_geometry(k_pools[0])
    assert v_pools.shape == k_pools.shape and v_pools.stride() == k_pools.stride()
    st = lib().copy_kv_slots(_ptr(k_pools), _ptr(v_pools), layers, k_pools.stride(0), n, P,
                             page_stride, H, D, _dtype(k_pools), _ptr(src_slots), _ptr(dst_slots),
                             src_slots.numel(), PKV_FLAG_CHECKED if checked else 0, _ptr(err),
                             _stream(stream))
    _check("copy_kv_slots", st)


LAYOUT_COMMITTED_PER_BLOCK = 93
LAYOUT_CURRENT_PER_BLOCK = 62


def causal_layout_buffers(num_staged, block_size, row_stride, device="cuda"):
    """Output tensors of :func:`causal_layout` for a forward of ``num_staged``
    tokens in blocks of ``block_size`` (allocated here, by the caller's side)."""
    import torch
    nb = (num_staged + block_size - 1) // block_size
    i32 = dict(dtype=torch.int32, device=device)
    i64 = dict(dtype=torch.int64, device=device)
    return dict(rows=torch.full((nb, row_stride), -1, **i32), kv_lens=torch.zeros(nb, **i32),
                q_indptr=torch.zeros(nb + 1, **i32), staged_slots=torch.full((num_staged,), -1, **i64),
                staged_slots2=torch.full((num_staged,), -1, **i64),
                committed_src=torch.full((nb * LAYOUT_COMMITTED_PER_BLOCK,), -1, **i64),
                committed_dst=torch.full((nb * LAYOUT_COMMITTED_PER_BLOCK,), -1, **i64),
                current_src_idx=torch.full((nb * LAYOUT_CURRENT_PER_BLOCK,), -1, **i64),
                current_dst=torch.full((nb * LAYOUT_CURRENT_PER_BLOCK,), -1, **i64))


def causal_layout(table, committed, pin_tokens, window_tokens, num_staged, block_size,
                  private_pages, out, err=None, stream=None):
    """Per-block rows over exact windows (see ``include/pkv.h``).  ``table``:
    int32 logical page table; ``committed``: int64 device scalar (history
    tokens); ``private_pages``: int32 ``[blocks, stride]``; ``out``: the dict of
    :func:`causal_layout_buffers`, rewritten in place."""
    assert private_pages.dim() == 2 and private_pages.is_contiguous()
    rows = out["rows"]
    st = lib().causal_layout(_ptr(table), table.numel(), _ptr(committed), pin_tokens, window_tokens,
                             num_staged, block_size, _ptr(private_pages), private_pages.shape[1], 32,
                             _ptr(rows), rows.shape[1], _ptr(out["kv_lens"]), _ptr(out["q_indptr"]),
                             _ptr(out["staged_slots"]), _ptr(out["staged_slots2"]),
                             _ptr(out["committed_src"]), _ptr(out["committed_dst"]),
                             out["committed_src"].numel(), _ptr(out["current_src_idx"]),
                             _ptr(out["current_dst"]), out["current_src_idx"].numel(), _ptr(err),
                             _stream(stream))
    _check("causal_layout", st)


def plan_buffers(batch, group_row_stride, device="cuda"):
    """Output tensors of :func:`plan_shared_prefix` for a batch of ``batch`` rows."""
    import torch
    i32 = dict(dtype=torch.int32, device=device)
    return dict(group_rows=torch.full((batch, group_row_stride), -1, **i32),
                run_lens=torch.zeros(batch, **i32), group_indptr=torch.zeros(batch + 1, **i32),
                perm=torch.zeros(batch, **i32), group_of=torch.zeros(batch, **i32),
                tail_start=torch.zeros(batch, **i32), tail_lens=torch.zeros(batch, **i32),
                num_groups=torch.zeros(1, **i32))


def plan_shared_prefix(block_table, kv_lens, q_indptr, out, max_pages=None, err=None, stream=None):
    """Shared-prefix grouping of the batch's rows (see ``include/pkv.h``);
    ``out``: the dict of :func:`plan_buffers`, rewritten in place."""
    B = kv_lens.numel()
    mp = block_table.shape[1] if max_pages is None else max_pages
    gr = out["group_rows"]
    st = lib().plan_shared_prefix(_ptr(block_table), block_table.stride(0), _ptr(kv_lens), _ptr(q_indptr), B,
                                  mp, _ptr(gr), gr.shape[1], _ptr(out["run_lens"]), _ptr(out["group_indptr"]),
                                  _ptr(out["perm"]), _ptr(out["group_of"]), _ptr(out["tail_start"]),
                                  _ptr(out["tail_lens"]), _ptr(out["num_groups"]), _ptr(err),
                                  _stream(stream))
    _check("plan_shared_prefix", st)


def shared_prefix_attention_workspace_size(batch, max_q_len, max_group_tokens, max_group_keys,
                                           num_q_heads, num_kv_heads, head_dim, num_splits=0) -> int:
    return int(lib().shared_prefix_attention_workspace_size(batch, max_q_len, max_group_tokens,
                                                            max_group_keys, num_q_heads, num_kv_heads,
                                                            head_dim, num_splits))


def shared_prefix_attention(q, k_pool, v_pool, plan, q_indptr, out, *, max_q_len, max_group_tokens,
                            max_group_keys, lse=None, scale=0.0, workspace=None, num_splits=0, flags=0,
                            err=None, stream=None):
    """One-launch attention of a planned batch (``plan``: the dict of
    :func:`plan_buffers` after :func:`plan_shared_prefix`); outputs at the
    tokens' own positions in ``out [tokens, Hq, D]`` / ``lse [tokens, Hq]``."""
    n, P, H, D, page_stride = _pool_geometry(k_pool)
    assert v_pool.shape == k_pool.shape and v_pool.stride() == k_pool.stride()
    assert q.stride(2) == 1 and out.is_contiguous()
    B = q_indptr.numel() - 1
    gr = plan["group_rows"]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().shared_prefix_attention(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k_pool), _ptr(v_pool), n, P, page_stride, _ptr(gr),
        gr.stride(0), _ptr(plan["run_lens"]), _ptr(plan["group_indptr"]), _ptr(plan["perm"]),
        _ptr(plan["tail_start"]), _ptr(plan["tail_lens"]), _ptr(plan["num_groups"]), _ptr(q_indptr), B,
        max_q_len, max_group_tokens, max_group_keys, q.shape[1], H, D, scale, _ptr(out), _dtype(out),
        _ptr(lse), _ptr(workspace), ws_bytes, num_splits, flags, _ptr(err), _stream(stream))
    _check("shared_prefix_attention", st)
