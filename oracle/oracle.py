"""fp64 CPU oracle for the paged K/V attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` use it.  It shares no code with
the CUDA library (``paged_kv_cache_189_gb300/csrc``) and imports nothing from
it; both sides are fed from the seeded input generators alone.

It is deliberately plain and slow: literal loops for the byte-exact steps,
numpy float64 for the arithmetic, one matmul per (sequence, K/V head) as the
only library primitive.  Each function cites the passage it follows, using the
titles of the two pull-request pages the method comes from:

* [VG]  "Paged causal K/V cache and cached attention for VisualGen"
        (TensorRT-LLM pull request 19938);
* [SP]  "Support shared-prefix attention for n-sample requests in FMHA"
        (TensorRT-LLM pull request 20841).

Conventions (the readings taken where the pages are silent are marked READING):

* bf16 values are the top 16 bits of an IEEE float32; pools and queries are
  handled as raw uint16 bit patterns and widened exactly to float64.
* K and V pools are ``[num_pages, page_size, Hkv, D]``; slot ``s`` is page
  ``s // page_size``, offset ``s % page_size`` ([VG] Description, Cache: slot
  ids are view_page * tokens_per_page + slot).  READING: token-major page layout.
* Query row ``i < q_real`` of a sequence with ``kv_len`` keys sits at absolute
  position ``kv_len - q_real + i``: each block's new tokens are the last keys
  of its row ([VG] Description, Cache, "Exact window" bullet).
* LSE is the natural log of the sum of exponentials of the scaled scores.
  READING: [SP] mentions both a natural-log and a base-2 LSE; natural log is
  the one its FlashAttention-4 path keeps.
* Padding rows (``i >= q_real``) and rows with no visible key: O = 0,
  LSE = -inf ([VG] Description, Attention, seq_len bullet: padding rows come
  back zero; [SP] commit log: an empty run has LSE -inf).
* Softmax scale defaults to 1/sqrt(D).

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against something other than itself (library routines on a different
formulation, closed forms, hand-derived visible-key sets, invariants).
"""
from __future__ import annotations

import math

import numpy as np

MASK_NONE = "none"
MASK_CAUSAL = "causal"
MASK_BLOCK_CAUSAL = "block_causal"


# ----------------------------------------------------------------------------
# bf16 decoding
# ----------------------------------------------------------------------------

def bf16_bits(x) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 torch tensor or a uint16 array."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return x
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening: a bf16 is the upper half of a float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# (1) scatter of new K/V rows into pool slots
# ----------------------------------------------------------------------------

def kv_scatter_slots(k_src, v_src, slots, k_pool, v_pool, slots2=None, src_idx=None,
                     num_slots=None):
    """Copy token rows into pool slots, bit for bit.

    [VG] Description, Cache, "Chunk K/V write" bullet and the per-file notes on
    scatterKvSlots: every token is written to one or two pool slots, reading the
    source rows once with any token/head stride; optional source indices.

    ``k_src``/``v_src``: ``[T_src, Hkv, D]`` bit arrays (any dtype, copied as
    is).  ``slots``/``slots2``: ``[T]`` int64.  ``src_idx``: ``[T]`` or None
    (READING: destination token ``t`` reads source row ``src_idx[t]``).  A
    negative slot is skipped (READING: the sentinel the pages' slot copy uses).
    If ``num_slots`` is given, a slot >= num_slots or a source index out of
    range is skipped and reported (READING: the library's checked mode).

    Returns ``(k_pool_out, v_pool_out, n_rejected)`` as new arrays.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    num_pages, page_size = k_out.shape[0], k_out.shape[1]
    T = len(slots)
    n_src = k_src.shape[0]
    rejected = 0
    for t in range(T):
        src = t if src_idx is None else int(src_idx[t])
        if num_slots is not None and not (0 <= src < n_src):
            rejected += 1
            continue
        for dest in (slots, slots2):
            if dest is None:
                continue
            s = int(dest[t])
            if s < 0:
                continue
            if num_slots is not None and s >= num_slots:
                rejected += 1
                continue
            page, off = s // page_size, s % page_size
            k_out[page, off] = k_src[src]
            v_out[page, off] = v_src[src]
    return k_out, v_out, rejected


# ----------------------------------------------------------------------------
# (4) in-place row rotation of a rolling buffer
# ----------------------------------------------------------------------------

def rotate_rows(x: np.ndarray, shift: int) -> np.ndarray:
    """Rotate every row left by ``shift`` elements: ``out[r, c] = x[r, (c + shift) mod cols]``.

    [VG] Description, Cache: eviction is an in-place rotation (new op
    rotate_rows_), and the per-file notes: supported element sizes, shifts and
    strided rows; no-op cases.  READING: left rotation (``torch.roll`` by
    ``-shift``), shift taken modulo cols, negative shifts allowed.

    ``x``: ``[rows, cols, elem_bytes]`` uint8 (an element is an opaque group of
    bytes).  Returns a new array.
    """
    out = np.array(x, copy=True)
    rows, cols = x.shape[0], x.shape[1]
    if rows == 0 or cols <= 1:
        return out
    source_col = (np.arange(cols) + shift) % cols
    for r in range(rows):
        out[r] = x[r][source_col]
    return out


# ----------------------------------------------------------------------------
# (2) attention through the paged pool
# ----------------------------------------------------------------------------

def visible_keys(i: int, q_real: int, kv_len: int, mask: str, causal_block: int) -> int:
    """Number of leading keys (logical positions ``0 .. n-1``) query row ``i`` sees.

    * none: every key of the row.
    * causal: keys up to and including the row's own position
      ``kv_len - q_real + i``.
    * block_causal: [VG] Description, Cache, frame-causal bullet and the
      causal_block_size docstring: the real tokens are cut into consecutive
      blocks of ``causal_block``; full attention within a block, causal across
      blocks.  Row ``i`` is in block ``i // causal_block`` and sees all keys
      before this step's tokens plus every new token up to the end of its
      block.  READING: a last, shorter block when q_real is not a multiple.
    * padding rows (``i >= q_real``) see nothing ([VG] seq_len bullet).
    * READING: with more new tokens than keys (``q_real > kv_len``) the first
      positions fall below key 0; a row whose last visible position is below 0
      sees no key (count 0).
    """
    if i >= q_real:
        return 0
    first_new = kv_len - q_real
    if mask == MASK_NONE:
        return kv_len
    if mask == MASK_CAUSAL:
        return max(0, first_new + i + 1)
    if mask == MASK_BLOCK_CAUSAL:
        assert causal_block > 0
        block_end = (i // causal_block + 1) * causal_block
        return max(0, first_new + min(q_real, block_end))
    raise ValueError(mask)


def gather_sequence(pool_bits: np.ndarray, table_row, kv_len: int) -> np.ndarray:
    """Materialise one sequence's contiguous ``[kv_len, Hkv, D]`` float64 keys
    (or values): logical key ``j`` lives at page ``table_row[j // P]``, offset
    ``j % P`` ([VG] Description, Attention: paged attention over per-block
    rows through the page table)."""
    P = pool_bits.shape[1]
    j = np.arange(kv_len)
    pages = np.asarray(table_row)[j // P].astype(np.int64)
    return bf16_to_f64(pool_bits[pages, j % P])


def paged_attention(q, k_pool, v_pool, block_table, kv_lens, q_indptr, q_real=None,
                    mask=MASK_CAUSAL, causal_block=0, scale=None, rows=None):
    """Attention of every query row over its sequence's keys read through the
    block table: ``O = softmax(scale * q K^T + mask) V`` and
    ``LSE = ln sum_j exp(scale * q . k_j)`` over the visible keys.

    [VG] Description, Attention (paged attention over per-block rows; seq_len
    is the real query count and padding rows come back zero) and [SP] (the
    prefix / tail calls return output and LSE).

    ``q``: ``[rows, Hq, D]`` bf16 bits; pools ``[pages, P, Hkv, D]`` bf16 bits;
    ``block_table`` ``[B, max_pages]``; ``kv_lens`` ``[B]``; ``q_indptr``
    ``[B + 1]``; ``q_real`` ``[B]`` or None (all rows real).  Query head ``h``
    reads K/V head ``h // (Hq / Hkv)`` (grouped-query heads).
    ``rows``: optional iterable of query-row indices to compute (others are
    left NaN) for spot checks of large cases.

    Returns ``(O [rows, Hq, D] float64, LSE [rows, Hq] float64)``.
    """
    q_bits = bf16_bits(q)
    kb = bf16_bits(k_pool)
    vb = bf16_bits(v_pool)
    block_table = np.asarray(block_table)
    kv_lens = np.asarray(kv_lens)
    q_indptr = np.asarray(q_indptr)
    total_rows, Hq, D = q_bits.shape
    Hkv = kb.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    B = len(kv_lens)
    want = None if rows is None else set(int(r) for r in rows)
    O = np.full((total_rows, Hq, D), np.nan)
    LSE = np.full((total_rows, Hq), np.nan)
    for b in range(B):
        r0, r1 = int(q_indptr[b]), int(q_indptr[b + 1])
        seq_rows = [r for r in range(r0, r1) if want is None or r in want]
        if not seq_rows:
            continue
        kv_len = int(kv_lens[b])
        qr = (r1 - r0) if q_real is None else int(np.asarray(q_real)[b])
        K = gather_sequence(kb, block_table[b], kv_len)   # [kv_len, Hkv, D]
        V = gather_sequence(vb, block_table[b], kv_len)
        Qb = bf16_to_f64(q_bits[seq_rows])                  # [n, Hq, D]
        nvis = np.array([visible_keys(r - r0, qr, kv_len, mask, causal_block)
                         for r in seq_rows])
        visible = np.arange(kv_len)[None, :] < nvis[:, None]   # [n, kv_len]
        for h in range(Hq):
            kvh = h // G
            s = scale * (Qb[:, h, :] @ K[:, kvh, :].T)          # [n, kv_len]
            s = np.where(visible, s, -np.inf)
            has_keys = nvis > 0
            m = np.where(has_keys, s.max(axis=1, initial=-np.inf), 0.0)
            w = np.exp(s - m[:, None])                          # exactly 0 on masked keys
            tot = w.sum(axis=1)
            safe_tot = np.where(has_keys, tot, 1.0)
            o = (w @ V[:, kvh, :]) / safe_tot[:, None]
            O[seq_rows, h] = np.where(has_keys[:, None], o, 0.0)
            LSE[seq_rows, h] = np.where(has_keys, m + np.log(safe_tot), -np.inf)
    return O, LSE


# ----------------------------------------------------------------------------
# (3) exact merge of two attention states
# ----------------------------------------------------------------------------

def merge_attn_states(o_a, lse_a, o_b, lse_b):
    """Join two partial attention states over disjoint key sets.

    [SP] Dev/commit notes: the prefix attention and the private-tail attention
    each return an output and its LSE, and one merge kernel joins them; an
    empty run has LSE -inf.  With ``m = max(La, Lb)``, ``wa = e^(La - m)``,
    ``wb = e^(Lb - m)``: ``O = (wa Oa + wb Ob) / (wa + wb)`` and
    ``L = m + ln(wa + wb)``.  READING: two empty states give O = 0, L = -inf.

    ``o_*``: ``[..., D]`` float; ``lse_*``: ``[...]``.  Returns float64 arrays.
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    la = np.asarray(lse_a, dtype=np.float64)
    lb = np.asarray(lse_b, dtype=np.float64)
    o = np.zeros(np.broadcast_shapes(o_a.shape, o_b.shape))
    lse = np.full(np.broadcast_shapes(la.shape, lb.shape), -np.inf)
    for idx in np.ndindex(*lse.shape):
        a, b = la[idx], lb[idx]
        if a == -np.inf and b == -np.inf:
            continue
        m = max(a, b)
        wa = math.exp(a - m) if a != -np.inf else 0.0
        wb = math.exp(b - m) if b != -np.inf else 0.0
        o[idx] = (wa * o_a[idx] + wb * o_b[idx]) / (wa + wb)
        lse[idx] = m + math.log(wa + wb)
    return o, lse


def merge_many(os_, lses):
    """n-way merge of partial states, folded left with the two-way merge."""
    o, lse = os_[0], lses[0]
    for o_i, l_i in zip(os_[1:], lses[1:]):
        o, lse = merge_attn_states(o, lse, o_i, l_i)
    return np.asarray(o, dtype=np.float64), np.asarray(lse, dtype=np.float64)


# ----------------------------------------------------------------------------
# fused rotary embedding + paged K/V write (the step before the scatter)
# ----------------------------------------------------------------------------

def rope_rotate(x, cos, sin):
    """NeoX-style rotary embedding of one vector set: the two halves of the
    head dimension form the pairs (x[i], x[i + D/2]), each rotated by its own
    angle: ``out[i] = x[i] cos_i - x[i+D/2] sin_i``,
    ``out[i+D/2] = x[i+D/2] cos_i + x[i] sin_i``.

    [SP] commit notes: the library rotates Q and K with NeoX RoPE (no or
    linear scaling); the kernel rope_write_kv_paged rotates Q in place and
    writes the rotated K and the V straight to the pool, RoPE at the absolute
    positions.  READING: the caller supplies the cos/sin of every (position,
    pair) as a table, so that scaling variants live in the table.

    ``x``: ``[..., D]`` float64; ``cos``, ``sin``: broadcastable ``[..., D/2]``.
    """
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def rope_write_kv_paged(q, k_src, v_src, positions, cos_sin, slots, k_pool, v_pool):
    """Rotate every query head of token t at ``positions[t]`` (in place in the
    result), rotate its K heads the same way and write them, with its V heads
    unrotated, into pool slot ``slots[t]`` (negative: no write).

    [SP] commit notes: rope_write_kv_paged rotates Q in place and writes the
    rotated K and the V straight to the pool, at the absolute positions.

    ``q``: ``[T, Hq, D]`` bf16 bits; ``k_src``/``v_src``: ``[T, Hkv, D]`` bf16
    bits; ``cos_sin``: ``[max_pos, D]`` float (cos of the D/2 pairs, then their
    sin); pools ``[pages, P, Hkv, D]`` bf16 bits.

    Returns ``(q_rot, k_rot, k_pool_out, v_pool_out, k_written)``:

    * ``q_rot`` float64 ``[T, Hq, D]`` and ``k_rot`` float64 ``[T, Hkv, D]``:
      the rotated values exactly (the device rounds them to bf16);
    * ``k_pool_out`` float64 ``[pages, P, Hkv, D]``: the K pool after the
      write, every slot ``slots[t] >= 0`` holding the exact ``k_rot[t]`` and
      every other slot the exact value of its unchanged bf16 entry;
    * ``v_pool_out``: the V pool's bf16 bits after the write (V is copied bit
      for bit);
    * ``k_written`` bool ``[pages, P]``: the slots the call wrote.
    """
    qf = bf16_to_f64(bf16_bits(q))
    kf = bf16_to_f64(bf16_bits(k_src))
    cs = np.asarray(cos_sin, dtype=np.float64)
    h = qf.shape[-1] // 2
    pos = np.asarray(positions, dtype=np.int64)
    cos = cs[pos, :h][:, None, :]
    sin = cs[pos, h:][:, None, :]
    q_rot = rope_rotate(qf, cos, sin)
    k_rot = rope_rotate(kf, cos, sin)
    k_out = bf16_to_f64(bf16_bits(k_pool))
    v_out = np.array(bf16_bits(v_pool), copy=True)
    vb = bf16_bits(v_src)
    P = k_out.shape[1]
    written = np.zeros(k_out.shape[:2], dtype=bool)
    for t, s_ in enumerate(np.asarray(slots)):
        s_ = int(s_)
        if s_ < 0:
            continue
        k_out[s_ // P, s_ % P] = k_rot[t]
        v_out[s_ // P, s_ % P] = vb[t]
        written[s_ // P, s_ % P] = True
    return q_rot, k_rot, k_out, v_out, written


# ----------------------------------------------------------------------------
# pool-to-pool slot copy (fills private pages at commit)
# ----------------------------------------------------------------------------

def copy_kv_slots(k_pools, v_pools, src_slots, dst_slots):
    """Copy whole slot rows (every K/V head) from slot ``src[c]`` to slot
    ``dst[c]`` in every layer's K and V pool; an entry with a negative source
    or destination is a sentinel and is skipped.

    [VG] Description, Cache (one pool-to-pool copy, copy_kv_slots_, fills the
    private pages at commit) and the per-file notes on causalLayout.cu (the
    pool-to-pool copy with sentinel entries; copies across layers, K/V and
    heads).  READING: all sources are read before any destination is written
    (the device kernel requires source and destination slots to be disjoint
    for this to hold).

    ``k_pools``/``v_pools``: ``[layers, pages, P, Hkv, D]`` bit arrays.
    Returns new arrays.
    """
    k_out = np.array(k_pools, copy=True)
    v_out = np.array(v_pools, copy=True)
    P = k_out.shape[2]
    pairs = [(int(s_), int(d_)) for s_, d_ in zip(src_slots, dst_slots) if s_ >= 0 and d_ >= 0]
    k_rows = [np.array(k_pools[:, s_ // P, s_ % P]) for s_, _ in pairs]
    v_rows = [np.array(v_pools[:, s_ // P, s_ % P]) for s_, _ in pairs]
    for (s_, d_), kr, vr in zip(pairs, k_rows, v_rows):
        k_out[:, d_ // P, d_ % P] = kr
        v_out[:, d_ // P, d_ % P] = vr
    return k_out, v_out


# ----------------------------------------------------------------------------
# exact-window layout of the frame-causal blocks (per-block rows with private
# pages), computed at commit
# ----------------------------------------------------------------------------

def causal_blocks(num_staged: int, block_size: int):
    """Causal blocks of a forward's staged tokens: consecutive runs of
    ``block_size`` tokens, the last one shorter when ``num_staged`` is not a
    multiple.  Returns ``[(first, count), ...]`` in staged-token indices.

    [VG] Description, Attention and Cache ("Frame-causal attention needs no
    mask" bullet: the staged tokens are cut into causal blocks that run as one
    ragged batch; block sizes are declared with the geometry).
    READING: one block size per forward, the last block partial.
    """
    out = []
    t = 0
    while t < num_staged:
        n = min(block_size, num_staged - t)
        out.append((t, n))
        t += n
    return out


def exact_window_keys(pin: int, committed: int, window: int, num_staged: int, block_size: int,
                      k: int):
    """Logical key positions causal block ``k`` attends to.

    The cache is one long sequence [fixed region | committed history | staged
    tokens] ([VG] Description, Cache): the first ``pin`` tokens are the fixed
    region, ``committed`` tokens of history follow, then this forward's
    ``num_staged`` staged tokens.  Block ``k`` sees the whole fixed region,
    the ``window`` tokens just before its own first token (history and the
    earlier blocks of this forward), and its own tokens.
    READING: the window slides with the block (each block's window starts
    ``window`` tokens before the block; the pages count a per-block
    window-start page among the partly visible pages) and never reaches into
    the fixed region.
    """
    first, n = causal_blocks(num_staged, block_size)[k]
    s = pin + committed + first
    ws = max(pin, s - window)
    return list(range(pin)) + list(range(ws, s + n))


def causal_layout(table, pin: int, committed: int, window: int, num_staged: int,
                  block_size: int, private_pages, page_size: int = 32):
    """Per-block rows that read exactly each causal block's window, in one
    ragged batch without a mask and without a duplicated key.

    [VG] Description, Cache ("Exact window" bullet and the commit bullet:
    a layout kernel reads the table and rewrites every per-block tensor at
    commit; one pool-to-pool copy fills the private pages), and the review
    notes on the private pages (committed_private: copies of committed tokens
    made at commit; current_private: copies of earlier blocks' tokens of the
    same forward, written every forward).

    ``table[lp]`` is the physical page of logical page ``lp`` of the long
    sequence (slot of logical position p = table[p // P] * P + p % P).
    ``private_pages[k]`` lists the physical pages reserved for block ``k``'s
    private region.

    Row of block k, in key order:
      1. every logical page that is fully visible to the block and ends at or
         before the block's first token, by reference, in logical order;
      2. its private pages, holding every other visible token in logical order:
         the visible tokens of partly visible pages (fixed-region tail,
         window-start page, the earlier tokens of the block's start page) and
         then the block's own tokens, which therefore stay the row's last keys.
    READING: the pages name the three kinds of partly visible page but not the
    order inside the private region; logical order is taken.

    The i-th private token of block k lives at slot
    ``private_pages[k][i // P] * P + i % P`` and is filled by one of:
      * committed (position < pin + committed): a slot-to-slot copy at commit,
        ``(src slot, dst slot)``;
      * current (an earlier block's staged token): a write from the staged
        source row every forward, ``(staged index, dst slot)``;
      * own: the staged token's second destination.
    Every staged token's first destination is its own logical slot (it becomes
    history at commit).

    Returns a dict: ``rows`` (list of page lists), ``kv_lens``, ``q_indptr``,
    ``staged_slots``, ``staged_slots2``, ``committed`` (list of (src, dst)),
    ``current`` (list of (staged index, dst)).
    """
    P = page_size
    base = pin + committed

    def slot(p):
        return int(table[p // P]) * P + p % P

    blocks = causal_blocks(num_staged, block_size)
    rows, kv_lens, q_indptr = [], [], [0]
    staged_slots = [slot(base + t) for t in range(num_staged)]
    staged_slots2 = [-1] * num_staged
    committed_copies, current_copies = [], []
    for k, (first, n) in enumerate(blocks):
        s = base + first
        vis = exact_window_keys(pin, committed, window, num_staged, block_size, k)
        vis_set = set(vis)
        end = s + n
        direct = []
        for lp in range((end + P - 1) // P):
            a = lp * P
            if a + P <= s and all(a + o in vis_set for o in range(P)):
                direct.append(lp)
        covered = set()
        for lp in direct:
            covered.update(range(lp * P, lp * P + P))
        private_tokens = [p for p in vis if p not in covered]
        private_tokens.sort()
        need = (len(private_tokens) + P - 1) // P
        if need > len(private_pages[k]):
            raise ValueError(f"block {k} needs {need} private pages, has {len(private_pages[k])}")
        row = [int(table[lp]) for lp in direct] + [int(private_pages[k][j]) for j in range(need)]
        rows.append(row)
        kv_lens.append(len(direct) * P + len(private_tokens))
        q_indptr.append(q_indptr[-1] + n)
        for i, p in enumerate(private_tokens):
            dst = int(private_pages[k][i // P]) * P + i % P
            if p < base:
                committed_copies.append((slot(p), dst))
            elif p < s:
                current_copies.append((p - base, dst))
            else:
                staged_slots2[p - base] = dst
    return dict(rows=rows, kv_lens=kv_lens, q_indptr=q_indptr, staged_slots=staged_slots,
                staged_slots2=staged_slots2, committed=committed_copies, current=current_copies)


def exact_window_attention(q, k_seq, v_seq, pin: int, committed: int, window: int,
                           num_staged: int, block_size: int, scale=None, rows=None):
    """Attention of each staged query token over exactly its causal block's
    window, read straight from the logical sequence (no pages, no layout).

    [VG] Description, Cache ("Exact window" bullet: the fp32 exact-window
    reference both backends are compared with) and the frame-causal bullet.
    ``q``: ``[num_staged, Hq, D]`` bf16 bits; ``k_seq``/``v_seq``:
    ``[pin + committed + num_staged, Hkv, D]`` bf16 bits of the long sequence
    by logical position.  Visible set of block k: ``exact_window_keys``.
    Returns ``(O [num_staged, Hq, D] f64, LSE [num_staged, Hq] f64)``;
    ``rows`` restricts the computation to those staged indices (others 0 / -inf).
    """
    qf = bf16_to_f64(np.asarray(q))
    Kf = bf16_to_f64(np.asarray(k_seq))
    Vf = bf16_to_f64(np.asarray(v_seq))
    T, Hq, D = qf.shape
    Hkv = Kf.shape[1]
    G = Hq // Hkv
    sc = 1.0 / np.sqrt(D) if scale is None else scale
    O = np.zeros((T, Hq, D))
    L = np.full((T, Hq), -np.inf)
    want = set(range(T)) if rows is None else set(int(r) for r in rows)
    for k, (first, n) in enumerate(causal_blocks(num_staged, block_size)):
        ts = [t for t in range(first, first + n) if t in want]
        if not ts:
            continue
        vis = np.array(exact_window_keys(pin, committed, window, num_staged, block_size, k))
        for kvh in range(Hkv):
            Kb, Vb = Kf[vis, kvh], Vf[vis, kvh]
            for g in range(G):
                h = kvh * G + g
                S = sc * (qf[ts, h] @ Kb.T)           # [rows, keys]
                m = S.max(axis=1, keepdims=True)
                W_ = np.exp(S - m)
                l = W_.sum(axis=1)
                O[ts, h] = (W_ @ Vb) / l[:, None]
                L[ts, h] = m[:, 0] + np.log(l)
    return O, L


# ----------------------------------------------------------------------------
# shared-prefix planner: groups of rows sharing their leading pages
# ----------------------------------------------------------------------------

def plan_shared_prefix(block_table, kv_lens, q_lens, page_size: int = 32):
    """Group the rows of a decode / verification batch whose block tables
    start with the same pages, and split every row into its group's shared run
    and its private tail.

    [SP] commit notes: rows whose K/V block tables start with identical pages
    are grouped, each group's shared pages are read once and merged with every
    row's private tail; once per step a device kernel builds each row's page
    table from its group's shared run onward (batch order) and its K/V length
    past the run; the planner's grouping is keyed on every block-table entry
    it read (entries past a row's last page ignored).

    READINGS: two rows belong together when their first pages are equal (the
    pages' grouping key) and both have at least one whole page before their
    first new token; a group's shared run is the longest run of leading pages
    identical in every member, cut at the first page that holds a member's new
    tokens (only whole, committed pages are shared); a row alone in its group
    shares nothing (run 0).  Groups are ordered by their first row, members by
    row index.

    ``block_table`` ``[B, width]``; ``kv_lens`` ``[B]`` keys including this
    step's ``q_lens`` ``[B]`` new tokens (the row's last keys).
    Returns a dict: ``groups`` (list of member-row lists), ``run_pages`` (per
    group), ``group_rows`` (per group: run pages then every member's tail pages
    in member order), ``tail_start`` (per row: its tail's first page index in
    its group's row), ``tail_lens`` (per row), ``group_of`` (per row), ``perm``
    (rows in group order).
    """
    P = page_size
    table = np.asarray(block_table)
    kv = [int(x) for x in kv_lens]
    ql = [int(x) for x in q_lens]
    B = len(kv)
    committed_pages = [(kv[r] - ql[r]) // P for r in range(B)]
    leader = list(range(B))
    for r in range(B):
        if committed_pages[r] < 1:
            continue
        for r2 in range(r):
            if committed_pages[r2] >= 1 and table[r2][0] == table[r][0]:
                leader[r] = leader[r2]
                break
    order = []
    for r in range(B):
        if leader[r] == r:
            order.append(r)
    groups = [[r for r in range(B) if leader[r] == g] for g in order]
    run_pages, group_rows = [], []
    tail_start, tail_lens, group_of = [0] * B, [0] * B, [0] * B
    for gi, members in enumerate(groups):
        run = 0
        if len(members) > 1:
            cap = min(committed_pages[m] for m in members)
            first = members[0]
            while run < cap and all(table[m][run] == table[first][run] for m in members):
                run += 1
        row = [int(x) for x in table[members[0]][:run]]
        for m in members:
            group_of[m] = gi
            tail_start[m] = len(row)
            tl = kv[m] - run * P
            tail_lens[m] = tl
            row.extend(int(x) for x in table[m][run:run + (tl + P - 1) // P])
        run_pages.append(run)
        group_rows.append(row)
    perm = [m for members in groups for m in members]
    return dict(groups=groups, run_pages=run_pages, group_rows=group_rows, tail_start=tail_start,
                tail_lens=tail_lens, group_of=group_of, perm=perm)
