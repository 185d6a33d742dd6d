"""Seeded synthetic inputs for the paged K/V attention path.

This module only draws inputs: random bf16 tensors, sequence lengths, page
permutations and the block tables / slot ids that name where each token lives.
It computes nothing the method itself computes (no scores, softmax, merge or
rotation), so the CUDA path and the fp64 oracle can both be fed from it.

Geometry follows the pages' framing:

* K and V pools are separate tensors ``[num_pages, page_size, Hkv, D]`` (bf16);
  slot id ``s = page * page_size + offset`` names one ``[Hkv, D]`` row
  ("Paged causal K/V cache and cached attention for VisualGen", Description,
  Cache: slot ids are ``view_page * tokens_per_page + slot``).
* ``block_table[b, j]`` is the physical page of logical page ``j`` of sequence
  ``b``; entries past a row's last page hold ``-1`` and are never read.
* ``kv_lens[b]`` counts the keys of sequence ``b`` including this step's new
  tokens; ``q_real[b]`` counts its real query rows and ``q_indptr`` packs the
  query rows (padding rows included) of all sequences.

Random numbers: Q/K/V are N(0, 1) drawn in float32 from a seeded CPU
``torch.Generator`` and rounded to bf16; lengths and permutations come from
``numpy.random.default_rng(seed)``.  Everything is returned on the CPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_SIZE = 32

__all__ = [
    "PAGE_SIZE", "PagedCase", "randn_bf16", "slot_of", "build_pool_case",
    "tiny_decode", "gqa_decode", "multi_token_decode", "chunked_prefill", "shared_prefix",
    "block_causal_video", "random_case", "WORKLOADS",
]


def randn_bf16(shape, gen: torch.Generator, scale: float = 1.0) -> torch.Tensor:
    """N(0, scale^2) samples rounded to bf16, drawn in chunks to bound memory."""
    numel = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(numel, dtype=torch.bfloat16)
    chunk = 1 << 24
    for s in range(0, numel, chunk):
        e = min(numel, s + chunk)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        out[s:e] = x.to(torch.bfloat16)
    return out.view(*shape)


def slot_of(block_table_row: np.ndarray, pos: int, page_size: int = PAGE_SIZE) -> int:
    """Slot id of logical position ``pos`` in a sequence (page * page_size + offset)."""
    return int(block_table_row[pos // page_size]) * page_size + pos % page_size


@dataclass
class PagedCase:
    """One synthetic step: new K/V rows to scatter, then attention over the pool."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    k_pool: torch.Tensor          # [num_pages, P, Hkv, D] bf16 (before the scatter)
    v_pool: torch.Tensor
    block_table: torch.Tensor     # [B, max_pages] int32, -1 past a row's pages
    kv_lens: torch.Tensor         # [B] int32, keys after the scatter
    q: torch.Tensor               # [rows, Hq, D] bf16
    q_indptr: torch.Tensor        # [B + 1] int32
    q_real: torch.Tensor          # [B] int32
    new_k: torch.Tensor           # [T, Hkv, D] bf16, rows to scatter
    new_v: torch.Tensor
    slots: torch.Tensor           # [T] int64, -1 = skip (padding rows)
    mask: str = "causal"          # "none" | "causal" | "block_causal"
    causal_block: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.kv_lens.numel())

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_q_rows(self) -> int:
        qi = self.q_indptr.numpy()
        return int((qi[1:] - qi[:-1]).max()) if self.batch else 0

    @property
    def max_kv_len(self) -> int:
        return int(self.kv_lens.max()) if self.batch else 0


def _tables_from_permutation(rng, pages_per_seq, num_pages, max_pages):
    """Assign each sequence's logical pages to distinct physical pages drawn
    from a seeded permutation of the pool; unassigned pages stay free."""
    perm = rng.permutation(num_pages)
    table = np.full((len(pages_per_seq), max(max_pages, 1)), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[at:at + n]
        at += n
    assert at <= num_pages
    return table, perm[at:]


def build_pool_case(name, seed, kv_lens, q_rows, q_real, Hq, Hkv, D, *,
                    mask="causal", causal_block=0, page_size=PAGE_SIZE,
                    free_frac=0.10, min_free_pages=0, identity_pages=False,
                    q_scale=1.0, table_width=None) -> PagedCase:
    """Generic generator: each sequence b has ``kv_lens[b]`` keys of which the
    last ``q_real[b]`` are this step's new tokens (scattered from ``new_k`` /
    ``new_v``), and ``q_rows[b] >= q_real[b]`` query rows (the extra ones are
    padding, whose new-token slot is -1)."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    q_real = np.asarray(q_real, dtype=np.int64)
    B = len(kv_lens)
    pages_per_seq = [int(-(-int(L) // page_size)) for L in kv_lens]
    used = sum(pages_per_seq)
    num_pages = max(int(np.ceil(used * (1.0 + free_frac))), used + min_free_pages, 1)
    max_pages = table_width if table_width is not None else max(pages_per_seq + [1])
    if identity_pages:
        table = np.full((B, max_pages), -1, dtype=np.int32)
        at = 0
        for b, n in enumerate(pages_per_seq):
            table[b, :n] = np.arange(at, at + n)
            at += n
    else:
        table, _ = _tables_from_permutation(rng, pages_per_seq, num_pages, max_pages)

    k_pool = randn_bf16((num_pages, page_size, Hkv, D), gen)
    v_pool = randn_bf16((num_pages, page_size, Hkv, D), gen)
    total_rows = int(q_rows.sum())
    q = randn_bf16((total_rows, Hq, D), gen, scale=q_scale)
    new_k = randn_bf16((total_rows, Hkv, D), gen)
    new_v = randn_bf16((total_rows, Hkv, D), gen)
    slots = np.full(total_rows, -1, dtype=np.int64)
    q_indptr = np.zeros(B + 1, dtype=np.int32)
    q_indptr[1:] = np.cumsum(q_rows)
    for b in range(B):
        first_new = int(kv_lens[b] - q_real[b])
        for i in range(int(q_real[b])):
            slots[q_indptr[b] + i] = slot_of(table[b], first_new + i, page_size)
    return PagedCase(
        name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=page_size,
        k_pool=k_pool, v_pool=v_pool, block_table=torch.from_numpy(table),
        kv_lens=torch.from_numpy(kv_lens.astype(np.int32)), q=q,
        q_indptr=torch.from_numpy(q_indptr), q_real=torch.from_numpy(q_real.astype(np.int32)),
        new_k=new_k, new_v=new_v, slots=torch.from_numpy(slots),
        mask=mask, causal_block=causal_block)


# ----------------------------------------------------------------------------
# The five workloads (sizes as the pages' workloads are framed)
# ----------------------------------------------------------------------------

def tiny_decode(seed: int = 0) -> PagedCase:
    """Batch 2, 4 query / 2 K/V heads, D = 64, key counts {37, 100}, one query
    row each, a 16-page pool whose pages are a seeded permutation. Besides the
    decode step, ``extra['free_slots']`` holds two random slots that no
    sequence's keys use, for a standalone scatter of the two new rows."""
    kv_lens = [37, 100]
    case = build_pool_case("tiny_decode", seed, kv_lens, [1, 1], [1, 1], 4, 2, 64,
                           mask="causal", free_frac=0.0, min_free_pages=10)
    assert case.num_pages == 16
    rng = np.random.default_rng(seed + 1000)
    table = case.block_table.numpy()
    used = set()
    for b, L in enumerate(kv_lens):
        for pos in range(L):
            used.add(slot_of(table[b], pos))
    free = np.array(sorted(set(range(case.num_pages * PAGE_SIZE)) - used), dtype=np.int64)
    case.extra["free_slots"] = torch.from_numpy(rng.choice(free, size=2, replace=False))
    return case


def gqa_decode(seed: int = 1, batch: int = 64, lo: int = 512, hi: int = 8192,
               Hq: int = 32, Hkv: int = 8, D: int = 128) -> PagedCase:
    """Batch 64, 32 query / 8 K/V heads, D = 128, cached lengths L ~ U[512, 8192];
    the step scatters one new token per sequence at position L and attends over
    L + 1 keys. Pool = total pages + 10 % free, pages randomly permuted."""
    rng = np.random.default_rng(seed)
    L = rng.integers(lo, hi, size=batch, endpoint=True)
    return build_pool_case("gqa_decode", seed, L + 1, np.ones(batch), np.ones(batch),
                           Hq, Hkv, D, mask="causal")


def multi_token_decode(seed: int = 5, batch: int = 64, q_len: int = 4, lo: int = 512,
                       hi: int = 8192, Hq: int = 32, Hkv: int = 8, D: int = 128) -> PagedCase:
    """Speculative verification: each of 64 sequences with a cached length
    L ~ U[512, 8192] appends q_len = 4 new tokens (the last accepted token and
    the drafts), scattered first, and attends causally over L + q_len keys."""
    rng = np.random.default_rng(seed)
    L = rng.integers(lo, hi, size=batch, endpoint=True)
    return build_pool_case("multi_token_decode", seed, L + q_len, np.full(batch, q_len),
                           np.full(batch, q_len), Hq, Hkv, D, mask="causal")


def chunked_prefill(seed: int = 2, batch: int = 8, chunk: int = 512, lo: int = 2048,
                    hi: int = 16384, Hq: int = 32, Hkv: int = 8, D: int = 128) -> PagedCase:
    """Batch 8, 512 new query tokens appended to a cached context of
    U[2048, 16384] tokens, causal over context + chunk, 32/8 heads, D = 128,
    permuted pages; the chunk's K/V is scattered before attention."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, size=batch, endpoint=True)
    return build_pool_case("chunked_prefill", seed, ctx + chunk, np.full(batch, chunk),
                           np.full(batch, chunk), Hq, Hkv, D, mask="causal")


def shared_prefix(seed: int = 3, groups: int = 16, samples: int = 8, prefix: int = 4096,
                  tail_lo: int = 1, tail_hi: int = 1024, Hq: int = 32, Hkv: int = 8,
                  D: int = 128, q_len: int = 1) -> PagedCase:
    """16 prompt groups x 8 samples; each group's 4096-token prefix (128 whole
    pages) is referenced once, by the group's prefix table; each sample owns a
    private tail of U[1, 1024] tokens (the last ``q_len`` are this step's
    tokens, scattered first) in its own pages. ``q_len`` query rows per sample
    (1: decode; more: speculative verification of draft tokens).

    Returned case: ``block_table`` / ``kv_lens`` describe the full rows
    (prefix ++ tail) for the oracle; ``extra`` holds the split the method uses:
    ``prefix_table [G, 128]``, ``prefix_lens [G]``, ``tail_table [G*n, max]``,
    ``tail_lens [G*n]``."""
    P = PAGE_SIZE
    assert prefix % P == 0
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    n_rows = groups * samples
    tails = np.maximum(rng.integers(tail_lo, tail_hi, size=n_rows, endpoint=True), q_len)
    prefix_pages = prefix // P
    tail_pages = [int(-(-int(t) // P)) for t in tails]
    used = groups * prefix_pages + sum(tail_pages)
    num_pages = int(np.ceil(used * 1.10))
    perm = rng.permutation(num_pages)
    at = 0
    prefix_table = np.zeros((groups, prefix_pages), dtype=np.int32)
    for g in range(groups):
        prefix_table[g] = perm[at:at + prefix_pages]
        at += prefix_pages
    max_tail_pages = max(tail_pages)
    tail_table = np.full((n_rows, max_tail_pages), -1, dtype=np.int32)
    for r in range(n_rows):
        tail_table[r, :tail_pages[r]] = perm[at:at + tail_pages[r]]
        at += tail_pages[r]
    full_table = np.full((n_rows, prefix_pages + max_tail_pages), -1, dtype=np.int32)
    for r in range(n_rows):
        full_table[r, :prefix_pages] = prefix_table[r // samples]
        full_table[r, prefix_pages:prefix_pages + tail_pages[r]] = tail_table[r, :tail_pages[r]]

    k_pool = randn_bf16((num_pages, P, Hkv, D), gen)
    v_pool = randn_bf16((num_pages, P, Hkv, D), gen)
    q = randn_bf16((n_rows * q_len, Hq, D), gen)
    new_k = randn_bf16((n_rows * q_len, Hkv, D), gen)
    new_v = randn_bf16((n_rows * q_len, Hkv, D), gen)
    slots = np.array([slot_of(tail_table[r], int(tails[r]) - q_len + i) for r in range(n_rows)
                      for i in range(q_len)], dtype=np.int64)
    ones = np.full(n_rows, q_len, dtype=np.int32)
    case = PagedCase(
        name="shared_prefix", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
        k_pool=k_pool, v_pool=v_pool, block_table=torch.from_numpy(full_table),
        kv_lens=torch.from_numpy((prefix + tails).astype(np.int32)), q=q,
        q_indptr=torch.from_numpy(np.arange(n_rows + 1, dtype=np.int32) * q_len),
        q_real=torch.from_numpy(ones), new_k=new_k, new_v=new_v,
        slots=torch.from_numpy(slots), mask="causal")
    case.extra.update(
        groups=groups, samples=samples,
        prefix_table=torch.from_numpy(prefix_table),
        prefix_lens=torch.full((groups,), prefix, dtype=torch.int32),
        # the group's sample rows packed as one query "sequence" of n x q_len rows
        prefix_q_indptr=torch.from_numpy(np.arange(groups + 1, dtype=np.int32) * samples * q_len),
        prefix_q_real=torch.full((groups,), samples * q_len, dtype=torch.int32), q_len=q_len,
        tail_table=torch.from_numpy(tail_table),
        tail_lens=torch.from_numpy(tails.astype(np.int32)))
    return case


def block_causal_video(seed: int = 4, block: int = 1560, history_blocks: int = 3,
                       H: int = 40, D: int = 128) -> PagedCase:
    """One sequence, 40 heads (no GQA), D = 128, frame block of 1560 tokens:
    keys = pinned prefix (1 block) + rolling history (3 blocks) + the current
    block; the current block's 1560 real query rows are padded up to a page
    multiple (1568 rows) and the padding rows must come back zero. Pages are the
    identity range, so the history + current region is one contiguous run of
    slots; ``extra['rotate_first_token']``/``extra['rotate_tokens']`` give the
    rolling region that is rotated left by one block after attention."""
    P = PAGE_SIZE
    kv_len = block * (2 + history_blocks)
    rows = -(-block // P) * P
    case = build_pool_case("block_causal_video", seed, [kv_len], [rows], [block], H, H, D,
                           mask="block_causal", causal_block=block, free_frac=0.0,
                           identity_pages=True)
    case.extra.update(rotate_first_token=block, rotate_tokens=block * (1 + history_blocks),
                      rotate_shift_tokens=block)
    return case


def random_case(seed: int, batch: int, Hq: int, Hkv: int, D: int, kv_range=(1, 300),
                q_range=(1, 1), pad_range=(0, 0), mask="causal", causal_block=0,
                q_scale=1.0) -> PagedCase:
    """Small randomized cases for parity tests: ragged key and query counts,
    padding rows, permuted pages."""
    rng = np.random.default_rng(seed)
    q_real = rng.integers(q_range[0], q_range[1], size=batch, endpoint=True)
    pad = rng.integers(pad_range[0], pad_range[1], size=batch, endpoint=True)
    kv = rng.integers(kv_range[0], kv_range[1], size=batch, endpoint=True)
    kv = np.maximum(kv, q_real)
    return build_pool_case(f"random_{seed}", seed, kv, q_real + pad, q_real, Hq, Hkv, D,
                           mask=mask, causal_block=causal_block, q_scale=q_scale)


def nsample_tables(rng, n_groups: int = 5, loners: int = 4, width: int = 40, page: int = PAGE_SIZE):
    """Block tables of an n-sample batch for the shared-prefix planner: groups
    of 2-6 rows sharing 1-8 leading pages (distinct first pages per group),
    every other group's members also sharing the page that holds their new
    tokens (a plan must stop its shared run before it), private tails, and
    rows that share nothing; rows of different groups interleaved.  Returns
    ``(table [B, width] int32, kv_lens, q_lens, truth)`` with ``truth`` the
    built groups as ``(sorted member rows, shared pages)``."""
    P = page
    next_page = [1000]

    def fresh(n):
        out = list(range(next_page[0], next_page[0] + n))
        next_page[0] += n
        return out

    rows, truth = [], []
    for gi in range(n_groups):
        shared = fresh(int(rng.integers(1, 9)))
        common_last = fresh(1) if gi % 2 else None
        members = []
        for _ in range(int(rng.integers(2, 7))):
            q = int(rng.integers(1, 5))
            if common_last is not None:
                tail = common_last
                kv = len(shared) * P + int(rng.integers(q, P + 1))
            else:
                tail_pages = int(rng.integers(1, 6))
                tail = fresh(tail_pages)
                kv = (len(shared) + tail_pages - 1) * P + int(rng.integers(1, P + 1))
                kv = max(kv, len(shared) * P + q)
            members.append(len(rows))
            rows.append((shared + tail, kv, q))
        truth.append((members, len(shared)))
    for _ in range(loners):
        pages = fresh(int(rng.integers(1, 6)))
        rows.append((pages, (len(pages) - 1) * P + int(rng.integers(1, P + 1)), 1))
    order = rng.permutation(len(rows))
    rows = [rows[i] for i in order]
    inv = {int(o): i for i, o in enumerate(order)}
    truth = [(sorted(inv[m] for m in members), run) for members, run in truth]
    table = np.full((len(rows), width), -1, np.int32)
    for r, (pages, _, _) in enumerate(rows):
        table[r, :len(pages)] = pages
    kv = np.array([x[1] for x in rows])
    ql = np.array([x[2] for x in rows])
    return table, kv, ql, truth


@dataclass
class ExactWindowCase:
    """One forward of the exact-window cache: a long sequence [fixed region |
    committed history | staged tokens] in a paged pool, the forward's staged
    K/V and queries, and each causal block's reserved private pages."""
    name: str
    pin: int                      # fixed-region tokens
    committed: int                # committed history tokens
    window: int                   # window tokens before each block
    staged: int                   # the forward's tokens
    block: int                    # causal block size
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    k_pool: torch.Tensor          # [pages, P, Hkv, D] bf16; committed tokens at their slots
    v_pool: torch.Tensor
    table: torch.Tensor           # [logical pages] int32, physical page of each logical page
    private_pages: torch.Tensor   # [blocks, cap] int32
    new_k: torch.Tensor           # [staged, Hkv, D] bf16
    new_v: torch.Tensor
    q: torch.Tensor               # [staged, Hq, D] bf16

    @property
    def num_blocks(self) -> int:
        return -(-self.staged // self.block)

    @property
    def max_kv_len(self) -> int:
        return self.pin + self.window + self.block

    @property
    def row_stride(self) -> int:
        return -(-self.max_kv_len // PAGE_SIZE) + 4


def exact_window(seed: int, pin: int, committed: int, window: int, staged: int, block: int,
                 Hq: int = 32, Hkv: int = 8, D: int = 128, name: str = "exact_window") -> ExactWindowCase:
    """Pages of the long sequence and the blocks' private pages are drawn from a
    seeded permutation of the pool; every pool value (private pages included,
    so a missing copy shows) is N(0, 1) bf16."""
    P = PAGE_SIZE
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    total = pin + committed + staged
    n_log = -(-total // P)
    nb = -(-staged // block)
    cap = -(-(3 * (P - 1) + block) // P)
    num_pages = n_log + nb * cap + 8
    perm = rng.permutation(num_pages).astype(np.int32)
    table = perm[:n_log]
    private = perm[n_log:n_log + nb * cap].reshape(nb, cap)
    return ExactWindowCase(
        name=name, pin=pin, committed=committed, window=window, staged=staged, block=block,
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        k_pool=randn_bf16((num_pages, P, Hkv, D), gen), v_pool=randn_bf16((num_pages, P, Hkv, D), gen),
        table=torch.from_numpy(table.copy()), private_pages=torch.from_numpy(private.copy()),
        new_k=randn_bf16((staged, Hkv, D), gen), new_v=randn_bf16((staged, Hkv, D), gen),
        q=randn_bf16((staged, Hq, D), gen))


def exact_window_video(seed: int = 6, blocks_per_chunk: int = 4) -> ExactWindowCase:
    """The exact-window geometry of the cache's benchmark: a 512-token prompt,
    96 finished frames of 394 tokens as history, a window of 95 frames, a chunk
    of 4 frames (1576 tokens); 32 query / 8 K/V heads of 128.  The clean pass
    cuts the chunk into 4 frame-causal blocks; a denoising forward is one
    block (``blocks_per_chunk=1``)."""
    frame = 394
    chunk = 4 * frame
    return exact_window(seed, pin=512, committed=96 * frame, window=95 * frame, staged=chunk,
                        block=chunk // blocks_per_chunk,
                        name="exact_window_video" if blocks_per_chunk > 1 else "exact_window_denoise")


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "gqa_decode": gqa_decode,
    "chunked_prefill": chunked_prefill,
    "shared_prefix": shared_prefix,
    "block_causal_video": block_causal_video,
    "multi_token_decode": multi_token_decode,
}
