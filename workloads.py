"""Seeded synthetic inputs for the decode-time MSA lightning indexer.

This module only draws inputs.  It holds none of the indexer's arithmetic
(no dot products, no block maxima, no selection), so both the CPU oracle and
the CUDA path can be fed from it without sharing any code of the method.

Shapes follow the decode indexer described on the pages:

* four index-query heads of dimension 128 per decode token
  (vLLM PR #57832, "Problem": index heads shard like KV heads, 4 of them;
  SGLang PR #41488, "Modifications": four index heads, dimension 128);
* one shared-head index-K cache paged in 128-token blocks reached through a
  block table (vLLM PR #57832, "Problem" and "Solution"; SGLang PR #41488,
  "Modifications": 128-token blocks);
* top-k = 16 with sink and sliding-window blocks pinned
  (vLLM PR #57832, "Test Plan": top-16, init/local pins).

All arrays are numpy.  bf16 values are carried as their uint16 bit patterns,
produced by rounding float32 draws to nearest-even, so every consumer reads
the very same bits.

The five named workloads are the decode configurations the indexer is
checked and measured on: a tiny case, the GB300 decode point of TensorRT-LLM
PR #17008 ("Performance", kernel table: batch 16, kv_len ~8700), the batch-32
128K case of SGLang PR #41488 ("Speed Tests and Profiling"), a ragged batch
with one long row (same table, "One 128K row, remaining 1K"), and an
adversarial tie-heavy case.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional, Sequence

import numpy as np

HEADS = 4
DIM = 128
PAGE = 128

BF16_NAN = np.uint16(0x7FC0)
BF16_BIG = np.uint16(0x4780)  # 65536.0: a large finite value used as poison

_GEN_CHUNK_PAGES = 512


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """One seeded decode batch for the indexer.

    q           uint16 [B, 4, 128]           bf16 bits of the post-RoPE index queries
    pool        uint16 [num_pages, 128, 128] bf16 bits of the paged index-K cache
    block_table int32  [B, bt_stride]        logical block -> physical page (-1 past the end)
    seq_lens    int32  [B]                   tokens per request (the current token included)
    """

    name: str
    q: np.ndarray
    pool: np.ndarray
    block_table: np.ndarray
    seq_lens: np.ndarray
    k: int = 16
    n_sink: int = 1
    n_window: int = 2
    max_model_len: int = 0
    seed: int = 0
    exact_integers: bool = False
    split_blocks_hint: int = 0
    notes: Dict[str, object] = field(default_factory=dict)
    pool8: Optional[np.ndarray] = None   # uint8 [num_pages, 128, 128] E4M3 codes (fp8 cache)
    kscale: Optional[np.ndarray] = None  # float32 [num_pages, 128] per-token scales (fp8 cache)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.pool.shape[0])

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def num_blocks(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + PAGE - 1) // PAGE

    @property
    def index_k_bytes(self) -> int:
        """Algorithmic index-K bytes: every valid token's key, once (bf16: 256 B;
        fp8: 128 B of codes + its 4-byte scale)."""
        per_token = DIM + 4 if self.pool8 is not None else DIM * 2
        return int(self.seq_lens.astype(np.int64).sum()) * per_token

    @property
    def page_bytes(self) -> int:
        """Page-granular index-K bytes: every touched 128-token page, once."""
        return int(self.num_blocks.sum()) * PAGE * DIM * 2


def _normal_bits(rng: np.random.Generator, shape: Sequence[int], scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=tuple(shape), dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x)


def _normal_pool(rng: np.random.Generator, num_pages: int) -> np.ndarray:
    pool = np.empty((num_pages, PAGE, DIM), dtype=np.uint16)
    for p0 in range(0, num_pages, _GEN_CHUNK_PAGES):
        p1 = min(num_pages, p0 + _GEN_CHUNK_PAGES)
        pool[p0:p1] = _normal_bits(rng, (p1 - p0, PAGE, DIM))
    return pool


def _ternary_bits(rng: np.random.Generator, shape: Sequence[int]) -> np.ndarray:
    v = rng.integers(-1, 2, size=tuple(shape), dtype=np.int8).astype(np.float32)
    return f32_to_bf16_bits(v)


def _ternary_pool(rng: np.random.Generator, num_pages: int) -> np.ndarray:
    pool = np.empty((num_pages, PAGE, DIM), dtype=np.uint16)
    for p0 in range(0, num_pages, _GEN_CHUNK_PAGES):
        p1 = min(num_pages, p0 + _GEN_CHUNK_PAGES)
        pool[p0:p1] = _ternary_bits(rng, (p1 - p0, PAGE, DIM))
    return pool


def _assign_pages(seq_lens: np.ndarray, bt_stride: int, order: np.ndarray) -> np.ndarray:
    """Hand out pages from `order` to the rows in turn; -1 past each row's end."""
    nb = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    if int(nb.sum()) > order.shape[0]:
        raise ValueError("pool too small for the requested lengths")
    if int(nb.max(initial=0)) > bt_stride:
        raise ValueError("bt_stride too small for the requested lengths")
    bt = np.full((seq_lens.shape[0], bt_stride), -1, dtype=np.int32)
    cursor = 0
    for b, n in enumerate(nb):
        bt[b, :n] = order[cursor:cursor + n]
        cursor += int(n)
    return bt


def poison_tails(pool: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray) -> None:
    """Fill the unused token slots of each partial last page with NaN / huge values.

    The slots past seq_len in the last page are not part of the request; any
    result that depends on them is wrong.  Rows share no pages here.
    """
    for b, L in enumerate(seq_lens.tolist()):
        rem = L % PAGE
        if L <= 0 or rem == 0:
            continue
        page = int(block_table[b, (L - 1) // PAGE])
        tail = pool[page, rem:, :]
        tail[0::2, :] = BF16_NAN
        tail[1::2, :] = BF16_BIG


def random_workload(seq_lens: Sequence[int], *, num_pages: Optional[int] = None,
                    bt_stride: Optional[int] = None, seed: int = 0, q_scale: float = 1.0,
                    shuffle: bool = True, k: int = 16, n_sink: int = 1, n_window: int = 2,
                    max_model_len: Optional[int] = None, poison: bool = True,
                    name: str = "random") -> Workload:
    """q, K ~ N(0, 1) in bf16 (q optionally scaled), paged through a block table.

    With shuffle=True the pages of all rows are one random permutation of the
    pool, sliced into rows (no page is shared); otherwise rows get consecutive
    pages.
    """
    rng = np.random.default_rng(seed)
    seq = np.asarray(seq_lens, dtype=np.int32)
    nb = (seq.astype(np.int64) + PAGE - 1) // PAGE
    need = int(nb.sum())
    if num_pages is None:
        num_pages = max(1, need)
    if max_model_len is None:
        max_model_len = max(PAGE, int(nb.max(initial=1)) * PAGE)
    if bt_stride is None:
        bt_stride = max(1, (max_model_len + PAGE - 1) // PAGE)
    B = seq.shape[0]
    q = _normal_bits(rng, (B, HEADS, DIM), scale=q_scale)
    pool = _normal_pool(rng, num_pages)
    order = rng.permutation(num_pages).astype(np.int32) if shuffle else np.arange(num_pages, dtype=np.int32)
    bt = _assign_pages(seq, bt_stride, order)
    if poison:
        poison_tails(pool, bt, seq)
    return Workload(name=name, q=q, pool=pool, block_table=bt, seq_lens=seq, k=k,
                    n_sink=n_sink, n_window=n_window, max_model_len=int(max_model_len), seed=seed)


def tiny(seed: int = 0) -> Workload:
    """B=2, seq_lens {1000, 700}: 8 and 6 blocks (fewer than k); contiguous pages."""
    w = random_workload([1000, 700], seed=seed, q_scale=1.0 / np.sqrt(DIM), shuffle=False,
                        max_model_len=1024, name="tiny")
    return w


def decode_point(seed: int = 1) -> Workload:
    """B=16 x 8700 tokens (68 blocks, last partial); 2048-page pool, permuted."""
    return random_workload([8700] * 16, num_pages=2048, seed=seed, q_scale=1.0 / np.sqrt(DIM),
                           max_model_len=8704, name="decode_point")


def long_context(seed: int = 2, batch: int = 32) -> Workload:
    """B=32 x 131072 tokens (1024 full blocks); 32768-page (1 GiB) pool, shuffled."""
    return random_workload([131072] * batch, num_pages=1024 * batch, seed=seed,
                           max_model_len=131072, name="long_context")


def ragged(seed: int = 3, permute_rows: bool = False) -> Workload:
    """B=16: one 131072-token row, one empty row, one 129-token row, 13 rows of 1024."""
    seq = [131072, 0, 129] + [1024] * 13
    if permute_rows:
        seq = list(np.random.default_rng(seed + 1000).permutation(np.asarray(seq)))
    return random_workload(seq, num_pages=2048, seed=seed, max_model_len=131072,
                           name="ragged_permuted" if permute_rows else "ragged")


ADV_BIASED_FIRST = 64
ADV_BIASED_COUNT = 40


def adversarial(seed: int = 4, batch: int = 32, seq_len: int = 32768,
                biased_first: int = ADV_BIASED_FIRST, biased_count: int = ADV_BIASED_COUNT) -> Workload:
    """Tie-heavy integer inputs with all winners in one contiguous block range.

    q and K are drawn uniformly from {-1, 0, +1}.  In every row, the tokens of
    blocks [biased_first, biased_first + biased_count) get 2 * (sum of the
    row's four query heads) added, which pushes those blocks up for every head.
    Every value is a small integer, exact in bf16, and every score is an exact
    integer in fp32, so equal scores are common and the tie-break decides.
    """
    rng = np.random.default_rng(seed)
    B = batch
    seq = np.full(B, seq_len, dtype=np.int32)
    nb = (seq_len + PAGE - 1) // PAGE
    num_pages = nb * B
    q_vals = rng.integers(-1, 2, size=(B, HEADS, DIM), dtype=np.int8).astype(np.float32)
    q = f32_to_bf16_bits(q_vals)
    pool = _ternary_pool(rng, num_pages)
    order = rng.permutation(num_pages).astype(np.int32)
    bt = _assign_pages(seq, nb, order)
    for b in range(B):
        bias = (2.0 * q_vals[b].sum(axis=0)).astype(np.float32)  # [DIM], values in [-8, 8]
        for j in range(biased_first, min(nb, biased_first + biased_count)):
            page = int(bt[b, j])
            vals = bf16_bits_to_f32(pool[page]) + bias[None, :]
            pool[page] = f32_to_bf16_bits(vals)
    return Workload(name="adversarial", q=q, pool=pool, block_table=bt, seq_lens=seq, k=16,
                    n_sink=1, n_window=2, max_model_len=int(nb * PAGE), seed=seed,
                    exact_integers=True, split_blocks_hint=biased_first,
                    notes={"biased_blocks": (biased_first, biased_first + biased_count)})


FP8_MAX = 448.0
E4M3_NAN = np.uint8(0x7F)
E4M3_MAX_CODE = np.uint8(0x7E)


def to_fp8(w: Workload, name: Optional[str] = None) -> Workload:
    """The same batch with its index-K cache stored as FP8 E4M3 + one fp32 scale per token.

    Each token's 128 values (the bf16 keys of `w`) are divided by
    scale = max|K[t,:]| / 448 and rounded to E4M3 (nearest even, saturating);
    an all-zero token gets scale 1.  Tail slots of partial last pages hold
    NaN / 448 codes with a 1e4 scale, so a result that reads them is wrong.
    """
    import torch
    pool = bf16_bits_to_f32(w.pool)  # [P, 128, 128]
    amax = np.abs(np.nan_to_num(pool, nan=0.0)).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(FP8_MAX), np.float32(1.0)).astype(np.float32)
    codes = np.empty(pool.shape, dtype=np.uint8)
    for p0 in range(0, pool.shape[0], _GEN_CHUNK_PAGES):
        p1 = min(pool.shape[0], p0 + _GEN_CHUNK_PAGES)
        x = torch.from_numpy(np.nan_to_num(pool[p0:p1] / scale[p0:p1, :, None], nan=0.0))
        codes[p0:p1] = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for b, L in enumerate(w.seq_lens.tolist()):
        rem = L % PAGE
        if L <= 0 or rem == 0:
            continue
        page = int(w.block_table[b, (L - 1) // PAGE])
        codes[page, rem::2, :] = E4M3_NAN
        codes[page, rem + 1::2, :] = E4M3_MAX_CODE
        scale[page, rem:] = np.float32(1e4)
    return Workload(name=name or (w.name + "_fp8"), q=w.q, pool=w.pool, block_table=w.block_table,
                    seq_lens=w.seq_lens, k=w.k, n_sink=w.n_sink, n_window=w.n_window,
                    max_model_len=w.max_model_len, seed=w.seed, pool8=codes, kscale=scale,
                    notes=dict(w.notes))


CONFIGS = {
    "tiny": tiny,
    "decode_point": decode_point,
    "long_context": long_context,
    "ragged": ragged,
    "adversarial": adversarial,
}


def make(name: str, **kw) -> Workload:
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
    return CONFIGS[name](**kw)
