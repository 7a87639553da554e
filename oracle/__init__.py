"""CPU oracle for the decode-time MSA lightning indexer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``msa_oracle.c`` (plain C,
fp64) through ctypes and shares no code with the CUDA library.  See the
header of ``msa_oracle.c`` for what each function computes and the passages
of the pages it follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

HEADS = 4
DIM = 128
PAGE = 128

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "msa_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libmsa_oracle.so")

_lock = threading.Lock()
_default = None


def build(src: str = SOURCE, out: str = LIBRARY, openmp: bool = True) -> str:
    """Compile the oracle into a shared library with gcc (host only)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-Wall", "-Wextra"]
    if openmp:
        cmd.append("-fopenmp")
    cmd += ["-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build(out: str, src: str) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        c_i64, c_int = ctypes.c_int64, ctypes.c_int
        P = ctypes.c_void_p
        lib.msa_oracle_block_scores.argtypes = [P, P, c_i64, P, c_i64, P, c_int, P]
        lib.msa_oracle_block_scores.restype = c_int
        lib.msa_oracle_select.argtypes = [P, c_int, c_i64, P, c_int, c_int, c_int, P, P]
        lib.msa_oracle_select.restype = c_int
        lib.msa_oracle_select_split.argtypes = [P, c_int, c_i64, P, c_int, c_int, c_int, c_i64, P, P]
        lib.msa_oracle_select_split.restype = c_int
        lib.msa_oracle_expand_pages.argtypes = [P, c_int, c_int, P, P, c_i64, c_int, P, P]
        lib.msa_oracle_expand_pages.restype = c_int
        lib.msa_oracle_block_scores_fp8.argtypes = [P, P, P, c_i64, P, c_i64, P, c_int, P]
        lib.msa_oracle_block_scores_fp8.restype = c_int
        lib.msa_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.msa_oracle_e4m3_value.restype = ctypes.c_double
        lib.msa_oracle_num_threads.argtypes = []
        lib.msa_oracle_num_threads.restype = c_int
        lib.msa_oracle_set_num_threads.argtypes = [c_int]
        lib.msa_oracle_set_num_threads.restype = None
        self.lib = lib

    @staticmethod
    def _ptr(a: np.ndarray) -> int:
        return a.ctypes.data

    def num_threads(self) -> int:
        return int(self.lib.msa_oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Host threads for later calls (the arithmetic does not depend on it)."""
        self.lib.msa_oracle_set_num_threads(int(n))

    def block_scores(self, q: np.ndarray, pool: np.ndarray, block_table: np.ndarray,
                     seq_lens: np.ndarray) -> np.ndarray:
        """fp64 block scores [B, 4, bt_stride]; -inf past each row's last block."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        pool = np.ascontiguousarray(pool, dtype=np.uint16)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, stride = bt.shape
        assert q.shape == (B, HEADS, DIM) and seq.shape == (B,)
        assert pool.ndim == 3 and pool.shape[1:] == (PAGE, DIM)
        out = np.empty((B, HEADS, stride), dtype=np.float64)
        rc = self.lib.msa_oracle_block_scores(self._ptr(q), self._ptr(pool), pool.shape[0],
                                              self._ptr(bt), stride, self._ptr(seq), B,
                                              self._ptr(out))
        if rc != 0:
            raise ValueError(f"oracle refused the inputs (code {rc})")
        return out

    def e4m3_value(self, code: int) -> float:
        return float(self.lib.msa_oracle_e4m3_value(code))

    def block_scores_fp8(self, q: np.ndarray, pool8: np.ndarray, kscale: np.ndarray,
                         block_table: np.ndarray, seq_lens: np.ndarray) -> np.ndarray:
        """fp64 block scores on an E4M3 cache with per-token scales."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        pool8 = np.ascontiguousarray(pool8, dtype=np.uint8)
        kscale = np.ascontiguousarray(kscale, dtype=np.float32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, stride = bt.shape
        assert pool8.ndim == 3 and pool8.shape[1:] == (PAGE, DIM)
        assert kscale.shape == pool8.shape[:2]
        out = np.empty((B, HEADS, stride), dtype=np.float64)
        rc = self.lib.msa_oracle_block_scores_fp8(self._ptr(q), self._ptr(pool8), self._ptr(kscale),
                                                  pool8.shape[0], self._ptr(bt), stride,
                                                  self._ptr(seq), B, self._ptr(out))
        if rc != 0:
            raise ValueError(f"oracle refused the inputs (code {rc})")
        return out

    def select(self, scores: np.ndarray, seq_lens: np.ndarray, k: int, n_sink: int,
               n_window: int) -> Tuple[np.ndarray, np.ndarray]:
        """Per-head selection: (ids int32 [B,4,k], scores fp64 [B,4,k])."""
        scores = np.ascontiguousarray(scores, dtype=np.float64)
        seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, H, stride = scores.shape
        assert H == HEADS and seq.shape == (B,)
        ids = np.empty((B, HEADS, k), dtype=np.int32)
        out = np.empty((B, HEADS, k), dtype=np.float64)
        rc = self.lib.msa_oracle_select(self._ptr(scores), B, stride, self._ptr(seq), k, n_sink,
                                        n_window, self._ptr(ids), self._ptr(out))
        if rc != 0:
            raise ValueError(f"oracle refused the selection arguments (code {rc})")
        return ids, out

    def select_split(self, scores: np.ndarray, seq_lens: np.ndarray, k: int, n_sink: int,
                     n_window: int, split_blocks: int) -> Tuple[np.ndarray, np.ndarray]:
        """The selection reached through contiguous splits of `split_blocks` blocks."""
        scores = np.ascontiguousarray(scores, dtype=np.float64)
        seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, H, stride = scores.shape
        ids = np.empty((B, HEADS, k), dtype=np.int32)
        out = np.empty((B, HEADS, k), dtype=np.float64)
        rc = self.lib.msa_oracle_select_split(self._ptr(scores), B, stride, self._ptr(seq), k,
                                              n_sink, n_window, split_blocks, self._ptr(ids),
                                              self._ptr(out))
        if rc != 0:
            raise ValueError(f"oracle refused the selection arguments (code {rc})")
        return ids, out

    def expand_pages(self, ids: np.ndarray, seq_lens: np.ndarray, kv_block_table: np.ndarray,
                     page_tokens: int = 16) -> Tuple[np.ndarray, np.ndarray]:
        """Selected blocks -> small KV page ids: (pages [B,4,k*128/pt], counts [B,4])."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
        kvb = np.ascontiguousarray(kv_block_table, dtype=np.int32)
        B, H, k = ids.shape
        width = k * (PAGE // page_tokens)
        pages = np.empty((B, HEADS, width), dtype=np.int32)
        num = np.empty((B, HEADS), dtype=np.int32)
        rc = self.lib.msa_oracle_expand_pages(self._ptr(ids), B, k, self._ptr(seq), self._ptr(kvb),
                                              kvb.shape[1], page_tokens, self._ptr(pages),
                                              self._ptr(num))
        if rc != 0:
            raise ValueError(f"oracle refused the expansion arguments (code {rc})")
        return pages, num

    def run_multi(self, q: np.ndarray, pool: np.ndarray, block_table: np.ndarray,
                  seq_lens: np.ndarray, k: int, n_sink: int, n_window: int,
                  pool8: Optional[np.ndarray] = None, kscale: Optional[np.ndarray] = None):
        """Several query positions per request (speculative-decode verification).

        q is [B, Q, 4, 128]: the last Q tokens of each request.  Position i
        sees the first seq_len - (Q - 1 - i) tokens: TensorRT-LLM PR #17008,
        "Description", causal clamp eff_kv = min(q_end + offset_q, kv_len) with
        offset_q = kv_len - Q.  Each position is then one decode query over
        its own context, so this is the single-query oracle on B*Q rows.
        Returns (scores [B,Q,4,stride], ids [B,Q,4,k], sel [B,Q,4,k], lens [B,Q]).
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        B, Q = q.shape[:2]
        seq = np.asarray(seq_lens, dtype=np.int64)
        lens = seq[:, None] - (Q - 1 - np.arange(Q))[None, :]
        lens = np.maximum(lens, 0).astype(np.int32)
        rows_q = q.reshape(B * Q, HEADS, DIM)
        rows_bt = np.repeat(np.ascontiguousarray(block_table, dtype=np.int32), Q, axis=0)
        rows_len = lens.reshape(B * Q)
        if pool8 is not None:
            s = self.block_scores_fp8(rows_q, pool8, kscale, rows_bt, rows_len)
        else:
            s = self.block_scores(rows_q, pool, rows_bt, rows_len)
        ids, sel = self.select(s, rows_len, k, n_sink, n_window)
        stride = s.shape[2]
        return (s.reshape(B, Q, HEADS, stride), ids.reshape(B, Q, HEADS, k),
                sel.reshape(B, Q, HEADS, k), lens)

    def run_prefill(self, q: np.ndarray, cu_seqlens_q: np.ndarray, pool: Optional[np.ndarray],
                    block_table: np.ndarray, seq_lens: np.ndarray, k: int, n_sink: int,
                    n_window: int, pool8: Optional[np.ndarray] = None,
                    kscale: Optional[np.ndarray] = None):
        """Prefill: the new tokens of every request, each over its own causal prefix.

        q is [total_q, 4, 128]; request b's new tokens are rows
        [cu_seqlens_q[b], cu_seqlens_q[b+1]) and are its last n_b tokens
        (vLLM PR #57832, "Question ... mixed batches": the prefill branch
        scores iq[nd:] with cu_seqlens_q).  New token t of request b sits at
        position seq_len - n_b + t and sees the first seq_len - n_b + t + 1
        tokens, so each row is one decode query over that length.  With pool8 /
        kscale the keys are the E4M3 cache of block_scores_fp8.
        Returns (scores [total_q,4,stride], ids [total_q,4,k], sel, lens [total_q]).
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        cu = np.asarray(cu_seqlens_q, dtype=np.int64)
        seq = np.asarray(seq_lens, dtype=np.int64)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        rows_bt, lens = [], []
        for b in range(seq.shape[0]):
            n = int(cu[b + 1] - cu[b])
            for t in range(n):
                rows_bt.append(bt[b])
                lens.append(max(0, int(seq[b]) - n + t + 1))
        lens = np.asarray(lens, dtype=np.int32)
        rows_bt = np.asarray(rows_bt, dtype=np.int32).reshape(-1, bt.shape[1])
        if pool8 is not None:
            s = self.block_scores_fp8(q, pool8, kscale, rows_bt, lens)
        else:
            s = self.block_scores(q, pool, rows_bt, lens)
        ids, sel = self.select(s, lens, k, n_sink, n_window)
        return s, ids, sel, lens

    def run(self, w, k: Optional[int] = None, n_sink: Optional[int] = None,
            n_window: Optional[int] = None):
        """Block scores and selection for a `workloads.Workload` (bf16 or fp8 cache)."""
        k = w.k if k is None else k
        n_sink = w.n_sink if n_sink is None else n_sink
        n_window = w.n_window if n_window is None else n_window
        if getattr(w, "pool8", None) is not None:
            s = self.block_scores_fp8(w.q, w.pool8, w.kscale, w.block_table, w.seq_lens)
        else:
            s = self.block_scores(w.q, w.pool, w.block_table, w.seq_lens)
        ids, sc = self.select(s, w.seq_lens, k, n_sink, n_window)
        return s, ids, sc


def load(path: Optional[str] = None) -> Oracle:
    """The oracle library (built on first use when missing or stale)."""
    global _default
    if path is not None:
        return Oracle(path)
    with _lock:
        if _default is None:
            if _needs_build(LIBRARY, SOURCE):
                build()
            _default = Oracle(LIBRARY)
        return _default
