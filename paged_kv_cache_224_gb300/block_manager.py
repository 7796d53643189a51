"""Python face of the native block manager (``pa_bm_*`` in ``include/pa.h``).

Argument marshalling only: the bookkeeping (allocation, reference counts,
copy-on-write, prefix tree, eviction) runs in ``libpa.so``.  Host-only; no
GPU is needed.
"""
from __future__ import annotations

import ctypes

import numpy as np

from .capi import PAError, lib


class _Counters(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("free_blocks", ctypes.c_int),
                ("cached_free_blocks", ctypes.c_int), ("used_blocks", ctypes.c_int),
                ("num_sequences", ctypes.c_int), ("query_tokens", ctypes.c_longlong),
                ("hit_tokens", ctypes.c_longlong), ("evictions", ctypes.c_longlong),
                ("cow_copies", ctypes.c_longlong)]


class BlockManager:
    """Physical blocks of one paged pool: tables, refcounts, copy-on-write,
    automatic prefix caching.  See ``pa_bm_*`` in ``include/pa.h``."""

    def __init__(self, num_blocks: int, block_size: int, prefix_cache: bool = True):
        self._L = lib()
        self._h = self._L.pa_bm_create(int(num_blocks), int(block_size), 1 if prefix_cache else 0)
        if not self._h:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            self._L.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def _check(self, fn: str, rc: int) -> int:
        if rc < 0:
            raise PAError(fn, rc)
        return rc

    def add_sequence(self, seq_id: int, tokens) -> tuple:
        """Register a prompt.  Returns (slots int64 [n] with -1 for tokens
        whose K/V came from the prefix cache, number of cached tokens)."""
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        slots = np.empty(tok.size, dtype=np.int64)
        cached = ctypes.c_int(0)
        rc = self._L.pa_bm_add_sequence(self._h, int(seq_id), tok.ctypes.data, tok.size,
                                         slots.ctypes.data, ctypes.byref(cached))
        self._check("pa_bm_add_sequence", rc)
        return slots, int(cached.value)

    def fork(self, parent_id: int, child_id: int) -> None:
        self._check("pa_bm_fork", self._L.pa_bm_fork(self._h, int(parent_id), int(child_id)))

    def append_token(self, seq_id: int, token: int) -> tuple:
        """One more token.  Returns (slot, (src, dst) copy-on-write pair or None)."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        rc = self._L.pa_bm_append_token(self._h, int(seq_id), int(token), ctypes.byref(slot),
                                         ctypes.byref(src), ctypes.byref(dst))
        self._check("pa_bm_append_token", rc)
        pair = None if src.value < 0 else (int(src.value), int(dst.value))
        return int(slot.value), pair

    def free_sequence(self, seq_id: int) -> None:
        self._check("pa_bm_free_sequence", self._L.pa_bm_free_sequence(self._h, int(seq_id)))

    def block_table(self, seq_id: int) -> np.ndarray:
        n = self.seq_len(seq_id)
        cap = max(1, -(-n // self.block_size))
        out = np.empty(cap, dtype=np.int32)
        k = self._check("pa_bm_block_table", self._L.pa_bm_block_table(self._h, int(seq_id), out.ctypes.data, cap))
        return out[:k].copy()

    def seq_len(self, seq_id: int) -> int:
        return self._check("pa_bm_seq_len", int(self._L.pa_bm_seq_len(self._h, int(seq_id))))

    def refcount(self, block: int) -> int:
        return self._check("pa_bm_block_refcount", self._L.pa_bm_block_refcount(self._h, int(block)))

    def stats(self) -> dict:
        c = _Counters()
        self._check("pa_bm_stats", self._L.pa_bm_stats(self._h, ctypes.byref(c)))
        d = {f: getattr(c, f) for f, _ in _Counters._fields_}
        d["hit_rate"] = d["hit_tokens"] / d["query_tokens"] if d["query_tokens"] else 0.0
        return d

    def tables(self, seq_ids, max_blocks: int | None = None) -> np.ndarray:
        """Block-table rows of ``seq_ids`` as the kernels take them (int32, -1 padded)."""
        rows = [self.block_table(s) for s in seq_ids]
        mb = max_blocks or max(1, max(len(r) for r in rows))
        out = np.full((len(rows), mb), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            out[i, :len(r)] = r
        return out
