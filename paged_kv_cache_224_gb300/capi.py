"""Thin Python binding of the C ABI in ``include/pa.h`` (ctypes).

Argument marshalling only: every function takes torch CUDA tensors, checks
dtypes and shapes, passes raw device pointers and the current CUDA stream to
the C entry point of the same name, and raises :class:`PAError` on a
non-zero status.  All computation happens in the CUDA kernels of
``libpa.so``; there is no fallback of any kind -- if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_F16, PA_BF16 = 0, 1
DEVERR = {"slot_range": 0x1, "block_range": 0x2, "context_range": 0x4, "copy_pair": 0x8,
          "timeout": 0x10, "prefix": 0x20}
EXPORTED = ("pa_status_string", "pa_reshape_and_cache", "pa_decode_partition_tokens",
            "pa_decode_workspace_bytes", "pa_decode", "pa_copy_blocks_workspace_bytes", "pa_copy_blocks",
            "pa_prefill_chunk", "pa_prefill_workspace_bytes",
            "pa_decode_noalloc", "pa_decode_shared_prefix_workspace_bytes", "pa_decode_shared_prefix",
            "pa_bm_create", "pa_bm_destroy", "pa_bm_add_sequence", "pa_bm_fork", "pa_bm_append_token",
            "pa_bm_free_sequence", "pa_bm_block_table", "pa_bm_seq_len", "pa_bm_block_refcount",
            "pa_bm_stats", "pa_prefill_batch", "pa_decode_step_host_staging_bytes", "pa_decode_step_host",
            "pa_mixed_step", "pa_mixed_step_workspace_bytes", "pa_bounded_wait_polls", "pa_selftest_bounded_wait")
PA_ERR_NO_BLOCKS = -8
PA_ERR_SCRATCH_LIMIT = -7
NOALLOC_SCRATCH_BYTES = 64 << 20

_lib = None


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {pa_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load ``libpa.so`` (built by ``build.py``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"paged-KV CUDA library not built: {LIB_PATH} is missing "
                               "(run paged_kv_cache_224_gb300.build.build())")
        L = ctypes.CDLL(LIB_PATH)
        p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.pa_status_string.argtypes = [i]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_reshape_and_cache.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, p]
        L.pa_reshape_and_cache.restype = i
        L.pa_decode_partition_tokens.argtypes = [i, i, i, i, i, i]
        L.pa_decode_partition_tokens.restype = i
        L.pa_decode_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        L.pa_decode_workspace_bytes.restype = sz
        L.pa_decode.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, ctypes.c_float, i, i,
                                p, sz, p, p]
        L.pa_decode.restype = i
        L.pa_decode_noalloc.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, ctypes.c_float,
                                        i, i, p, p]
        L.pa_decode_noalloc.restype = i
        L.pa_decode_shared_prefix_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        L.pa_decode_shared_prefix_workspace_bytes.restype = sz
        L.pa_decode_shared_prefix.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, i, i,
                                              ctypes.c_float, i, i, p, sz, p, p]
        L.pa_decode_shared_prefix.restype = i
        i64 = ctypes.c_int64
        L.pa_bm_create.argtypes = [i, i, i]
        L.pa_bm_create.restype = p
        L.pa_bm_destroy.argtypes = [p]
        L.pa_bm_destroy.restype = None
        L.pa_bm_add_sequence.argtypes = [p, i64, p, i, p, ctypes.POINTER(i)]
        L.pa_bm_add_sequence.restype = i
        L.pa_bm_fork.argtypes = [p, i64, i64]
        L.pa_bm_fork.restype = i
        L.pa_bm_append_token.argtypes = [p, i64, ctypes.c_int32, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                         ctypes.POINTER(i64)]
        L.pa_bm_append_token.restype = i
        L.pa_bm_free_sequence.argtypes = [p, i64]
        L.pa_bm_free_sequence.restype = i
        L.pa_bm_block_table.argtypes = [p, i64, p, i]
        L.pa_bm_block_table.restype = i
        L.pa_bm_seq_len.argtypes = [p, i64]
        L.pa_bm_seq_len.restype = i64
        L.pa_bm_block_refcount.argtypes = [p, i]
        L.pa_bm_block_refcount.restype = i
        L.pa_bm_stats.argtypes = [p, p]
        L.pa_bm_stats.restype = i
        L.pa_copy_blocks_workspace_bytes.argtypes = [i]
        L.pa_copy_blocks_workspace_bytes.restype = sz
        L.pa_copy_blocks.argtypes = [p, p, p, i, i, i, i, i, i, p, sz, p, p]
        L.pa_copy_blocks.restype = i
        L.pa_prefill_chunk.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float, i, p, sz, p, p]
        L.pa_prefill_chunk.restype = i
        L.pa_prefill_batch.argtypes = [p, p, p, p, p, i, p, p, i, i, i, i, i, i, ctypes.c_float, i, p, sz, p, p]
        L.pa_prefill_batch.restype = i
        L.pa_prefill_workspace_bytes.argtypes = [i, i, i, i, i]
        L.pa_prefill_workspace_bytes.restype = sz
        L.pa_decode_step_host_staging_bytes.argtypes = [i] * 12
        L.pa_decode_step_host_staging_bytes.restype = sz
        L.pa_decode_step_host.argtypes = [p, p, p, p, p, i, p, i, p, i, p, i, i, i, i, i, i, i, i, p, p, i,
                                          ctypes.c_float, i, i, p, sz, p, p]
        L.pa_decode_step_host.restype = i
        L.pa_mixed_step.argtypes = [p, p, p, i, p, p, i, p, p, p, i, p, i, i, i, p, sz, p, p, i, i, i, i, i,
                                    ctypes.c_float, i, p, p]
        L.pa_mixed_step.restype = i
        L.pa_mixed_step_workspace_bytes.argtypes = [i] * 9
        L.pa_mixed_step_workspace_bytes.restype = sz
        L.pa_bounded_wait_polls.argtypes = []
        L.pa_bounded_wait_polls.restype = i
        L.pa_selftest_bounded_wait.argtypes = [i, p, p, p]
        L.pa_selftest_bounded_wait.restype = i
        _lib = L
    return _lib


def pa_status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dev(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensor must be on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensor must be contiguous")


def _stream(t: torch.Tensor, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise PAError(fn, rc)


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, d_err=None, stream=None):
    """key/value [T][Hkv][D]; caches [NB][Hkv][bs][D]; slot_mapping int64 [T]."""
    _dev(key, value, k_cache, v_cache, slot_mapping, d_err)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    NB, Hkv, bs, D = k_cache.shape
    T = key.shape[0]
    if key.shape != (T, Hkv, D) or value.shape != key.shape or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch")
    if not (key.dtype == value.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("dtype mismatch")
    rc = lib().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(slot_mapping), T, Hkv, D, bs, NB, _dt(k_cache),
                                    _ptr(d_err), _stream(k_cache, stream))
    _check("pa_reshape_and_cache", rc)


def pa_decode_partition_tokens(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                               partition_tokens=0) -> int:
    return lib().pa_decode_partition_tokens(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                                            partition_tokens)


def pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                              partition_tokens=0) -> int:
    return lib().pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                           max_context_len, partition_tokens)


def decode_workspace(query, num_kv_heads, block_size, max_context_len, partition_tokens=0):
    """Allocate (with torch) a workspace big enough for ``pa_decode``."""
    B, Hq, D = query.shape
    n = pa_decode_workspace_bytes(B, Hq, num_kv_heads, D, block_size, max_context_len, partition_tokens)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=query.device)


def pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
              partition_tokens=0, workspace=None, d_err=None, stream=None):
    """out/query [B][Hq][D]; caches [NB][Hkv][bs][D]; block_tables int32 [B][MB];
    context_lens int32 [B].  ``workspace`` defaults to a fresh torch buffer."""
    _dev(out, query, k_cache, v_cache, block_tables, context_lens, workspace, d_err)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    NB, Hkv, bs, D = k_cache.shape
    B, Hq, Dq = query.shape
    if Dq != D or out.shape != query.shape or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch")
    if not (out.dtype == query.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("dtype mismatch")
    if workspace is None:
        workspace = decode_workspace(query, Hkv, bs, max_context_len, partition_tokens)
    rc = lib().pa_decode(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                         block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs, NB,
                         int(max_context_len), float(scale), int(partition_tokens), _dt(query),
                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _ptr(d_err), _stream(query, stream))
    _check("pa_decode", rc)


def pa_decode_shared_prefix_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                            max_context_len, prefix_blocks, partition_tokens=0) -> int:
    return lib().pa_decode_shared_prefix_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                         max_context_len, prefix_blocks, partition_tokens)


def pa_decode_shared_prefix(out, query, k_cache, v_cache, block_tables, context_lens, scale,
                            max_context_len, group_size, prefix_blocks, partition_tokens=0,
                            workspace=None, d_err=None, stream=None):
    """``pa_decode`` for batches whose consecutive groups of ``group_size``
    sequences share their first ``prefix_blocks`` physical blocks."""
    _dev(out, query, k_cache, v_cache, block_tables, context_lens, workspace, d_err)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    NB, Hkv, bs, D = k_cache.shape
    B, Hq, Dq = query.shape
    if Dq != D or out.shape != query.shape or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch")
    if not (out.dtype == query.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("dtype mismatch")
    if workspace is None:
        n = pa_decode_shared_prefix_workspace_bytes(B, Hq, Hkv, D, bs, max_context_len, prefix_blocks,
                                                    partition_tokens)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=query.device)
    rc = lib().pa_decode_shared_prefix(
        _ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, int(group_size), int(prefix_blocks), Hq, Hkv, D, bs, NB,
        int(max_context_len), float(scale), int(partition_tokens), _dt(query), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(d_err), _stream(query, stream))
    _check("pa_decode_shared_prefix", rc)


def pa_decode_noalloc(out, query, k_cache, v_cache, block_tables, context_lens, scale,
                      max_context_len, partition_tokens=0, d_err=None, stream=None):
    """``pa_decode`` without a workspace: the split-K partials go to the
    library's fixed device scratch array (``NOALLOC_SCRATCH_BYTES``).  Raises
    PAError(PA_ERR_SCRATCH_LIMIT) for sizes that do not fit."""
    _dev(out, query, k_cache, v_cache, block_tables, context_lens, d_err)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    NB, Hkv, bs, D = k_cache.shape
    B, Hq, Dq = query.shape
    if Dq != D or out.shape != query.shape or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch")
    if not (out.dtype == query.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("dtype mismatch")
    rc = lib().pa_decode_noalloc(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq,
                                 Hkv, D, bs, NB, int(max_context_len), float(scale),
                                 int(partition_tokens), _dt(query), _ptr(d_err), _stream(query, stream))
    _check("pa_decode_noalloc", rc)


def _host(*ts):
    for t in ts:
        if t is not None:
            if t.is_cuda:
                raise ValueError("tensor must be in host memory")
            if not t.is_contiguous():
                raise ValueError("tensor must be contiguous")


def pa_decode_step_host_staging_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                      max_context_len, num_new_tokens, num_pairs=0, group_size=0, prefix_blocks=0,
                                      partition_tokens=0) -> int:
    return lib().pa_decode_step_host_staging_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                   max_blocks_per_seq, max_context_len, num_new_tokens, num_pairs,
                                                   group_size, prefix_blocks, partition_tokens)


def pa_decode_step_host(out, query, new_key, new_value, slot_mapping, block_tables, context_lens, k_cache,
                        v_cache, scale, max_context_len, pairs=None, group_size=0, prefix_blocks=0,
                        partition_tokens=0, staging=None, d_err=None, stream=None):
    """One decode step from host tensors (pinned for asynchronous copies):
    out/query [B][Hq][D], new_key/new_value [T][Hkv][D], slot_mapping int64 [T],
    block_tables int32 [B][MB], context_lens int32 [B], pairs int64 [n][2] or
    None; the pool (k_cache, v_cache) and ``staging`` are on the device.  The
    result lands in ``out`` once the stream has finished the step."""
    _host(out, query, new_key, new_value, slot_mapping, block_tables, context_lens, pairs)
    _dev(k_cache, v_cache, staging, d_err)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if slot_mapping.dtype != torch.int64 or (pairs is not None and pairs.dtype != torch.int64):
        raise TypeError("slot_mapping and pairs must be int64")
    NB, Hkv, bs, D = k_cache.shape
    B, Hq, Dq = query.shape
    T = new_key.shape[0]
    n = pairs.shape[0] if pairs is not None and pairs.numel() else 0
    if Dq != D or out.shape != query.shape or block_tables.shape[0] != B or context_lens.shape != (B,) or \
            new_value.shape != new_key.shape or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch")
    if not (out.dtype == query.dtype == new_key.dtype == new_value.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("dtype mismatch")
    MB = block_tables.shape[1]
    if staging is None:
        need = pa_decode_step_host_staging_bytes(B, Hq, Hkv, D, bs, MB, max_context_len, T, n, group_size,
                                                 prefix_blocks, partition_tokens)
        staging = torch.empty(max(need, 1), dtype=torch.uint8, device=k_cache.device)
    rc = lib().pa_decode_step_host(
        _ptr(out), _ptr(query), _ptr(new_key), _ptr(new_value), _ptr(slot_mapping), T, _ptr(pairs), n,
        _ptr(block_tables), MB, _ptr(context_lens), B, int(group_size), int(prefix_blocks), Hq, Hkv, D, bs, NB,
        _ptr(k_cache), _ptr(v_cache), int(max_context_len), float(scale), int(partition_tokens), _dt(query),
        _ptr(staging), staging.numel() * staging.element_size(), _ptr(d_err), _stream(k_cache, stream))
    _check("pa_decode_step_host", rc)


def pa_mixed_step(prefill_out, prefill_query, prefill_block_tables, prefix_lens, chunk_lens, decode_out,
                  decode_query, decode_block_tables, context_lens, k_cache, v_cache, scale, max_context_len,
                  partition_tokens=0, workspace=None, d_err=None, stream=None):
    """One continuous-batching step: the prompt chunks (as ``pa_prefill_batch``)
    and the decoding sequences (as ``pa_decode``) together, in one launch when
    the shape allows (see include/pa.h), else two concurrent ones.
    prefix_lens / chunk_lens are host int sequences; the rest as for those calls.
    ``workspace``: from ``mixed_workspace`` (zero-filled; reuse it across steps),
    or None to allocate one here."""
    _dev(prefill_out, prefill_query, prefill_block_tables, decode_out, decode_query, decode_block_tables,
         context_lens, k_cache, v_cache, workspace, d_err)
    for bt in (prefill_block_tables, decode_block_tables, context_lens):
        if bt.dtype != torch.int32:
            raise TypeError("block tables and context_lens must be int32")
    NB, Hkv, bs, D = k_cache.shape
    B, Hq, Dq = decode_query.shape
    R, Hq2, Dq2 = prefill_query.shape
    P = np.ascontiguousarray(np.asarray(prefix_lens, dtype=np.int32))
    C = np.ascontiguousarray(np.asarray(chunk_lens, dtype=np.int32))
    n = P.shape[0]
    if Dq != D or Dq2 != D or Hq2 != Hq or decode_out.shape != decode_query.shape or \
            prefill_out.shape != prefill_query.shape or C.shape != (n,) or int(C.sum()) != R or \
            prefill_block_tables.shape[0] != n or decode_block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch")
    if not (decode_query.dtype == prefill_query.dtype == decode_out.dtype == prefill_out.dtype == k_cache.dtype ==
            v_cache.dtype):
        raise TypeError("dtype mismatch")
    if workspace is None:
        workspace = mixed_workspace(prefill_query, decode_query, Hkv, bs, n, max_context_len, partition_tokens)
    rc = lib().pa_mixed_step(
        _ptr(prefill_out), _ptr(prefill_query), _ptr(prefill_block_tables), prefill_block_tables.shape[1],
        P.ctypes.data_as(ctypes.c_void_p), C.ctypes.data_as(ctypes.c_void_p), n, _ptr(decode_out),
        _ptr(decode_query), _ptr(decode_block_tables), decode_block_tables.shape[1], _ptr(context_lens), B,
        int(max_context_len), int(partition_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(k_cache), _ptr(v_cache), Hq, Hkv, D, bs, NB, float(scale), _dt(decode_query), _ptr(d_err),
        _stream(k_cache, stream))
    _check("pa_mixed_step", rc)


def mixed_workspace(prefill_query, decode_query, num_kv_heads, block_size, num_prefill, max_context_len,
                    partition_tokens=0):
    """A zero-filled uint8 CUDA workspace for ``pa_mixed_step`` (zero-filled
    once; the calls keep it usable)."""
    R, Hq, D = prefill_query.shape
    B = decode_query.shape[0]
    n = int(lib().pa_mixed_step_workspace_bytes(int(num_prefill), R, B, Hq, int(num_kv_heads), D, int(block_size),
                                                int(max_context_len), int(partition_tokens)))
    return torch.zeros(max(n, 1), dtype=torch.uint8, device=decode_query.device)


def pa_selftest_bounded_wait(max_polls, d_err, d_cycles=None, stream=None):
    """Run the kernels' bounded wait on a barrier nothing arrives on; it must
    give up after ``max_polls`` polls and set the timeout bit in ``d_err``."""
    _dev(d_err, d_cycles)
    rc = lib().pa_selftest_bounded_wait(int(max_polls), _ptr(d_err), _ptr(d_cycles), _stream(d_err, stream))
    _check("pa_selftest_bounded_wait", rc)


def pa_copy_blocks_workspace_bytes(num_pairs: int) -> int:
    return int(lib().pa_copy_blocks_workspace_bytes(int(num_pairs)))


def pa_copy_blocks(k_cache, v_cache, pairs, d_err=None, stream=None, workspace=None):
    """pairs int64 [n][2] of (src, dst) physical block ids.  ``workspace``:
    a uint8 CUDA tensor of at least ``pa_copy_blocks_workspace_bytes(n)``
    bytes; allocated here when not given."""
    _dev(k_cache, v_cache, pairs, d_err, workspace)
    if pairs.dtype != torch.int64:
        raise TypeError("pairs must be int64")
    NB, Hkv, bs, D = k_cache.shape
    n = pairs.shape[0] if pairs.numel() else 0
    if workspace is None:
        workspace = torch.empty(max(1, pa_copy_blocks_workspace_bytes(n)), dtype=torch.uint8,
                                device=k_cache.device)
    rc = lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), n, Hkv, D, bs, NB,
                              _dt(k_cache), _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _ptr(d_err), _stream(k_cache, stream))
    _check("pa_copy_blocks", rc)


def pa_prefill_workspace_bytes(num_seqs, total_chunk_len, num_heads, num_kv_heads, head_dim) -> int:
    return int(lib().pa_prefill_workspace_bytes(int(num_seqs), int(total_chunk_len), int(num_heads),
                                                int(num_kv_heads), int(head_dim)))


def prefill_workspace(query, num_kv_heads, num_seqs=1):
    """A zero-filled uint8 CUDA workspace big enough for prefill of ``query``'s
    rows in ``num_seqs`` chunks (zero-filled once; the calls keep it usable)."""
    R, Hq, D = query.shape
    n = pa_prefill_workspace_bytes(num_seqs, R, Hq, num_kv_heads, D)
    return torch.zeros(max(n, 1), dtype=torch.uint8, device=query.device)


def _ws(workspace):
    if workspace is None:
        return ctypes.c_void_p(0), 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def pa_prefill_chunk(out, query, k_cache, v_cache, block_table, prefix_len, scale, d_err=None,
                     stream=None, workspace=None):
    """out/query [C][Hq][D]; block_table int32 [>= ceil((P+C)/bs)].  ``workspace``:
    None (one CTA per unit) or a uint8 CUDA tensor from ``prefill_workspace``."""
    _dev(out, query, k_cache, v_cache, block_table, d_err, workspace)
    if block_table.dtype != torch.int32:
        raise TypeError("block_table must be int32")
    NB, Hkv, bs, D = k_cache.shape
    C, Hq, Dq = query.shape
    if Dq != D or out.shape != query.shape:
        raise ValueError("shape mismatch")
    if block_table.shape[0] * bs < prefix_len + C:
        raise ValueError("block table too short for prefix + chunk")
    wp, wb = _ws(workspace)
    rc = lib().pa_prefill_chunk(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_table), int(prefix_len), C, Hq, Hkv, D, bs, NB,
                                float(scale), _dt(query), wp, wb, _ptr(d_err), _stream(query, stream))
    _check("pa_prefill_chunk", rc)


def pa_prefill_batch(out, query, k_cache, v_cache, block_tables, prefix_lens, chunk_lens, scale,
                     d_err=None, stream=None, workspace=None):
    """Several sequences' chunks in one launch.  out/query [sum(chunk_lens)][Hq][D];
    block_tables int32 [n][MB] on the device; prefix_lens, chunk_lens: n host ints;
    ``workspace`` as for ``pa_prefill_chunk`` (``prefill_workspace(query, Hkv, n)``)."""
    _dev(out, query, k_cache, v_cache, block_tables, d_err, workspace)
    if block_tables.dtype != torch.int32:
        raise TypeError("block_tables must be int32")
    NB, Hkv, bs, D = k_cache.shape
    R, Hq, Dq = query.shape
    pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    cl = np.ascontiguousarray(chunk_lens, dtype=np.int32)
    n = int(cl.size)
    if Dq != D or out.shape != query.shape or pl.size != n or block_tables.shape[0] != n or int(cl.sum()) != R:
        raise ValueError("shape mismatch")
    wp, wb = _ws(workspace)
    rc = lib().pa_prefill_batch(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                block_tables.shape[1], pl.ctypes.data, cl.ctypes.data, n, Hq, Hkv, D, bs, NB,
                                float(scale), _dt(query), wp, wb, _ptr(d_err), _stream(query, stream))
    _check("pa_prefill_batch", rc)
