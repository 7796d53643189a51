"""CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (``oracle.c``) of what the paged-attention path
computes, wrapped with ctypes.  It shares no code with the CUDA library and
does not import it.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.

Arguments are numpy arrays: 16-bit element data is passed as ``np.uint16``
bit patterns together with a dtype tag ("f16" or "bf16"); the oracle decodes
the bits itself.  Attention results come back as ``np.float64``.

What each function follows (page "vLLM PagedAttention chuyen sau", locionic.com):
  * ``reshape_and_cache``: growth of a sequence by writing new tokens into
    slots of its physical blocks (section "Tuong tu phan trang bo nho ao",
    dynamic resizing) -- a bit copy;
  * ``copy_blocks``: copy-on-write of a shared block (section "Co che APC",
    step 3) -- a bit copy;
  * ``decode``: the three steps of section "Co che PagedAttention": look up
    the physical blocks, gather K/V into contiguous fp64, textbook softmax
    attention;
  * ``prefill_chunk``: the same over one prompt chunk with a causal mask
    (section "Chunked Prefill", mechanism).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_DTYPES = {"f16": 0, "bf16": 1}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_oracle.so`` with the host C compiler."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", _LIB, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_reshape_and_cache.argtypes = [p, p, p, p, p, i, i, i, i, i]
        lib.oracle_reshape_and_cache.restype = i
        lib.oracle_copy_blocks.argtypes = [p, p, p, i, i, i, i, i]
        lib.oracle_copy_blocks.restype = i
        lib.oracle_decode.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, ctypes.c_double, i, i]
        lib.oracle_decode.restype = i
        lib.oracle_prefill_chunk.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_double, i, i]
        lib.oracle_prefill_chunk.restype = i
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {a.dtype}")
    return a


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def decode_bits(bits, dtype: str) -> np.ndarray:
    """Decode 16-bit patterns to float64 with the oracle's own decoder."""
    lib = _load()
    fn = lib.oracle_bf16_to_f64 if dtype == "bf16" else lib.oracle_f16_to_f64
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([fn(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, block_size: int) -> int:
    """Write new tokens' K/V rows into their slots, in place.

    key, value: uint16 [T][Hkv][D]; k_cache, v_cache: uint16 [NB][Hkv][bs][D]
    (modified in place, must be C-contiguous); slot_mapping: int64 [T].
    Returns the number of slots that fell outside the pool (skipped).
    """
    lib = _load()
    key, value = _u16(key), _u16(value)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous")
    slots = _c(slot_mapping, np.int64)
    T, Hkv, D = key.shape
    NB = k_cache.shape[0]
    return lib.oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(slots), T, Hkv, D, block_size, NB)


def copy_blocks(k_cache, v_cache, pairs) -> int:
    """Copy whole blocks src -> dst for each (src, dst) row of ``pairs``, in place.

    Returns the number of invalid pairs (skipped): out-of-pool ids, src == dst,
    a dst used twice, or a dst that is also some pair's src.
    """
    lib = _load()
    pairs = _c(pairs, np.int64).reshape(-1, 2)
    NB, Hkv, bs, D = k_cache.shape
    return lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0],
                                  Hkv, D, bs, NB)


def decode(query, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: str,
           num_threads: int = 1) -> np.ndarray:
    """Paged single-query decode attention in fp64.

    query uint16 [B][Hq][D]; caches uint16 [NB][Hkv][bs][D];
    block_tables int32 [B][MB]; context_lens int32 [B].  Returns float64 [B][Hq][D].
    """
    lib = _load()
    query, k_cache, v_cache = _u16(query), _u16(k_cache), _u16(v_cache)
    bt = _c(block_tables, np.int32)
    lens = _c(context_lens, np.int32)
    B, Hq, D = query.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and bt.shape[0] == B and lens.shape[0] == B
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = lib.oracle_decode(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                           bt.shape[1], _ptr(lens), B, Hq, Hkv, D, bs, NB, float(scale),
                           _DTYPES[dtype], int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_decode: invalid input (rc={rc})")
    return out


def prefill_chunk(query, k_cache, v_cache, block_table, prefix_len: int, scale: float, dtype: str,
                  num_threads: int = 1) -> np.ndarray:
    """Causal attention of a prompt chunk over its paged prefix plus itself, fp64.

    query uint16 [C][Hq][D]; block_table int32 [>= ceil((P+C)/bs)].
    Returns float64 [C][Hq][D].
    """
    lib = _load()
    query, k_cache, v_cache = _u16(query), _u16(k_cache), _u16(v_cache)
    bt = _c(block_table, np.int32)
    C, Hq, D = query.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert D2 == D
    if bt.shape[0] * bs < prefix_len + C:
        raise ValueError("block table too short for prefix + chunk")
    out = np.zeros((C, Hq, D), dtype=np.float64)
    rc = lib.oracle_prefill_chunk(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                  int(prefix_len), C, Hq, Hkv, D, bs, NB, float(scale),
                                  _DTYPES[dtype], int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_prefill_chunk: invalid input (rc={rc})")
    return out


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
