"""CPU-side checks of the C ABI: the library builds, loads, exports every
symbol ``include/pa.h`` declares, and rejects bad arguments on the host
without launching anything (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_224_gb300 import build
    build.build()
    import paged_kv_cache_224_gb300 as pa
    return pa.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_copy_blocks", "pa_prefill_chunk",
              "pa_decode_workspace_bytes", "pa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n
    from paged_kv_cache_224_gb300 import capi
    assert sorted(capi.EXPORTED) == sorted(declared_symbols())


def test_status_strings(lib):
    import paged_kv_cache_224_gb300 as pa
    assert pa.pa_status_string(0) == "PA_OK"
    assert "WORKSPACE" in pa.pa_status_string(-5)
    assert "unknown" in pa.pa_status_string(1234)


def test_workspace_and_partition_rules(lib):
    import paged_kv_cache_224_gb300 as pa
    # every sequence fits one partition -> no workspace
    assert pa.pa_decode_workspace_bytes(4, 4, 4, 64, 16, 64, 0) == 0
    # the automatic length on the decode workloads: LLaMA GQA, long context, OPT MHA
    assert pa.pa_decode_partition_tokens(256, 32, 8, 16, 4096, 0) == 1024
    assert pa.pa_decode_partition_tokens(8, 64, 8, 16, 131072, 0) == 2048
    assert pa.pa_decode_partition_tokens(64, 40, 40, 16, 2048, 0) == 512
    # few, short sequences: the shortest partitions; huge batches: the longest
    assert pa.pa_decode_partition_tokens(1, 8, 8, 16, 1024, 0) == 256
    assert pa.pa_decode_partition_tokens(4096, 64, 8, 16, 32768, 0) == 4096
    assert pa.pa_decode_partition_tokens(1, 8, 8, 128, 16, 0) == 256
    n = pa.pa_decode_workspace_bytes(256, 32, 8, 128, 16, 4096, 0)
    parts = 4
    assert n >= 256 * 32 * parts * (128 + 2) * 4
    # explicit partitions must be multiples of block_size
    assert pa.pa_decode_partition_tokens(4, 4, 4, 16, 100, 24) == 0
    assert pa.pa_decode_partition_tokens(4, 4, 4, 16, 100, 32) == 32
    assert pa.pa_decode_partition_tokens(4, 6, 4, 16, 100, 32) == 0   # heads not a multiple of kv heads


def call_decode(lib, **kw):
    a = dict(out=1 << 20, query=1 << 20, k=1 << 20, v=1 << 20, bt=1 << 20, mb=4, lens=1 << 20, B=2,
             Hq=8, Hkv=2, D=128, bs=16, NB=64, maxlen=64, scale=0.1, pt=0, dt=1, ws=None, wsb=0)
    a.update(kw)
    p = ctypes.c_void_p
    return lib.pa_decode(p(a["out"]), p(a["query"]), p(a["k"]), p(a["v"]), p(a["bt"]), a["mb"],
                         p(a["lens"]), a["B"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"], a["maxlen"],
                         a["scale"], a["pt"], a["dt"], p(a["ws"]), a["wsb"], None, None)


def test_copy_blocks_workspace_is_linear_in_the_pairs(lib):
    # a hash table of 16-byte entries, a power of two >= 4 per pair (at least 64)
    assert lib.pa_copy_blocks_workspace_bytes(0) == 0
    assert lib.pa_copy_blocks_workspace_bytes(1) == 64 * 16
    assert lib.pa_copy_blocks_workspace_bytes(224) == 1024 * 16
    assert lib.pa_copy_blocks_workspace_bytes(4096) == 16384 * 16
    assert lib.pa_copy_blocks_workspace_bytes(-1) == 0
    assert lib.pa_copy_blocks_workspace_bytes((1 << 26) + 1) == 0


def test_python_error_bits_match_the_header(lib):
    from paged_kv_cache_224_gb300 import capi
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    bits = {m.group(1).lower(): int(m.group(2), 16)
            for m in re.finditer(r"#define\s+PA_DEVERR_(\w+)\s+0x([0-9a-fA-F]+)", text)}
    assert bits and bits == capi.DEVERR


def test_decode_rejects_bad_arguments_on_host(lib):
    # These return before any CUDA call, so no device is touched.
    assert call_decode(lib, out=0) == -1                  # null pointer
    assert call_decode(lib, Hq=7) == -1                   # Hq % Hkv != 0
    assert call_decode(lib, D=96) == -2                   # unsupported head_dim
    assert call_decode(lib, bs=24) == -2                  # unsupported block_size
    assert call_decode(lib, bs=256) == -2
    assert call_decode(lib, Hq=32, Hkv=2) == -2           # group 16 unsupported
    assert call_decode(lib, dt=7) == -1                   # bad dtype
    assert call_decode(lib, query=(1 << 20) + 2) == -6    # misaligned
    assert call_decode(lib, scale=float("inf")) == -3
    assert call_decode(lib, pt=24) == -3                  # not a multiple of block_size
    assert call_decode(lib, maxlen=5000) == -5            # split needs a workspace
    assert call_decode(lib, B=0) == 0                     # nothing to do


def test_cache_calls_reject_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    buf = p(1 << 20)
    assert lib.pa_reshape_and_cache(buf, buf, buf, buf, None, 4, 2, 128, 16, 64, 1, None, None) == -1
    assert lib.pa_reshape_and_cache(buf, buf, buf, buf, buf, 4, 2, 12, 16, 64, 1, None, None) == -2
    assert lib.pa_reshape_and_cache(buf, buf, buf, buf, buf, 0, 2, 128, 16, 64, 1, None, None) == 0
    ws = lib.pa_copy_blocks_workspace_bytes(3)
    assert lib.pa_copy_blocks(buf, None, buf, 3, 2, 128, 16, 64, 1, buf, ws, None, None) == -1
    assert lib.pa_copy_blocks(buf, buf, buf, 0, 2, 128, 16, 64, 1, None, 0, None, None) == 0
    assert lib.pa_copy_blocks(buf, buf, buf, 3, 2, 128, 16, 64, 1, None, 0, None, None) == -5   # no workspace
    assert lib.pa_copy_blocks(buf, buf, buf, 3, 2, 128, 16, 64, 1, buf, ws - 1, None, None) == -5
    assert lib.pa_copy_blocks(buf, buf, buf, 3, 2, 128, 16, 64, 1, p((1 << 20) + 8), ws, None, None) == -6
    assert lib.pa_copy_blocks(buf, buf, buf, (1 << 26) + 1, 2, 128, 16, 64, 1, buf, 1 << 40, None, None) == -3
    assert lib.pa_prefill_chunk(buf, buf, buf, buf, buf, 8, 4, 7, 2, 128, 16, 64, 0.1, 1, None, 0, None, None) == -1
    # a workspace too small for the stream-K schedule, or misaligned (both found before any CUDA call)
    assert lib.pa_prefill_chunk(buf, buf, buf, buf, buf, 8, 4, 8, 2, 128, 16, 64, 0.1, 1, buf, 16, None, None) == -5
    need = lib.pa_prefill_workspace_bytes(1, 4, 8, 2, 128)
    assert need > 0 and lib.pa_prefill_workspace_bytes(1, 4, 7, 2, 128) == 0
    assert lib.pa_prefill_chunk(buf, buf, buf, buf, buf, 8, 4, 8, 2, 128, 16, 64, 0.1, 1, p((1 << 20) + 16), need,
                                None, None) == -6


def test_shared_prefix_and_batch_prefill_reject_bad_arguments_on_host(lib):
    # all of these return before any CUDA call
    p = ctypes.c_void_p
    buf = p(1 << 20)
    f = ctypes.c_float

    def sp(B=8, S=4, pb=2, Hq=4, Hkv=4, D=128, bs=16, maxlen=100, ws=1 << 30, wsp=buf):
        return lib.pa_decode_shared_prefix(buf, buf, buf, buf, buf, 16, buf, B, S, pb, Hq, Hkv, D, bs, 64,
                                           maxlen, f(0.1), 0, 1, wsp, ws, None, None)
    assert sp(S=3) == -1                       # 8 sequences are not groups of 3
    assert sp(pb=0) == -1                      # no shared prefix
    assert sp(pb=20) == -3                     # prefix longer than the table
    assert sp(Hq=8, Hkv=2, S=4) == -2          # head group 16
    assert sp(ws=16) == -5                     # workspace too small
    assert sp(B=0) == 0
    assert lib.pa_decode_shared_prefix_workspace_bytes(8, 4, 4, 128, 16, 100, 2, 0) > 0
    assert lib.pa_decode_shared_prefix_workspace_bytes(8, 4, 4, 128, 16, 100, 0, 0) == 0

    pl = (ctypes.c_int * 3)(10, 0, 5)
    cl = (ctypes.c_int * 3)(4, 0, 3)
    bad = (ctypes.c_int * 3)(4, -1, 3)
    big = (ctypes.c_int * 3)(4, 0, 500)

    def pb(prefix=pl, chunk=cl, n=3, Hq=4, Hkv=2, scale=0.1, mb=4):
        return lib.pa_prefill_batch(buf, buf, buf, buf, buf, mb, prefix, chunk, n, Hq, Hkv, 128, 16, 64,
                                    f(scale), 1, None, 0, None, None)
    assert pb(chunk=bad) == -1                 # negative chunk length
    assert pb(chunk=big) == -3                 # prefix + chunk past the table row
    assert pb(Hq=3) == -1
    assert pb(scale=-1.0) == -3
    assert pb(n=0) == 0
    zero = (ctypes.c_int * 3)(0, 0, 0)
    assert pb(chunk=zero) == 0                 # nothing to attend


def test_host_step_rejects_bad_arguments_on_host(lib):
    # every check happens before any copy is queued
    p = ctypes.c_void_p
    buf = p(1 << 20)
    f = ctypes.c_float
    need = lib.pa_decode_step_host_staging_bytes(4, 8, 2, 128, 16, 8, 100, 4, 0, 0, 0, 0)
    # out + query (4*8*128*2 each), new K and V (4*2*128*2 each), slots, tables, lengths, 256-byte aligned
    assert need == 2 * 8192 + 2 * 2048 + 256 + 256 + 256
    assert lib.pa_decode_step_host_staging_bytes(4, 8, 2, 128, 16, 8, 100, 4, 0, 2, 0, 0) == 0  # no prefix
    assert lib.pa_decode_step_host_staging_bytes(4, 8, 2, 128, 16, 8, 100, 4, 2, 2, 1, 0) > need

    def step(out=buf, q=buf, nk=buf, T=4, pairs=None, n=0, B=4, S=0, pb=0, stg=buf, stg_bytes=1 << 30):
        return lib.pa_decode_step_host(out, q, nk, buf, buf, T, pairs, n, buf, 8, buf, B, S, pb, 8, 2, 128, 16,
                                       64, buf, buf, 100, f(0.1), 0, 1, stg, stg_bytes, None, None)
    assert step(B=0) == -1
    assert step(out=None) == -1
    assert step(q=None) == -1
    assert step(nk=None) == -1                  # new tokens without their keys
    assert step(n=2) == -1                      # copy pairs without the list
    assert step(S=2) == -1                      # groups without a shared prefix
    assert step(stg=None) == -5
    assert step(stg_bytes=need - 1) == -5
    assert step(stg=p((1 << 20) + 16)) == -6    # staging not 256-byte aligned


def test_mixed_step_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    buf = p(1 << 20)
    f = ctypes.c_float
    pl = (ctypes.c_int * 2)(10, 0)
    cl = (ctypes.c_int * 2)(4, 3)

    def mixed(npf=2, ndec=3, Hq=8, Hkv=2, scale=0.1):
        return lib.pa_mixed_step(buf, buf, buf, 4, pl, cl, npf, buf, buf, buf, 4, buf, ndec, 64, 0, buf, 1 << 30,
                                 buf, buf, Hq, Hkv, 128, 16, 64, f(scale), 1, None, None)
    assert mixed(npf=-1) == -1
    assert mixed(ndec=-1) == -1
    assert mixed(npf=0, ndec=0) == 0            # nothing to do, no CUDA call
    assert mixed(npf=0, Hq=6, Hkv=4) == -1      # heads not a multiple of kv heads
    assert mixed(ndec=0, scale=-1.0) == -3      # prefill half rejects a negative scale


def test_block_manager_status_strings(lib):
    assert b"no free block" in lib.pa_status_string(-8) or b"exhausted" in lib.pa_status_string(-8)


def test_product_path_has_no_oracle_import():
    # the package must not reach the CPU oracle (only tests, smoke and the
    # benchmark's CPU legs may)
    pkg = os.path.join(ROOT, "paged_kv_cache_224_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.c" not in text, f
