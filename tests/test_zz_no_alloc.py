"""pa_decode_noalloc: the decode entry point for callers that cannot allocate.

Some hosts cannot call cudaMalloc on the decode path -- an engine that has
given nearly all HBM to its KV-cache pool, or a loop that cannot take the
device-wide synchronisation an allocation implies.  For them the library
keeps the split-K partials in its own fixed device array.  These tests call
that entry point through the C ABI and check that it gives bit-identical
outputs to pa_decode with a caller-owned workspace (the same kernels and
partitions; only where the partials live differs) and outputs within the
attention tolerance of the CPU oracle, on two calls in a row -- including a
small call right after a large one has filled the array, since the array
keeps the previous call's contents -- and that sizes beyond the array are
refused without launching anything.

This file is collected last on purpose: a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl
from tests.helpers import check_attention, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _decode_both(case, t, partition_tokens):
    bt = torch.as_tensor(case.block_tables, device=DEV)
    lens = torch.as_tensor(case.context_lens, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref = torch.full_like(t["query"], float("nan"))
    pa.pa_decode(ref, t["query"], t["k_cache"], t["v_cache"], bt, lens, case.scale, case.max_context_len,
                 partition_tokens=partition_tokens, d_err=err)
    got = torch.full_like(t["query"], float("nan"))
    # straight through the C ABI: no workspace argument exists
    L = pa.lib()
    rc = L.pa_decode_noalloc(
        ctypes.c_void_p(got.data_ptr()), ctypes.c_void_p(t["query"].data_ptr()),
        ctypes.c_void_p(t["k_cache"].data_ptr()), ctypes.c_void_p(t["v_cache"].data_ptr()),
        ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(lens.data_ptr()),
        case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim, case.block_size,
        case.num_blocks, case.max_context_len, case.scale, partition_tokens,
        1 if case.dtype == "bf16" else 0, ctypes.c_void_p(err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert rc == 0, pa.pa_status_string(rc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ref, got


def _oracle_decode(case, t):
    return oracle.decode(wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"]), case.block_tables,
                         case.context_lens, case.scale, case.dtype, num_threads=8)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("partition_tokens", [0, 512])
def test_noalloc_matches_pa_decode_on_two_calls(dtype, partition_tokens):
    # lengths span one and many partitions, so the scratch holds partials
    lens_a = [1, 17, 700, 1500, 3000, 4096, 513, 64]
    lens_b = [2500, 5, 1024, 1025, 33, 3999]
    for i, lens in enumerate((lens_a, lens_b)):
        c = wl.make_decode_case(f"noalloc{i}", lens, 8, 2, 128, 16, dtype, seed=500 + i)
        assert pa.pa_decode_workspace_bytes(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size,
                                            c.max_context_len, partition_tokens) > 0
        t = c.materialize(DEV)
        ref, got = _decode_both(c, t, partition_tokens=partition_tokens)
        assert torch.equal(got, ref)
        check_attention(to_f64(got), _oracle_decode(c, t), dtype, c.name)


def test_noalloc_small_call_after_a_large_one_is_exact():
    # the first call fills most of the scratch with partials (many sequences,
    # 256-token partitions, head group 8 on the tensor cores); the second,
    # much smaller call on the same stream reads only what it wrote itself
    rng = np.random.default_rng(77)
    big_lens = [int(x) for x in rng.integers(3000, 8192, size=48)]
    big = wl.make_decode_case("noalloc_big", big_lens, 64, 8, 128, 16, "bf16", seed=71)
    need = pa.pa_decode_workspace_bytes(big.num_seqs, big.num_heads, big.num_kv_heads, big.head_dim,
                                        big.block_size, big.max_context_len, 256)
    assert pa.capi.NOALLOC_SCRATCH_BYTES // 2 < need <= pa.capi.NOALLOC_SCRATCH_BYTES
    tb = big.materialize(DEV)
    ref_b, got_b = _decode_both(big, tb, partition_tokens=256)
    assert torch.equal(got_b, ref_b)
    small = wl.make_decode_case("noalloc_small", [300, 1, 1200, 77], 8, 2, 128, 16, "bf16", seed=72)
    ts = small.materialize(DEV)
    ref_s, got_s = _decode_both(small, ts, partition_tokens=256)
    assert torch.equal(got_s, ref_s)
    check_attention(to_f64(got_s), _oracle_decode(small, ts), "bf16", small.name)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    c = wl.make_decode_case("tiny", [8], 4, 1, 128, 16, "bf16", seed=1)
    t = c.materialize(DEV)
    B, Hq, D, bs, maxlen = 512, 64, 128, 16, 131072  # partials far beyond 64 MiB
    need = pa.pa_decode_workspace_bytes(B, Hq, 8, D, bs, maxlen, 0)
    assert need > pa.capi.NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p
    rc = pa.lib().pa_decode_noalloc(p(t["query"].data_ptr()), p(t["query"].data_ptr()),
                                    p(t["k_cache"].data_ptr()), p(t["v_cache"].data_ptr()),
                                    p(t["k_cache"].data_ptr()), maxlen // bs, p(t["k_cache"].data_ptr()),
                                    B, Hq, 8, D, bs, c.num_blocks, maxlen, 0.1, 0, 1, None, None)
    assert rc == pa.capi.PA_ERR_SCRATCH_LIMIT
    assert "scratch" in pa.pa_status_string(rc)
