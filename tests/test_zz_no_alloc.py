"""pa_decode_noalloc: the decode entry point for callers that cannot allocate.

Some hosts cannot call cudaMalloc on the decode path -- an engine that has
given nearly all HBM to its KV-cache pool, or a loop that cannot take the
device-wide synchronisation an allocation implies.  For them the library
keeps the split-K partials in its own fixed device array.  These tests call
that entry point through the C ABI and check that it gives the same outputs
as pa_decode with a caller-owned workspace, on two calls in a row (the array
keeps the previous call's contents), and that sizes beyond the array are
refused without launching anything.

This file is collected last on purpose: a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl
from tests.helpers import TOL, to_f64

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


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_noalloc_matches_pa_decode_on_two_calls(dtype):
    # lengths span one and many 512-token partitions, so the scratch holds partials
    lens_a = [1, 17, 700, 1500, 3000, 4096, 513, 64]
    lens_b = [2500, 5, 1024, 1025, 33, 3999]
    for i, lens in enumerate((lens_a, lens_b)):
        c = wl.make_decode_case(f"noalloc{i}", lens, 8, 2, 128, 16, dtype, seed=500 + i)
        assert pa.pa_decode_workspace_bytes(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size,
                                            c.max_context_len, 0) > 0
        t = c.materialize(DEV)
        ref, got = _decode_both(c, t, partition_tokens=0)
        assert torch.isfinite(got.float()).all()
        diff = (to_f64(got) - to_f64(ref))
        assert np.abs(diff).max() <= TOL[dtype]


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
