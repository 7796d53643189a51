"""Failure detection without a GPU fault.

Every wait inside the kernels is bounded: when a copy or MMA completion never
arrives, the wait gives up, the kernel flags PA_DEVERR_TIMEOUT in the
caller's error word and returns, and the context stays usable.  The
self-test entry point runs that same wait on a barrier nothing ever arrives
on (a flag that nothing sets) -- no fault, no trap, no endless loop.
"""
import pytest
import torch

import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl
from tests.helpers import check_attention, oracle_inputs, oracle_step, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def test_bounded_wait_gives_up_flags_and_leaves_the_context_usable():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cyc = torch.zeros(1, dtype=torch.int64, device=DEV)
    pa.pa_selftest_bounded_wait(1000, err, cyc)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.capi.DEVERR["timeout"]
    assert int(cyc.item()) > 0
    # how long the kernels' own bound lasts on this GPU
    err.zero_()
    pa.pa_selftest_bounded_wait(1 << 16, err, cyc)
    torch.cuda.synchronize()
    per_poll = int(cyc.item()) / (1 << 16)
    bound_s = per_poll * pa.lib().pa_bounded_wait_polls() / 2.0e9
    print(f"bounded wait: {per_poll:.1f} cycles per poll, kernel bound {bound_s:.3f} s at 2 GHz")
    assert int(err.item()) == pa.capi.DEVERR["timeout"]
    assert 0.05 < bound_s < 5.0  # about a second: long enough for any real wait, short enough to report a stall
    # the context still runs the decode path and gets it right
    import oracle
    c = wl.make_decode_case("after_timeout", [1, 130, 700], 8, 2, 128, 16, "bf16", seed=31)
    t = c.materialize(DEV)
    ref = oracle_step(oracle, c, oracle_inputs(c, t, range(c.num_seqs)))
    err.zero_()
    pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"],
                            torch.as_tensor(c.slot_mapping, device=DEV), d_err=err)
    out = torch.empty_like(t["query"])
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(c.block_tables, device=DEV),
                 torch.as_tensor(c.context_lens, device=DEV), c.scale, c.max_context_len, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_attention(to_f64(out), ref, c.dtype, c.name)
