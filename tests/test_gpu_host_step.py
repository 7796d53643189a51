"""A whole decode step from host-resident inputs (pa_decode_step_host).

The step a scheduler runs per generated token: copy-on-write pairs, the new
tokens' K/V into their slots, attention over the block tables (page "vLLM
PagedAttention chuyen sau", sections "Co che PagedAttention" and "Co che
APC").  Through the host entry point the output and the pool it leaves must
equal, bit for bit, the same step made of the device-pointer calls, and the
output must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl
from tests.helpers import check_attention, oracle_inputs, oracle_step, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def device_step(case, t, grouped, partition_tokens):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if case.cow_pairs.shape[0]:
        pa.pa_copy_blocks(t["k_cache"], t["v_cache"], torch.as_tensor(case.cow_pairs, device=DEV), d_err=err)
    if case.slot_mapping.size:
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"],
                                torch.as_tensor(case.slot_mapping, device=DEV), d_err=err)
    out = torch.full_like(t["query"], float("nan"))
    bt = torch.as_tensor(case.block_tables, device=DEV)
    lens = torch.as_tensor(case.context_lens, device=DEV)
    if grouped:
        pa.pa_decode_shared_prefix(out, t["query"], t["k_cache"], t["v_cache"], bt, lens, case.scale,
                                   case.max_context_len, case.group_size, case.shared_blocks,
                                   partition_tokens=partition_tokens, d_err=err)
    else:
        pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], bt, lens, case.scale, case.max_context_len,
                     partition_tokens=partition_tokens, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def host_step(case, t, grouped, partition_tokens):
    pin = lambda x: x.cpu().pin_memory()  # noqa: E731
    out = torch.full(tuple(t["query"].shape), float("nan"), dtype=t["query"].dtype).pin_memory()
    pairs = pin(torch.as_tensor(case.cow_pairs)) if case.cow_pairs.shape[0] else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_decode_step_host(out, pin(t["query"]), pin(t["new_key"]), pin(t["new_value"]),
                           pin(torch.as_tensor(case.slot_mapping)), pin(torch.as_tensor(case.block_tables)),
                           pin(torch.as_tensor(case.context_lens)), t["k_cache"], t["v_cache"], case.scale,
                           case.max_context_len, pairs=pairs, group_size=case.group_size if grouped else 0,
                           prefix_blocks=case.shared_blocks if grouped else 0, partition_tokens=partition_tokens,
                           d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


@pytest.mark.parametrize("G,dtype,pt", [(4, "bf16", 0), (1, "f16", 256), (8, "bf16", 512)])
def test_host_step_equals_the_device_calls_and_the_oracle(G, dtype, pt):
    lens = [1, 130, 700, 2049, 0, 513, 64]
    c = wl.make_decode_case(f"host_g{G}", lens, 2 * G, 2, 128, 16, dtype, seed=60 + G)
    t = c.materialize(DEV)
    ref = oracle_step(oracle, c, oracle_inputs(c, t, range(c.num_seqs)))
    t_dev = {k: v.clone() for k, v in t.items()}
    out_dev = device_step(c, t_dev, False, pt)
    out_host = host_step(c, t, False, pt)
    assert torch.equal(out_host, out_dev.cpu())
    assert torch.equal(t["k_cache"], t_dev["k_cache"]) and torch.equal(t["v_cache"], t_dev["v_cache"])
    check_attention(to_f64(out_host), ref, dtype, c.name)


def test_host_step_shared_prefix_with_copy_on_write():
    c = wl.make_shared_prefix_case("host_sp", num_prompts=3, samples=4, prefix_len=200, max_tail=300,
                                   num_heads=8, head_dim=128, block_size=16, dtype="bf16", seed=61,
                                   num_kv_heads=4)
    assert c.cow_pairs.shape[0] > 0
    t = c.materialize(DEV)
    t_dev = {k: v.clone() for k, v in t.items()}
    out_dev = device_step(c, t_dev, True, 0)
    out_host = host_step(c, t, True, 0)
    assert torch.equal(out_host, out_dev.cpu())
    assert torch.equal(t["k_cache"], t_dev["k_cache"]) and torch.equal(t["v_cache"], t_dev["v_cache"])
    assert np.isfinite(to_f64(out_host)).all()


def test_host_step_without_new_tokens_or_pairs():
    # a step that only attends (the new tokens were written earlier): no cache
    # write is queued, and the output equals the device-pointer decode
    c = wl.make_decode_case("host_noop", [1, 300, 700], 8, 2, 128, 16, "bf16", seed=66)
    t = c.materialize(DEV)
    ref = torch.full_like(t["query"], float("nan"))
    pa.pa_decode(ref, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(c.block_tables, device=DEV),
                 torch.as_tensor(c.context_lens, device=DEV), c.scale, c.max_context_len)
    before = t["k_cache"].clone()
    out = torch.full(tuple(t["query"].shape), float("nan"), dtype=t["query"].dtype).pin_memory()
    empty_kv = t["new_key"][:0].cpu().pin_memory()
    pa.pa_decode_step_host(out, t["query"].cpu().pin_memory(), empty_kv, empty_kv,
                           torch.zeros(0, dtype=torch.int64).pin_memory(),
                           torch.as_tensor(c.block_tables).pin_memory(), torch.as_tensor(c.context_lens).pin_memory(),
                           t["k_cache"], t["v_cache"], c.scale, c.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out, ref.cpu())
    assert torch.equal(t["k_cache"], before)


def test_host_step_pageable_and_unaligned_inputs_equal_the_pinned_step():
    # page-locked inputs are read by one gather kernel (16-byte vectors, or
    # bytes when an end or the size is not a multiple of 16) and a
    # page-locked, aligned output is written by the kernels in place; anything
    # else is copied with cudaMemcpyAsync.  Every route gives the same bits.
    c = wl.make_decode_case("host_mix", [5, 130, 701, 33, 1000], 8, 2, 128, 16, "bf16", seed=67)
    t = c.materialize(DEV)
    t_pin, t_page, t_odd = ({k: v.clone() for k, v in t.items()} for _ in range(3))
    out_pin = host_step(c, t_pin, False, 0)

    def run(tt, conv):
        out = conv(torch.full(tuple(tt["query"].shape), float("nan"), dtype=tt["query"].dtype))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        pa.pa_decode_step_host(out, conv(tt["query"]), conv(tt["new_key"]), conv(tt["new_value"]),
                               conv(torch.as_tensor(c.slot_mapping)), conv(torch.as_tensor(c.block_tables)),
                               conv(torch.as_tensor(c.context_lens)), tt["k_cache"], tt["v_cache"], c.scale,
                               c.max_context_len, d_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        return out

    def odd(x):
        # page-locked, but starting one element past a 16-byte boundary
        x = x.cpu()
        buf = torch.empty(x.numel() + 1, dtype=x.dtype).pin_memory()
        v = buf[1:].view(x.shape)
        v.copy_(x)
        return v

    out_page = run(t_page, lambda x: x.cpu())
    out_odd = run(t_odd, odd)
    assert torch.equal(out_page, out_pin) and torch.equal(out_odd, out_pin)
    for tt in (t_page, t_odd):
        assert torch.equal(tt["k_cache"], t_pin["k_cache"]) and torch.equal(tt["v_cache"], t_pin["v_cache"])
