"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic partitioning): every output element of every
sequence is compared with the oracle, plus whole-output properties (every new
row at its slot, every copy-on-write destination equal to its source).

Workloads: OPT-13B-shaped MHA (64 seqs, fp16), LLaMA-style GQA (256 seqs,
bf16), parallel sampling with a shared 1000-token prefix (32x8, fp16,
copy-on-write), long context (8 seqs of 32k-131k tokens, bs 16 and 32,
split-K) -- the tiny workload is covered in full in test_gpu_decode.
"""
import os

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


def full_step_and_check(case, partition_tokens=0):
    t = case.materialize(DEV)
    seqs = list(range(case.num_seqs))
    inp = oracle_inputs(case, t, seqs)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if case.cow_pairs.shape[0]:
        pairs = torch.as_tensor(case.cow_pairs, device=DEV)
        pa.pa_copy_blocks(t["k_cache"], t["v_cache"], pairs, d_err=err)
        # property: every destination now equals its source, bit for bit
        torch.cuda.synchronize()
        assert torch.equal(t["k_cache"][pairs[:, 1]], t["k_cache"][pairs[:, 0]])
        assert torch.equal(t["v_cache"][pairs[:, 1]], t["v_cache"][pairs[:, 0]])
    slots = torch.as_tensor(case.slot_mapping, device=DEV)
    pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)
    out = torch.full_like(t["query"], float("nan"))
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(case.block_tables, device=DEV),
                 torch.as_tensor(case.context_lens, device=DEV), case.scale, case.max_context_len,
                 partition_tokens=partition_tokens, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    # property over every new token: its rows sit exactly at its slot
    blk = slots // case.block_size
    off = slots % case.block_size
    assert torch.equal(t["k_cache"][blk, :, off, :], t["new_key"])
    assert torch.equal(t["v_cache"][blk, :, off, :], t["new_value"])
    # property over every output: finite
    assert torch.isfinite(out.float()).all()
    ref = oracle_step(oracle, case, inp, threads=os.cpu_count() or 8)
    got = to_f64(out[torch.as_tensor(seqs, device=DEV)])
    return check_attention(got, ref, case.dtype, case.name)


def test_opt13b_mha_full_size():
    full_step_and_check(wl.opt13b_case())


def test_llama_gqa_full_size():
    c = wl.llama_gqa_case()
    assert c.num_seqs == 256 and c.max_blocks_per_seq == wl.blocks_for(c.max_context_len, 16)
    assert 1 <= c.context_lens.min() and c.context_lens.max() <= 4096
    full_step_and_check(c)


def test_shared_prefix_full_size():
    c = wl.shared_prefix_case()
    assert c.cow_pairs.shape == (224, 2)
    assert int(c.refcounts.max()) == 8
    full_step_and_check(c)


@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_full_size(bs):
    c = wl.long_context_case(block_size=bs)
    assert pa.pa_decode_partition_tokens(c.num_seqs, c.num_heads, c.num_kv_heads, bs, c.max_context_len) == 2048
    full_step_and_check(c)
