"""GPU parity of the shared-prefix decode (parallel sampling) against the oracle.

Samples of one prompt reference the same physical prefix blocks ("vLLM
PagedAttention chuyen sau", section "Co che APC"; "vLLM", section
"PagedAttention").  pa_decode_shared_prefix reads each shared block once per
group and merges it with each sample's own tokens; its outputs must equal
the oracle's attention over every sequence's whole context (which knows
nothing about sharing) within the attention tolerance, and match pa_decode.
Covered: MHA and GQA groups, tails of zero tokens, a prefix with a
copy-on-write partial block, the full-size 32x8 workload on sampled
sequences, and the device checks of the sharing promise.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl
from tests.helpers import TOL, check_attention, oracle_inputs, oracle_step, sample_seqs, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def run_step(case, t, shared=True, partition_tokens=0):
    """Copy-on-write, cache write, then the shared-prefix (or plain) decode."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if case.cow_pairs.shape[0]:
        pa.pa_copy_blocks(t["k_cache"], t["v_cache"], torch.as_tensor(case.cow_pairs, device=DEV), d_err=err)
    if case.slot_mapping.size:
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"],
                                torch.as_tensor(case.slot_mapping, device=DEV), d_err=err)
    out = torch.full_like(t["query"], float("nan"))
    bt = torch.as_tensor(case.block_tables, device=DEV)
    lens = torch.as_tensor(case.context_lens, device=DEV)
    if shared:
        pa.pa_decode_shared_prefix(out, t["query"], t["k_cache"], t["v_cache"], bt, lens, case.scale,
                                   case.max_context_len, case.group_size, case.shared_blocks,
                                   partition_tokens=partition_tokens, d_err=err)
    else:
        pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], bt, lens, case.scale, case.max_context_len,
                     partition_tokens=partition_tokens, d_err=err)
    torch.cuda.synchronize()
    return out, int(err.item())


CASES = [
    # (prompts, samples, prefix_len, max_tail, Hq, Hkv, D, bs, dtype)
    (3, 4, 100, 80, 4, 4, 128, 16, "f16"),     # MHA, COW partial block, vgroup 4
    (2, 8, 96, 40, 3, 3, 128, 16, "bf16"),     # MHA, prefix = whole blocks, vgroup 8
    (2, 4, 200, 600, 8, 4, 128, 32, "bf16"),   # GQA G=2 x 4 samples, tails over a partition
    (4, 2, 530, 30, 8, 2, 64, 16, "f16"),      # GQA G=4 x 2, prefix spans two partitions, D=64
    (2, 2, 64, 0, 2, 2, 128, 16, "bf16"),      # every tail empty: L == prefix
    (2, 1, 160, 300, 16, 2, 128, 16, "bf16"),  # GQA G=8, one sample: both passes are group-of-8 decodes
    (2, 2, 256, 100, 8, 2, 128, 64, "f16"),    # GQA G=4 x 2 samples at block_size 64
]


@pytest.mark.parametrize("P,S,prefix,tail,Hq,Hkv,D,bs,dtype", CASES)
def test_shared_prefix_matches_oracle_and_plain_decode(P, S, prefix, tail, Hq, Hkv, D, bs, dtype):
    case = wl.make_shared_prefix_case(f"sp{P}x{S}_{prefix}", P, S, prefix, tail, Hq, D, bs, dtype,
                                      seed=prefix + tail + S, num_kv_heads=Hkv)
    assert case.group_size == S and case.shared_blocks == prefix // bs
    t = case.materialize(DEV)
    inp = oracle_inputs(case, t, range(case.num_seqs))
    t2 = {k: v.clone() for k, v in t.items()}
    out, err = run_step(case, t)
    assert err == 0, f"device error flags {err:#x}"
    ref = oracle_step(oracle, case, inp)
    check_attention(to_f64(out), ref, dtype, case.name)
    plain, err2 = run_step(case, t2, shared=False)
    assert err2 == 0
    assert np.abs(to_f64(out) - to_f64(plain)).max() <= 2 * TOL[dtype]


def test_shared_prefix_partition_sizes_agree():
    case = wl.make_shared_prefix_case("sp_pt", 2, 4, 300, 300, 4, 128, 16, "bf16", seed=31, num_kv_heads=2)
    t = case.materialize(DEV)
    inp = oracle_inputs(case, t, range(case.num_seqs))
    ref = None
    for pt in (0, 64, 256, 1024):
        tt = {k: v.clone() for k, v in t.items()}
        out, err = run_step(case, tt, partition_tokens=pt)
        assert err == 0
        if ref is None:
            ref = oracle_step(oracle, case, inp)
        check_attention(to_f64(out), ref, "bf16", f"pt={pt}")


def test_shared_prefix_full_size_workload():
    case = wl.shared_prefix_case()
    assert (case.group_size, case.shared_blocks) == (8, 62)
    t = case.materialize(DEV)
    seqs = sample_seqs(case, 10)
    inp = oracle_inputs(case, t, seqs)
    out, err = run_step(case, t)
    assert err == 0, f"device error flags {err:#x}"
    assert torch.isfinite(out.float()).all()
    ref = oracle_step(oracle, case, inp, threads=16)
    check_attention(to_f64(out[torch.as_tensor(seqs, device=DEV)]), ref, case.dtype, case.name)


def test_broken_sharing_promises_are_flagged():
    case = wl.make_shared_prefix_case("sp_bad", 2, 4, 64, 20, 2, 128, 16, "f16", seed=5)
    t = case.materialize(DEV)
    run_step(case, t)  # apply the cache writes once
    bt = torch.as_tensor(case.block_tables, device=DEV)
    lens = torch.as_tensor(case.context_lens, device=DEV)
    out = torch.empty_like(t["query"])
    # a member whose prefix row points elsewhere
    bad = bt.clone()
    bad[1, 0] = bt[5, 0]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_decode_shared_prefix(out, t["query"], t["k_cache"], t["v_cache"], bad, lens, case.scale,
                               case.max_context_len, 4, case.shared_blocks, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x20
    # a context shorter than the shared prefix
    short = lens.clone()
    short[2] = case.shared_blocks * case.block_size - 1
    err.zero_()
    pa.pa_decode_shared_prefix(out, t["query"], t["k_cache"], t["v_cache"], bt, short, case.scale,
                               case.max_context_len, 4, case.shared_blocks, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x4


def test_shared_prefix_host_argument_errors():
    case = wl.make_shared_prefix_case("sp_args", 2, 4, 64, 20, 2, 128, 16, "f16", seed=6)
    t = case.materialize(DEV)
    bt = torch.as_tensor(case.block_tables, device=DEV)
    lens = torch.as_tensor(case.context_lens, device=DEV)
    out = torch.empty_like(t["query"])
    args = (out, t["query"], t["k_cache"], t["v_cache"], bt, lens, case.scale, case.max_context_len)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_shared_prefix(*args, 3, case.shared_blocks)  # 8 seqs not a multiple of 3
    assert e.value.status == -1
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_shared_prefix(*args, 8, 0)  # no prefix
    assert e.value.status == -1
    with pytest.raises(pa.PAError) as e:
        big = wl.make_shared_prefix_case("sp_g16", 1, 16, 32, 4, 1, 128, 16, "f16", seed=7)
        tb = big.materialize(DEV)
        pa.pa_decode_shared_prefix(torch.empty_like(tb["query"]), tb["query"], tb["k_cache"], tb["v_cache"],
                                   torch.as_tensor(big.block_tables, device=DEV),
                                   torch.as_tensor(big.context_lens, device=DEV), big.scale, big.max_context_len,
                                   16, big.shared_blocks)  # 16 samples per group: no such head group
    assert e.value.status == -2
    tiny = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_shared_prefix(*args, 4, case.shared_blocks, workspace=tiny)
    assert e.value.status == -5
