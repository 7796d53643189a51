"""GPU parity of chunked prefill against the CPU oracle, through the C ABI.

A chunk of C query rows at positions P..P+C-1 attends causally over the
paged prefix plus itself (page "vLLM PagedAttention chuyen sau", section
"Chunked Prefill").  Checked: small ragged cases against the oracle in full,
the full 8192-token-prefix / 512-token-chunk workload on every row, a whole
prompt prefilled chunk after chunk (each chunk's K/V written, then its
attention over everything written so far) against one oracle prefill of the
whole prompt, and the pages' "KV accumulates chunk by chunk" invariant:
writing a prompt's K/V chunk by chunk leaves the cache bit-identical to one
write.
"""
import os

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


def run_prefill(case, t, split=True):
    """Cache write then prefill; ``split``: with a workspace (stream-K over one
    CTA per SM, partial units merged), else one CTA per unit."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"],
                            torch.as_tensor(case.slot_mapping, device=DEV), d_err=err)
    out = torch.full_like(t["query"], float("nan"))
    ws = pa.prefill_workspace(t["query"], case.num_kv_heads) if split else None
    pa.pa_prefill_chunk(out, t["query"], t["k_cache"], t["v_cache"],
                        torch.as_tensor(case.block_table, device=DEV), case.prefix_len, case.scale, d_err=err,
                        workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    return out


CASES = [
    # (P, C, G, Hkv, bs, dtype)
    (40, 9, 2, 2, 16, "bf16"),
    (0, 17, 4, 1, 32, "f16"),
    (100, 64, 8, 2, 16, "bf16"),
    (333, 77, 1, 3, 16, "f16"),
    (1000, 130, 4, 2, 32, "bf16"),
    (64, 1, 8, 1, 16, "bf16"),
    (200, 150, 2, 2, 64, "bf16"),
    (300, 70, 8, 1, 128, "f16"),
]


@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("P,C,G,Hkv,bs,dtype", CASES)
def test_prefill_chunk_matches_oracle(P, C, G, Hkv, bs, dtype, split):
    case = wl.make_prefill_case(f"pf{P}_{C}", P, C, G * Hkv, Hkv, 128, bs, dtype, seed=P + 7 * C + G)
    t = case.materialize(DEV)
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc,
                                    case.slot_mapping, bs) == 0
    ref = oracle.prefill_chunk(wl.bits(t["query"]), kc, vc, case.block_table, P, case.scale, dtype,
                               num_threads=8)
    out = run_prefill(case, t, split)
    check_attention(to_f64(out), ref, dtype, case.name)


@pytest.mark.parametrize("P,C,G,Hkv,bs,dtype", [
    (8000, 32, 8, 1, 16, "bf16"),    # one unit of 64 key tiles over 64 CTAs: one tile each, 64 partials merged
    (0, 256, 1, 2, 16, "f16"),       # 2 units of 2 tiles over 4 CTAs: rows 0-127 see nothing in the second tile
    (300, 40, 4, 3, 32, "bf16"),     # units of 3 tiles, ranges of one or two tiles
    (5000, 700, 8, 2, 16, "bf16"),   # 22 units, several cut
])
def test_prefill_split_units_merge_to_the_oracle(P, C, G, Hkv, bs, dtype):
    # stream-K ranges cut units into segments whose partials are merged by
    # the last one to finish; some segments hold no visible key for some rows
    case = wl.make_prefill_case(f"pfsplit{P}_{C}", P, C, G * Hkv, Hkv, 128, bs, dtype, seed=11 + P + C)
    t = case.materialize(DEV, pool_fill=float("nan"))
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc,
                                    case.slot_mapping, bs) == 0
    ref = oracle.prefill_chunk(wl.bits(t["query"]), kc, vc, case.block_table, P, case.scale, dtype,
                               num_threads=8)
    out = run_prefill(case, t, split=True)
    assert torch.isfinite(out.float()).all()
    check_attention(to_f64(out), ref, dtype, case.name)
    # the merge follows key order, not arrival order: a second run gives the same bits
    again = run_prefill(case, t, split=True)
    assert torch.equal(out, again)


def test_prefill_full_size_every_row():
    case = wl.chunked_prefill_case()
    assert (case.prefix_len, case.chunk_len, case.num_heads, case.num_kv_heads) == (8192, 512, 64, 8)
    t = case.materialize(DEV)
    n = wl.blocks_for(case.prefix_len + case.chunk_len, case.block_size)
    idx = torch.as_tensor(case.block_table[:n], dtype=torch.long, device=DEV)
    kc = wl.bits(t["k_cache"].index_select(0, idx))
    vc = wl.bits(t["v_cache"].index_select(0, idx))
    compact = np.arange(n, dtype=np.int32)
    pos = np.arange(case.prefix_len, case.prefix_len + case.chunk_len)
    slots = compact[pos // case.block_size].astype(np.int64) * case.block_size + pos % case.block_size
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc, slots,
                                    case.block_size) == 0
    q = wl.bits(t["query"])
    out = run_prefill(case, t)          # the benchmark's schedule: stream-K with a workspace
    ref = oracle.prefill_chunk(q, kc, vc, compact, case.prefix_len, case.scale, case.dtype,
                               num_threads=os.cpu_count() or 8)
    check_attention(to_f64(out), ref, case.dtype, case.name)
    whole = run_prefill(case, t, split=False)
    check_attention(to_f64(whole), ref, case.dtype, case.name + " one CTA per unit")


@pytest.mark.parametrize("chunks,bs", [([512, 512, 512, 512], 16), ([700, 13, 1335], 16),
                                       ([512, 512, 512, 512], 32), ([1, 300, 1747], 32)])
def test_prompt_prefilled_chunk_after_chunk(chunks, bs):
    # one 2048-token prompt, 64/8 heads, bf16: for each chunk, write its K/V
    # into the paged cache, then attend over the prefix written so far plus
    # the chunk.  Every row of every chunk must match one oracle prefill of the
    # whole prompt over the final cache, and the final cache must equal the
    # oracle's, bit for bit.
    total = sum(chunks)
    case = wl.make_prefill_case(f"prompt{len(chunks)}_{bs}", 0, total, 64, 8, 128, bs, "bf16", seed=2048 + bs)
    t = case.materialize(DEV)
    kc0, vc0 = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc0, vc0,
                                    case.slot_mapping, bs) == 0
    ref = oracle.prefill_chunk(wl.bits(t["query"]), kc0, vc0, case.block_table, 0, case.scale, "bf16",
                               num_threads=os.cpu_count() or 8)
    slots = torch.as_tensor(case.slot_mapping, device=DEV)
    bt = torch.as_tensor(case.block_table, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full_like(t["query"], float("nan"))
    ws = pa.prefill_workspace(t["query"], case.num_kv_heads)
    a = 0
    for c in chunks:
        b = a + c
        pa.pa_reshape_and_cache(t["new_key"][a:b].contiguous(), t["new_value"][a:b].contiguous(), t["k_cache"],
                                t["v_cache"], slots[a:b].contiguous(), d_err=err)
        part = torch.full_like(t["query"][a:b], float("nan"))
        pa.pa_prefill_chunk(part, t["query"][a:b].contiguous(), t["k_cache"], t["v_cache"], bt, a, case.scale,
                            d_err=err, workspace=ws)
        out[a:b] = part
        a = b
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    assert np.array_equal(wl.bits(t["k_cache"]), kc0) and np.array_equal(wl.bits(t["v_cache"]), vc0)
    check_attention(to_f64(out), ref, "bf16", case.name)


def test_prefill_row_equals_gpu_decode_at_that_position():
    case = wl.make_prefill_case("pd", 500, 40, 8, 2, 128, 16, "bf16", seed=9)
    t = case.materialize(DEV)
    out = run_prefill(case, t)
    bt = torch.as_tensor(case.block_table[None, :], device=DEV)
    for i in (0, 17, 39):
        dec = torch.empty_like(t["query"][i:i + 1])
        L = torch.tensor([case.prefix_len + i + 1], dtype=torch.int32, device=DEV)
        pa.pa_decode(dec, t["query"][i:i + 1].contiguous(), t["k_cache"], t["v_cache"], bt, L, case.scale,
                     case.prefix_len + i + 1)
        torch.cuda.synchronize()
        assert (dec.float() - out[i:i + 1].float()).abs().max().item() <= 1e-2


def test_chunkwise_cache_writes_are_bit_identical_to_one_write():
    case = wl.make_prefill_case("acc", 0, 300, 4, 2, 128, 16, "bf16", seed=3)
    t = case.materialize(DEV)
    slots = torch.as_tensor(case.slot_mapping, device=DEV)
    kc1, vc1 = t["k_cache"].clone(), t["v_cache"].clone()
    pa.pa_reshape_and_cache(t["new_key"], t["new_value"], kc1, vc1, slots)
    kc2, vc2 = t["k_cache"].clone(), t["v_cache"].clone()
    for a in range(0, 300, 64):
        b = min(300, a + 64)
        pa.pa_reshape_and_cache(t["new_key"][a:b].contiguous(), t["new_value"][a:b].contiguous(), kc2, vc2,
                                slots[a:b].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)


@pytest.mark.parametrize("P,C,G,bs", [(37, 20, 4, 16), (500, 45, 8, 32), (0, 5, 1, 16)])
def test_prefill_ignores_nan_garbage_past_the_chunk(P, C, G, bs):
    # every slot past position P+C-1 holds NaN: only keys 0..P+i may reach row i
    case = wl.make_prefill_case(f"pfnan{P}_{C}", P, C, 2 * G, 2, 128, bs, "bf16", seed=900 + P + C)
    t = case.materialize(DEV, pool_fill=float("nan"))
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc,
                                    case.slot_mapping, bs) == 0
    ref = oracle.prefill_chunk(wl.bits(t["query"]), kc, vc, case.block_table, P, case.scale, "bf16",
                               num_threads=8)
    out = run_prefill(case, t)
    assert torch.isfinite(out.float()).all()
    check_attention(to_f64(out), ref, "bf16", case.name)


BATCHES = [
    # (prefix_lens, chunk_lens, G, Hkv, bs, dtype)
    ([40, 0, 333, 1000], [9, 17, 0, 130], 8, 2, 16, "bf16"),   # an empty chunk, a prefix of 0
    ([100, 64, 7], [64, 1, 200], 2, 2, 32, "f16"),
    ([0, 0, 0, 0, 0], [3, 300, 17, 64, 1], 4, 1, 16, "bf16"),
]


def _oracle_batch(case, t):
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc,
                                    case.slot_mapping, case.block_size) == 0
    q = wl.bits(t["query"])
    refs, row = [], 0
    for i, (P, C) in enumerate(zip(case.prefix_lens.tolist(), case.chunk_lens.tolist())):
        if C:
            refs.append((row, oracle.prefill_chunk(q[row:row + C], kc, vc, case.block_tables[i], P, case.scale,
                                                   case.dtype, num_threads=8)))
        row += C
    return refs


def _gpu_batch(case, t, split=False):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"],
                            torch.as_tensor(case.slot_mapping, device=DEV), d_err=err)
    out = torch.full_like(t["query"], float("nan"))
    ws = pa.prefill_workspace(t["query"], case.num_kv_heads, len(case.chunk_lens)) if split else None
    pa.pa_prefill_batch(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(case.block_tables, device=DEV),
                        case.prefix_lens, case.chunk_lens, case.scale, d_err=err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    return out


@pytest.mark.parametrize("P,C,G,Hkv,bs,dtype", BATCHES)
def test_prefill_batch_matches_oracle_and_single_calls(P, C, G, Hkv, bs, dtype):
    case = wl.make_prefill_batch_case(f"pfb{len(P)}", P, C, G * Hkv, Hkv, 128, bs, dtype, seed=sum(P) + sum(C))
    t = case.materialize(DEV)
    refs = _oracle_batch(case, t)
    split = _gpu_batch(case, t, split=True)
    for row, ref in refs:
        check_attention(to_f64(split[row:row + ref.shape[0]]), ref, dtype, f"{case.name} stream-K row {row}")
    out = _gpu_batch(case, t)
    for row, ref in refs:
        check_attention(to_f64(out[row:row + ref.shape[0]]), ref, dtype, f"{case.name} row {row}")
    # without a workspace each sequence's rows equal a pa_prefill_chunk call
    # on that sequence alone (also without one), bit for bit
    row = 0
    for i, (p_, c_) in enumerate(zip(case.prefix_lens.tolist(), case.chunk_lens.tolist())):
        if c_:
            one = torch.full_like(out[row:row + c_], float("nan"))
            pa.pa_prefill_chunk(one, t["query"][row:row + c_].contiguous(), t["k_cache"], t["v_cache"],
                                torch.as_tensor(case.block_tables[i], device=DEV), p_, case.scale)
            torch.cuda.synchronize()
            assert torch.equal(one, out[row:row + c_])
        row += c_


def test_prefill_batch_beyond_one_launch():
    # 70 sequences: two launches of the per-launch sequence table
    rng = np.random.default_rng(4)
    P = [int(x) for x in rng.integers(0, 300, size=70)]
    C = [int(x) for x in rng.integers(1, 40, size=70)]
    case = wl.make_prefill_batch_case("pfb70", P, C, 8, 2, 128, 16, "bf16", seed=70)
    t = case.materialize(DEV)
    refs = _oracle_batch(case, t)
    for split in (False, True):
        out = _gpu_batch(case, t, split=split)
        for row, ref in refs:
            check_attention(to_f64(out[row:row + ref.shape[0]]), ref, "bf16", f"row {row} split {split}")


def test_prefill_batch_full_size_sampled_rows():
    case = wl.prefill_batch_case()
    t = case.materialize(DEV)
    out = _gpu_batch(case, t, split=True)
    assert torch.isfinite(out.float()).all()
    # sampled rows of two sequences against the oracle (a row is a decode at P+r+1)
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    nk, nv = wl.bits(t["new_key"]), wl.bits(t["new_value"])
    assert oracle.reshape_and_cache(nk, nv, kc, vc, case.slot_mapping, case.block_size) == 0
    q = wl.bits(t["query"])
    starts = np.concatenate([[0], np.cumsum(case.chunk_lens)])
    for i in (0, 3):
        P, C = int(case.prefix_lens[i]), int(case.chunk_lens[i])
        for r in (0, C // 2, C - 1):
            row = int(starts[i]) + r
            L = P + r + 1
            n = wl.blocks_for(L, case.block_size)
            ref = oracle.decode(q[row:row + 1], kc, vc, case.block_tables[i:i + 1, :n],
                                np.array([L], np.int32), case.scale, case.dtype, num_threads=8)
            check_attention(to_f64(out[row:row + 1]), ref, case.dtype, f"seq {i} row {r}")


@pytest.mark.parametrize("G,dtype", [(8, "bf16"), (2, "f16")])
def test_prefill_scores_growing_along_the_keys_rescale_the_accumulator(G, dtype):
    # K rows carry a ramp along one direction u (in the pool for the prefix,
    # in the chunk's new keys for its own positions) and each query points
    # along +u or -u: half the heads' scores climb by ~16 (log2 units) per
    # 128 keys, so every key tile raises each such row's running maximum past
    # the rescale threshold; the other half fall
    P, C, Hkv, bs, D = 700, 150, 2, 16, 128
    case = wl.make_prefill_case(f"pfgrow{G}", P, C, G * Hkv, Hkv, D, bs, dtype, seed=40 + G)
    t = case.materialize(DEV)
    g = torch.Generator(device=DEV).manual_seed(6)
    u = torch.randn(D, generator=g, device=DEV)
    u = u / u.norm()
    step = 16.0 / 128 / case.scale / np.log2(np.e) / 8.0  # raw q.k growth per key, for a query 8u
    nbp = wl.blocks_for(P, bs)
    blk = torch.as_tensor(case.block_table[:nbp].astype(np.int64), device=DEV)
    ramp = torch.as_tensor(step * np.arange(nbp * bs).reshape(nbp, bs), dtype=torch.float32, device=DEV)
    kc = t["k_cache"].float()
    kc[blk] += ramp[:, None, :, None] * u
    t["k_cache"].copy_(kc.to(t["k_cache"].dtype))
    nk = t["new_key"].float() + (step * (P + torch.arange(C, device=DEV)))[:, None, None] * u
    t["new_key"].copy_(nk.to(t["new_key"].dtype))
    sign = torch.tensor([1.0 if h % 2 == 0 else -1.0 for h in range(G * Hkv)], device=DEV)
    q = 8.0 * sign[None, :, None] * u + 0.1 * t["query"].float()
    t["query"].copy_(q.to(t["query"].dtype))
    kc0, vc0 = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc0, vc0,
                                    case.slot_mapping, bs) == 0
    ref = oracle.prefill_chunk(wl.bits(t["query"]), kc0, vc0, case.block_table, P, case.scale, dtype,
                               num_threads=8)
    out = run_prefill(case, t)
    check_attention(to_f64(out), ref, dtype, case.name)


def _random_prefill_configs(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.choice([0, int(rng.integers(1, 1500))]))
        C = int(rng.integers(1, 300))
        G = int(rng.choice([1, 2, 4, 8]))
        Hkv = int(rng.integers(1, 4))
        bs = int(rng.choice([16, 32, 64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        out.append((i, P, C, G, Hkv, bs, dtype))
    return out


@pytest.mark.parametrize("i,P,C,G,Hkv,bs,dtype", _random_prefill_configs(12, 2027))
def test_prefill_random_shapes(i, P, C, G, Hkv, bs, dtype):
    case = wl.make_prefill_case(f"pfrand{i}", P, C, G * Hkv, Hkv, 128, bs, dtype, seed=300 + i)
    t = case.materialize(DEV)
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc,
                                    case.slot_mapping, bs) == 0
    ref = oracle.prefill_chunk(wl.bits(t["query"]), kc, vc, case.block_table, P, case.scale, dtype, num_threads=8)
    out = run_prefill(case, t, split=i % 2 == 0)
    check_attention(to_f64(out), ref, dtype, case.name)
