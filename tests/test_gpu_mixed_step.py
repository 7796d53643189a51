"""One continuous-batching step (pa_mixed_step): prompt chunks and decodes
over one pool, together.

The pages' chunked prefill batches prompt chunks with the decodes of other
sequences (page "vLLM PagedAttention chuyen sau", section "Chunked
Prefill").  With 8 query heads per kv head the step is one launch (prefill
CTAs and persistent decode CTAs in one grid): both halves must match the
oracle, two steps in a row must give the same bits (the workspace is reused),
and garbage past the contexts must not leak in.  Otherwise (other groups, or
a workspace sized only for pa_decode) the step is two concurrent launches and
must give, bit for bit, what the two calls give one after the other.
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


def write_step_kv(case, t, err, slots=None):
    if slots is None:
        slots = torch.as_tensor(case.slot_mapping, device=DEV)
    pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)


def device_args(case):
    return (torch.as_tensor(case.prefill_tables, device=DEV), torch.as_tensor(case.decode_tables, device=DEV),
            torch.as_tensor(case.context_lens, device=DEV))


def mixed(case, t, err, pt=0, workspace=None):
    pbt, dbt, lens = device_args(case)
    pout = torch.full_like(t["prefill_query"], float("nan"))
    dout = torch.full_like(t["decode_query"], float("nan"))
    pa.pa_mixed_step(pout, t["prefill_query"], pbt, case.prefix_lens, case.chunk_lens, dout, t["decode_query"], dbt,
                     lens, t["k_cache"], t["v_cache"], case.scale, case.max_context_len, partition_tokens=pt,
                     workspace=workspace, d_err=err)
    return pout, dout


def two_launch_workspace(case, t, pt=0):
    # sized for pa_decode only: the step runs as two concurrent launches
    return pa.decode_workspace(t["decode_query"], case.num_kv_heads, case.block_size, case.max_context_len, pt)


def check_both_halves(c, t, pm, dm, what):
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    ref_d = oracle.decode(wl.bits(t["decode_query"]), kc, vc, c.decode_tables, c.context_lens, c.scale, c.dtype,
                          num_threads=os.cpu_count() or 8)
    check_attention(to_f64(dm), ref_d, c.dtype, f"{what}: decode half")
    q = wl.bits(t["prefill_query"])
    row = 0
    for i, (P, C) in enumerate(zip(c.prefix_lens.tolist(), c.chunk_lens.tolist())):
        if C:
            ref_p = oracle.prefill_chunk(q[row:row + C], kc, vc, c.prefill_tables[i], P, c.scale, c.dtype,
                                         num_threads=os.cpu_count() or 8)
            check_attention(to_f64(pm[row:row + C]), ref_p, c.dtype, f"{what}: prefill seq {i}")
        row += C


def separate(case, t, err, pt=0):
    pbt, dbt, lens = device_args(case)
    pout = torch.full_like(t["prefill_query"], float("nan"))
    dout = torch.full_like(t["decode_query"], float("nan"))
    pa.pa_prefill_batch(pout, t["prefill_query"], t["k_cache"], t["v_cache"], pbt, case.prefix_lens,
                        case.chunk_lens, case.scale, d_err=err)
    pa.pa_decode(dout, t["decode_query"], t["k_cache"], t["v_cache"], dbt, lens, case.scale, case.max_context_len,
                 partition_tokens=pt, d_err=err)
    return pout, dout


@pytest.mark.parametrize("G,dtype", [(4, "bf16"), (8, "f16"), (1, "bf16")])
def test_mixed_step_equals_the_two_calls_and_the_oracle(G, dtype):
    # two concurrent launches (a workspace sized for pa_decode only)
    c = wl.make_mixed_case(f"mixed_g{G}", [1, 300, 2049, 0, 700, 129], [40, 0, 333], [9, 17, 130], 2 * G, 2, 128,
                           16, dtype, seed=80 + G)
    t = c.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    pm, dm = mixed(c, t, err, pt=256, workspace=two_launch_workspace(c, t, 256))
    ps, ds = separate(c, t, err, pt=256)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(pm, ps) and torch.equal(dm, ds)
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    ref_d = oracle.decode(wl.bits(t["decode_query"]), kc, vc, c.decode_tables, c.context_lens, c.scale, dtype,
                          num_threads=8)
    check_attention(to_f64(dm), ref_d, dtype, "decode half")
    q = wl.bits(t["prefill_query"])
    row = 0
    for i, (P, C) in enumerate(zip(c.prefix_lens.tolist(), c.chunk_lens.tolist())):
        ref_p = oracle.prefill_chunk(q[row:row + C], kc, vc, c.prefill_tables[i], P, c.scale, dtype, num_threads=8)
        check_attention(to_f64(pm[row:row + C]), ref_p, dtype, f"prefill seq {i}")
        row += C


@pytest.mark.parametrize("prefix,chunks,lens,bs,dtype", [
    ([40, 0, 333], [9, 17, 130], [1, 300, 2049, 0, 700, 129], 16, "f16"),
    ([1000, 5], [64, 700], [5000, 1, 17, 2048, 128, 4097], 32, "bf16"),
    ([0], [1], [3], 16, "bf16"),
    ([8192], [512], [int(x) for x in np.random.default_rng(3).integers(1, 4097, size=40)], 16, "bf16"),
    ([130, 0, 4000], [200, 9, 64], [64, 1, 4096, 1000, 0, 63], 64, "f16"),
    ([2048], [333], [1, 127, 128, 129, 5000, 16384], 128, "bf16"),
    ([0, 5], [1, 1], [int(x) for x in np.random.default_rng(4).integers(0, 600, size=700)], 16, "bf16"),
])
def test_mixed_step_one_launch_matches_the_oracle(prefix, chunks, lens, bs, dtype):
    # one launch (8 query heads per kv head, a mixed-step workspace): every
    # output of both halves against the oracle; two steps in a row give the
    # same bits with the same workspace; NaN past every context stays out
    c = wl.make_mixed_case("mixed1", lens, prefix, chunks, 16, 2, 128, bs, dtype, seed=sum(lens) % 1000)
    t = c.materialize(DEV, pool_fill=float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    ws = pa.mixed_workspace(t["prefill_query"], t["decode_query"], c.num_kv_heads, bs, len(chunks), c.max_context_len)
    pm, dm = mixed(c, t, err, workspace=ws)
    pm2, dm2 = mixed(c, t, err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    assert torch.equal(pm, pm2) and torch.equal(dm, dm2)
    check_both_halves(c, t, pm, dm, "one launch")


@pytest.mark.parametrize("G,dtype", [(4, "bf16"), (2, "f16"), (1, "bf16")])
def test_mixed_step_one_launch_smaller_head_groups(G, dtype):
    # 2 or 4 query heads per kv head in one launch (the decode instances leave
    # the rest of the MMA's 16 head rows zero; LLaMA-like 32/8 heads at
    # G = 4); 1 runs as two launches (the CUDA-core decode)
    hkv = 8 if G == 4 else 2
    lens = [int(x) for x in np.random.default_rng(G).integers(1, 3000, size=60)] + [0, 1, 16384]
    c = wl.make_mixed_case(f"mixg{G}", lens, [1500, 0], [300, 77], G * hkv, hkv, 128, 16, dtype, seed=610 + G)
    t = c.materialize(DEV, pool_fill=float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    ws = pa.mixed_workspace(t["prefill_query"], t["decode_query"], hkv, 16, 2, c.max_context_len)
    pm, dm = mixed(c, t, err, workspace=ws)
    pm2, dm2 = mixed(c, t, err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    assert torch.equal(pm, pm2) and torch.equal(dm, dm2)
    check_both_halves(c, t, pm, dm, f"one launch, G={G}")


def test_mixed_step_one_launch_workspace_shared_by_steps_of_other_shapes():
    # the decode queue's counter and the stream-K counters live in the
    # workspace and must be back at zero after every step, whatever its shape:
    # steps A, B, A, B on one workspace give the bits of A and B run alone
    a = wl.make_mixed_case("mixed_a", [int(x) for x in np.random.default_rng(5).integers(0, 3000, size=300)],
                           [700], [200], 16, 2, 128, 16, "bf16", seed=7)
    b = wl.make_mixed_case("mixed_b", [5, 1, 4000], [0, 64], [300, 17], 16, 2, 128, 16, "bf16", seed=8)
    ta, tb = a.materialize(DEV), b.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(a, ta, err)
    write_step_kv(b, tb, err)
    # sized for the larger half of each (B's 317 chunk rows, A's 300 decodes)
    fresh = lambda: pa.mixed_workspace(tb["prefill_query"], ta["decode_query"], 2, 16, 2, 4096)
    ws = fresh()
    pa1, da1 = mixed(a, ta, err, workspace=fresh())
    pb1, db1 = mixed(b, tb, err, workspace=fresh())
    runs = [mixed(c, t, err, workspace=ws) for c, t in ((a, ta), (b, tb), (a, ta), (b, tb))]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for (pm, dm), (pr, dr) in zip(runs, [(pa1, da1), (pb1, db1)] * 2):
        assert torch.equal(pm, pr) and torch.equal(dm, dr)
    check_both_halves(a, ta, pa1, da1, "step A")
    check_both_halves(b, tb, pb1, db1, "step B")


def test_mixed_step_full_size_one_launch_matches_the_oracle_and_two_launches_match_the_calls():
    c = wl.mixed_case()
    t = c.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    pm, dm = mixed(c, t, err)                       # one launch
    p2, d2 = mixed(c, t, err, workspace=two_launch_workspace(c, t))
    ps, ds = separate(c, t, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(p2, ps) and torch.equal(d2, ds)
    check_both_halves(c, t, pm, dm, "full size, one launch")


@pytest.mark.parametrize("one_launch", [False, True])
def test_mixed_step_replays_from_a_cuda_graph(one_launch):
    # two launches: the fork onto the library's stream and the join back must
    # survive capture; one launch: the kernel replays with the same bits
    c = wl.make_mixed_case("mixed_graph", [1, 300, 2049, 700], [100], [64], 8, 2, 128, 16, "bf16", seed=90)
    t = c.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pbt, dbt, lens = device_args(c)
    slots = torch.as_tensor(c.slot_mapping, device=DEV)  # no host copies inside the capture
    ws = (pa.mixed_workspace(t["prefill_query"], t["decode_query"], 2, 16, len(c.chunk_lens), c.max_context_len, 256)
          if one_launch else two_launch_workspace(c, t, 256))
    pout = torch.empty_like(t["prefill_query"])
    dout = torch.empty_like(t["decode_query"])

    def step():
        write_step_kv(c, t, err, slots)
        pa.pa_mixed_step(pout, t["prefill_query"], pbt, c.prefix_lens, c.chunk_lens, dout, t["decode_query"], dbt,
                         lens, t["k_cache"], t["v_cache"], c.scale, c.max_context_len, partition_tokens=256,
                         workspace=ws, d_err=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref_p, ref_d = pout.clone(), dout.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    pout.zero_()
    dout.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(pout, ref_p) and torch.equal(dout, ref_d)
    assert int(err.item()) == 0
    assert not np.isnan(to_f64(pout)).any()


def test_mixed_step_with_one_half_empty_runs_that_half_alone():
    c = wl.make_mixed_case("mixed_one", [1, 300, 700], [50], [20], 16, 2, 128, 16, "bf16", seed=95)
    t = c.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    pbt, dbt, lens = device_args(c)
    ps, ds = separate(c, t, err)
    # decode only: an empty prompt-chunk list
    dout = torch.full_like(t["decode_query"], float("nan"))
    empty_q = t["prefill_query"][:0]
    pa.pa_mixed_step(empty_q.clone(), empty_q, pbt[:0], np.zeros(0, np.int32), np.zeros(0, np.int32), dout,
                     t["decode_query"], dbt, lens, t["k_cache"], t["v_cache"], c.scale, c.max_context_len,
                     d_err=err)
    # prefill only: no decoding sequences
    pout = torch.full_like(t["prefill_query"], float("nan"))
    empty_d = t["decode_query"][:0]
    pa.pa_mixed_step(pout, t["prefill_query"], pbt, c.prefix_lens, c.chunk_lens, empty_d.clone(), empty_d, dbt[:0],
                     lens[:0], t["k_cache"], t["v_cache"], c.scale, 1, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(dout, ds) and torch.equal(pout, ps)


def _random_mixed_configs(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        nd = int(rng.choice([1, 3, 17, 90]))
        lens = [int(x) for x in rng.integers(0, int(rng.choice([64, 1500, 5000])), size=nd)]
        npf = int(rng.integers(1, 4))
        prefix = [int(x) for x in rng.integers(0, 2000, size=npf)]
        chunks = [int(x) for x in rng.integers(0, 400, size=npf)]
        chunks[0] = max(chunks[0], 1)
        hkv = int(rng.integers(1, 4))
        bs = int(rng.choice([16, 32, 64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        G = int(rng.choice([1, 2, 4, 8]))
        out.append((i, lens, prefix, chunks, G, hkv, bs, dtype))
    return out


@pytest.mark.parametrize("i,lens,prefix,chunks,G,hkv,bs,dtype", _random_mixed_configs(12, 4242))
def test_mixed_step_one_launch_random_shapes(i, lens, prefix, chunks, G, hkv, bs, dtype):
    # everything drawn (head groups 2-8 run in one launch, 1 in two): every
    # output of both halves against the oracle
    c = wl.make_mixed_case(f"mixrand{i}", lens, prefix, chunks, G * hkv, hkv, 128, bs, dtype, seed=500 + i)
    t = c.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    ws = pa.mixed_workspace(t["prefill_query"], t["decode_query"], hkv, bs, len(chunks), c.max_context_len)
    pm, dm = mixed(c, t, err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    check_both_halves(c, t, pm, dm, f"random mixed {i}")


def test_mixed_step_one_launch_flags_a_bad_table_entry_and_finishes():
    # one decode sequence's table names a block past the pool: the kernel
    # fetches zeros for it, leaves it out of that sequence's softmax, flags
    # block_range and completes; the prompt chunk and the other decodes are
    # unaffected
    c = wl.make_mixed_case("mixbad", [700, 300, 50], [200], [64], 16, 2, 128, 16, "bf16", seed=77)
    t = c.materialize(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    write_step_kv(c, t, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pbt, dbt, lens = device_args(c)
    dbt[0, 3] = c.num_blocks + 1000
    ws = pa.mixed_workspace(t["prefill_query"], t["decode_query"], 2, 16, 1, c.max_context_len)
    pout = torch.full_like(t["prefill_query"], float("nan"))
    dout = torch.full_like(t["decode_query"], float("nan"))
    pa.pa_mixed_step(pout, t["prefill_query"], pbt, c.prefix_lens, c.chunk_lens, dout, t["decode_query"], dbt,
                     lens, t["k_cache"], t["v_cache"], c.scale, c.max_context_len, workspace=ws, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.capi.DEVERR["block_range"]
    assert not int(err.item()) & pa.capi.DEVERR["timeout"]
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    ref_d = oracle.decode(wl.bits(t["decode_query"]), kc, vc, c.decode_tables, c.context_lens, c.scale, c.dtype,
                          num_threads=8)
    check_attention(to_f64(dout[1:]), ref_d[1:], c.dtype, "decodes with good tables")
    assert np.isfinite(to_f64(dout[0])).all()
    ref_p = oracle.prefill_chunk(wl.bits(t["prefill_query"]), kc, vc, c.prefill_tables[0], int(c.prefix_lens[0]),
                                 c.scale, c.dtype, num_threads=8)
    check_attention(to_f64(pout), ref_p, c.dtype, "prompt chunk")
