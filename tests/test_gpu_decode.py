"""GPU parity of the paged decode path against the CPU oracle, through the C ABI.

Small and medium shapes that span several tiles, several partitions and a
ragged tail, plus the edge cases: empty and one-token contexts, lengths at
block boundaries, NaN garbage outside the context, invalid table entries and
lengths (flagged, never a fault), and the pages' invariants on the GPU
(physical placement, shared prefixes, copy-on-write).
"""
import numpy as np
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


def gpu_step(case, t, partition_tokens=0, check_err=True):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if case.cow_pairs.shape[0]:
        pa.pa_copy_blocks(t["k_cache"], t["v_cache"], torch.as_tensor(case.cow_pairs, device=DEV), d_err=err)
    if case.num_new_tokens:
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"],
                                torch.as_tensor(case.slot_mapping, device=DEV), d_err=err)
    out = torch.full_like(t["query"], float("nan"))
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(case.block_tables, device=DEV),
                 torch.as_tensor(case.context_lens, device=DEV), case.scale, case.max_context_len,
                 partition_tokens=partition_tokens, d_err=err)
    torch.cuda.synchronize()
    if check_err:
        assert int(err.item()) == 0, f"device error flags {int(err.item()):#x}"
    return out, int(err.item())


def parity(case, partition_tokens=0, pool_fill=None):
    t = case.materialize(DEV, pool_fill=pool_fill)
    seqs = list(range(case.num_seqs))
    inp = oracle_inputs(case, t, seqs)
    import oracle
    ref = oracle_step(oracle, case, inp)
    out, _ = gpu_step(case, t, partition_tokens)
    return check_attention(to_f64(out), ref, case.dtype, case.name), out, t


def test_tiny_workload_step_bit_exact_cache_and_decode():
    import oracle
    c = wl.tiny_case()
    t = c.materialize(DEV)
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    out, _ = gpu_step(c, t, partition_tokens=0)
    assert oracle.reshape_and_cache(wl.bits(t["new_key"]), wl.bits(t["new_value"]), kc, vc,
                                    c.slot_mapping, c.block_size) == 0
    assert np.array_equal(kc, wl.bits(t["k_cache"]))
    assert np.array_equal(vc, wl.bits(t["v_cache"]))
    ref = oracle.decode(wl.bits(t["query"]), kc, vc, c.block_tables, c.context_lens, c.scale, c.dtype)
    check_attention(to_f64(out), ref, c.dtype, "tiny")
    # the same step split into 16- and 32-token partitions
    for pt in (16, 32):
        t2 = c.materialize(DEV)
        out2, _ = gpu_step(c, t2, partition_tokens=pt)
        check_attention(to_f64(out2), ref, c.dtype, f"tiny pt={pt}")


SHAPES = [
    # (D, bs, G, Hkv, dtype)
    (128, 16, 4, 2, "bf16"),
    (128, 16, 1, 3, "f16"),
    (128, 16, 8, 1, "bf16"),
    (128, 16, 2, 2, "f16"),
    (128, 32, 4, 2, "bf16"),
    (128, 32, 8, 1, "f16"),
    (128, 8, 4, 2, "bf16"),
    (64, 16, 1, 4, "f16"),
    (64, 16, 4, 2, "bf16"),
    (64, 32, 2, 2, "f16"),
    (64, 8, 8, 1, "bf16"),
    (128, 64, 4, 2, "bf16"),
    (128, 128, 8, 1, "f16"),
    (64, 64, 2, 2, "f16"),
    (64, 128, 1, 2, "bf16"),
]


@pytest.mark.parametrize("D,bs,G,Hkv,dtype", SHAPES)
def test_decode_shapes_ragged_lengths(D, bs, G, Hkv, dtype):
    lens = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 511, 512, 513, 700, 1500, 2 * bs]
    c = wl.make_decode_case(f"d{D}_bs{bs}_g{G}", lens, G * Hkv, Hkv, D, bs, dtype, seed=D + bs + G)
    parity(c)


@pytest.mark.parametrize("pt", [0, 16, 64, 256, 4096])
def test_partition_size_invariance(pt):
    lens = [1, 17, 300, 1023, 1024, 1025, 2500, 3000]
    c = wl.make_decode_case("pt", lens, 8, 2, 128, 16, "bf16", seed=77)
    parity(c, partition_tokens=pt)


def test_single_token_context_is_bit_exact():
    c = wl.make_decode_case("one", [1] * 6, 8, 2, 128, 16, "bf16", seed=3)
    t = c.materialize(DEV)
    out, _ = gpu_step(c, t)
    # the only row is the token just written: out == new value row, bit for bit
    nv = t["new_value"]
    for s in range(c.num_seqs):
        for h in range(8):
            assert torch.equal(out[s, h], nv[s, h // 4])


def test_zero_length_and_nan_garbage_outside_context():
    lens = [0, 5, 16, 33, 0, 700]
    c = wl.make_decode_case("nan", lens, 4, 1, 128, 16, "f16", seed=4)
    stats, out, _ = parity(c, pool_fill=float("nan"))
    assert (out[0] == 0).all() and (out[4] == 0).all()


def test_physical_permutation_gives_identical_bits():
    c = wl.make_decode_case("perm", [40, 500, 1300, 7], 8, 2, 128, 16, "bf16", seed=5, num_blocks=140)
    t = c.materialize(DEV)
    out_a, _ = gpu_step(c, {k: v.clone() for k, v in t.items()})
    pi = torch.as_tensor(np.random.default_rng(2).permutation(c.num_blocks), device=DEV)
    t2 = {k: v.clone() for k, v in t.items()}
    t2["k_cache"] = torch.empty_like(t["k_cache"])
    t2["v_cache"] = torch.empty_like(t["v_cache"])
    t2["k_cache"][pi] = t["k_cache"]
    t2["v_cache"][pi] = t["v_cache"]
    pin = pi.cpu().numpy()
    c2 = wl.make_decode_case("perm2", c.context_lens, 8, 2, 128, 16, "bf16", seed=5, num_blocks=140,
                             tables=np.where(c.block_tables >= 0, pin[np.maximum(c.block_tables, 0)], -1))
    out_b, _ = gpu_step(c2, t2)
    assert torch.equal(out_a, out_b)


def test_shared_prefix_equals_private_copies_on_gpu():
    c = wl.make_shared_prefix_case("sp", num_prompts=3, samples=4, prefix_len=200, max_tail=300,
                                   num_heads=4, head_dim=128, block_size=16, dtype="f16", seed=8)
    t = c.materialize(DEV)
    out_shared, _ = gpu_step(c, {k: v.clone() for k, v in t.items()})
    # private pool: every table entry of every sequence gets its own block,
    # built from the same pre-step pool; copy-on-write then acts on copies
    rows, bt2 = [], np.full_like(c.block_tables, -1)
    for s in range(c.num_seqs):
        for j in range(wl.blocks_for(c.context_lens[s], 16)):
            bt2[s, j] = len(rows)
            rows.append(int(c.block_tables[s, j]))
    dst_of = {int(b): int(a) for a, b in c.cow_pairs}
    src_rows = [dst_of.get(r, r) for r in rows]  # a COW destination starts as its source's content
    idx = torch.as_tensor(src_rows, device=DEV)
    t2 = dict(t)
    t2["k_cache"] = t["k_cache"].index_select(0, idx).contiguous()
    t2["v_cache"] = t["v_cache"].index_select(0, idx).contiguous()
    slots = []
    for s, pos in zip(c.new_token_seq, c.new_token_pos):
        slots.append(int(bt2[s, pos // 16]) * 16 + int(pos) % 16)
    c2 = wl.DecodeCase(**{**c.__dict__, "num_blocks": len(rows), "block_tables": bt2,
                          "slot_mapping": np.array(slots, np.int64),
                          "cow_pairs": np.zeros((0, 2), np.int64), "tensors": {}})
    out_private, _ = gpu_step(c2, t2)
    assert torch.equal(out_shared, out_private)


def test_copy_blocks_bit_exact_and_conflicts_flagged():
    import oracle
    NB, Hkv, bs, D = 12, 3, 16, 128
    g = torch.Generator(device=DEV).manual_seed(1)
    kc = torch.randn((NB, Hkv, bs, D), generator=g, device=DEV, dtype=torch.float16)
    vc = torch.randn((NB, Hkv, bs, D), generator=g, device=DEV, dtype=torch.float16)
    k0, v0 = wl.bits(kc), wl.bits(vc)
    pairs = np.array([[0, 1], [2, 2], [3, 4], [5, 4], [6, 0], [7, 99], [8, 9], [10, 11]], np.int64)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_copy_blocks(kc, vc, torch.as_tensor(pairs, device=DEV), d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.capi.DEVERR["copy_pair"]
    assert oracle.copy_blocks(k0, v0, pairs) == 5
    assert np.array_equal(k0, wl.bits(kc)) and np.array_equal(v0, wl.bits(vc))


def test_copy_blocks_many_pairs_with_planted_conflicts():
    # 4096 pairs over a 10000-block pool: most valid, with planted duplicate
    # dsts, dsts that are other pairs' srcs, src == dst and ids outside the pool
    import oracle
    NB, Hkv, bs, D = 10000, 4, 16, 128
    rng = np.random.default_rng(4096)
    perm = rng.permutation(NB)
    n = 4096
    pairs = np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int64)
    k = 64
    pairs[rng.choice(n, k, replace=False), 1] = pairs[rng.choice(n, k, replace=False), 1]   # duplicate dsts
    idx = rng.choice(n, k, replace=False)
    pairs[idx, 1] = pairs[rng.choice(n, k, replace=False), 0]                                 # dst = some src
    idx = rng.choice(n, 16, replace=False)
    pairs[idx, 1] = pairs[idx, 0]                                                              # src == dst
    pairs[rng.choice(n, 8, replace=False), 0] = NB + 5                                         # src outside
    pairs[rng.choice(n, 8, replace=False), 1] = -3                                             # dst outside
    g = torch.Generator(device=DEV).manual_seed(2)
    kc = torch.randn((NB, Hkv, bs, D), generator=g, device=DEV, dtype=torch.float16)
    vc = torch.randn((NB, Hkv, bs, D), generator=g, device=DEV, dtype=torch.float16)
    k0, v0 = wl.bits(kc), wl.bits(vc)
    bad = oracle.copy_blocks(k0, v0, pairs)
    assert 100 < bad < n // 4
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(pa.pa_copy_blocks_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    ws.fill_(0xAB)  # the workspace's content on entry must not matter
    pa.pa_copy_blocks(kc, vc, torch.as_tensor(pairs, device=DEV), d_err=err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.capi.DEVERR["copy_pair"]
    assert np.array_equal(k0, wl.bits(kc)) and np.array_equal(v0, wl.bits(vc))
    # the same call again (the table is rebuilt, the copies are idempotent)
    pa.pa_copy_blocks(kc, vc, torch.as_tensor(pairs, device=DEV), d_err=err, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(k0, wl.bits(kc)) and np.array_equal(v0, wl.bits(vc))


def test_copy_on_write_isolates_the_writer_on_gpu():
    c = wl.make_shared_prefix_case("cow", num_prompts=1, samples=4, prefix_len=40, max_tail=0,
                                   num_heads=8, head_dim=128, block_size=16, dtype="bf16", seed=12)
    t = c.materialize(DEV)
    before, _ = gpu_step(c, t)
    # sample 0 appends one token into its private copy of the partial block
    lens = c.context_lens.copy()
    lens[0] += 1
    slot = torch.tensor([int(c.block_tables[0, 2]) * 16 + 8], device=DEV)
    nk = torch.randn((1, 8, 128), device=DEV, dtype=torch.bfloat16)
    pa.pa_reshape_and_cache(nk, nk, t["k_cache"], t["v_cache"], slot)
    out = torch.empty_like(t["query"])
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(c.block_tables, device=DEV),
                 torch.as_tensor(lens, device=DEV), c.scale, int(lens.max()))
    torch.cuda.synchronize()
    assert torch.equal(before[1:], out[1:])
    assert not torch.equal(before[0], out[0])


def test_bad_table_entries_and_lengths_are_flagged_not_faulted():
    c = wl.make_decode_case("bad", [40, 40, 40], 4, 1, 128, 16, "f16", seed=6)
    t = c.materialize(DEV)
    bt = c.block_tables.copy()
    bt[1, 1] = c.num_blocks + 1000       # outside the pool
    bt[2, 0] = -7
    lens = c.context_lens.copy()
    out = torch.empty_like(t["query"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(bt, device=DEV),
                 torch.as_tensor(lens, device=DEV), c.scale, c.max_context_len, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.capi.DEVERR["block_range"]
    assert torch.isfinite(out[0].float()).all()
    # a length past max_context_len is clamped and flagged
    lens2 = np.array([40, 40, 400], np.int32)
    err.zero_()
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(c.block_tables, device=DEV),
                 torch.as_tensor(lens2, device=DEV), c.scale, 40, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.capi.DEVERR["context_range"]
    # slot outside the pool in a cache write
    err.zero_()
    slot = torch.tensor([c.num_blocks * 16 + 3], device=DEV)
    pa.pa_reshape_and_cache(t["new_key"][:1], t["new_value"][:1], t["k_cache"], t["v_cache"], slot, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.capi.DEVERR["slot_range"]
    # the context is still usable
    out2, _ = gpu_step(c, c.materialize(DEV))
    assert torch.isfinite(out2.float()).all()


# Head groups of 8 at head_dim 128 run on the tensor cores (128-key tiles,
# one 4-D copy per block): the same edge cases again for that kernel, and for
# groups of 4 (CUDA cores) at every block size.
TC_SHAPES = [(8, 8, 2, "bf16"), (8, 16, 2, "f16"), (8, 32, 1, "bf16"), (8, 64, 2, "f16"), (8, 128, 1, "bf16"),
             (4, 8, 2, "f16"), (4, 16, 3, "f16"), (4, 32, 2, "f16"), (4, 64, 1, "bf16"), (4, 128, 2, "f16")]


@pytest.mark.parametrize("G,bs,Hkv,dtype", TC_SHAPES)
def test_tensor_core_decode_shapes(G, bs, Hkv, dtype):
    lens = [1, 127, 128, 129, 255, 256, 257, bs + 1, 3 * bs + 5, 1000, 2049]
    c = wl.make_decode_case(f"tc_g{G}_bs{bs}", lens, G * Hkv, Hkv, 128, bs, dtype, seed=100 + bs + G)
    parity(c)


@pytest.mark.parametrize("pt", [0, 16, 48, 128, 512, 4096])
def test_group8_partition_size_invariance(pt):
    # partitions shorter than, equal to and longer than a 128-key tile
    lens = [1, 17, 300, 1023, 1024, 1025, 2500, 3000]
    c = wl.make_decode_case("tc_pt", lens, 16, 2, 128, 16, "bf16", seed=78)
    parity(c, partition_tokens=pt)


def test_group8_single_token_context_is_bit_exact():
    c = wl.make_decode_case("tc_one", [1] * 5, 16, 2, 128, 16, "f16", seed=9)
    t = c.materialize(DEV)
    out, _ = gpu_step(c, t)
    nv = t["new_value"]
    for s in range(c.num_seqs):
        for h in range(16):
            assert torch.equal(out[s, h], nv[s, h // 8])


def test_group8_zero_length_and_nan_garbage_outside_context():
    lens = [0, 5, 128, 129, 0, 700, 16]
    c = wl.make_decode_case("tc_nan", lens, 8, 1, 128, 16, "bf16", seed=10)
    stats, out, _ = parity(c, pool_fill=float("nan"))
    assert (out[0] == 0).all() and (out[4] == 0).all()


def test_group8_physical_permutation_gives_identical_bits():
    c = wl.make_decode_case("tc_perm", [40, 500, 1300, 7], 16, 2, 128, 16, "bf16", seed=11, num_blocks=140)
    t = c.materialize(DEV)
    out_a, _ = gpu_step(c, {k: v.clone() for k, v in t.items()})
    pi = torch.as_tensor(np.random.default_rng(3).permutation(c.num_blocks), device=DEV)
    t2 = {k: v.clone() for k, v in t.items()}
    t2["k_cache"] = torch.empty_like(t["k_cache"])
    t2["v_cache"] = torch.empty_like(t["v_cache"])
    t2["k_cache"][pi] = t["k_cache"]
    t2["v_cache"][pi] = t["v_cache"]
    pin = pi.cpu().numpy()
    c2 = wl.make_decode_case("tc_perm2", c.context_lens, 16, 2, 128, 16, "bf16", seed=11, num_blocks=140,
                             tables=np.where(c.block_tables >= 0, pin[np.maximum(c.block_tables, 0)], -1))
    out_b, _ = gpu_step(c2, t2)
    assert torch.equal(out_a, out_b)


def test_group8_bad_table_entries_are_flagged_and_their_keys_left_out():
    import oracle
    c = wl.make_decode_case("tc_bad", [300, 300, 300], 8, 1, 128, 16, "bf16", seed=12)
    t = c.materialize(DEV)
    bt = c.block_tables.copy()
    bt[1, 3] = c.num_blocks + 1000       # outside the pool
    bt[2, 0] = -7
    out = torch.empty_like(t["query"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], torch.as_tensor(bt, device=DEV),
                 torch.as_tensor(c.context_lens, device=DEV), c.scale, c.max_context_len, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.capi.DEVERR["block_range"]
    # leaving a block's 16 keys out equals attention over the table without
    # that block and 16 fewer tokens (300 = 18*16 + 12, 284 = 17*16 + 12, so
    # the partial last block lines up)
    nb = wl.blocks_for(300, 16)
    tables = np.stack([c.block_tables[0, :nb],
                       np.concatenate([c.block_tables[1, :3], c.block_tables[1, 4:nb], [-1]]),
                       np.concatenate([c.block_tables[2, 1:nb], [-1]])]).astype(np.int32)
    lens = np.array([300, 284, 284], np.int32)
    ref = oracle.decode(wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"]), tables, lens,
                        c.scale, c.dtype, num_threads=8)
    check_attention(to_f64(out), ref, c.dtype, c.name)
    out2, _ = gpu_step(c, c.materialize(DEV))
    assert torch.isfinite(out2.float()).all()


@pytest.mark.parametrize("G,dtype,pt", [(1, "bf16", 0), (4, "bf16", 0), (4, "f16", 4096), (8, "bf16", 0),
                                         (8, "f16", 4096)])
def test_scores_growing_along_the_context_rescale_the_accumulator(G, dtype, pt):
    # K rows carry a ramp along one direction u and each query points along
    # +u or -u, so the scores of half the heads climb by ~16 (log2 units) per
    # 128 keys -- every tile raises the running maximum past the rescale
    # threshold -- and the other half fall (the maximum stays on the first tile)
    Hkv, bs, D = 2, 16, 128
    lens = [3000, 1500, 700, 129, 1]
    c = wl.make_decode_case(f"grow_g{G}", lens, G * Hkv, Hkv, D, bs, dtype, seed=300 + G)
    t = c.materialize(DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    u = torch.randn(D, generator=g, device=DEV)
    u = u / u.norm()
    blks, ramps = [], []
    for s, L in enumerate(c.context_lens):
        for bi in range(wl.blocks_for(int(L), bs)):
            blks.append(int(c.block_tables[s, bi]))
            ramps.append(16.0 / 128 * (bi * bs + np.arange(bs)) / c.scale / np.log2(np.e) / 8.0)
    blk = torch.as_tensor(blks, device=DEV)
    ramp = torch.as_tensor(np.stack(ramps), dtype=torch.float32, device=DEV)
    kc = t["k_cache"].float()
    kc[blk] += ramp[:, None, :, None] * u
    t["k_cache"].copy_(kc.to(t["k_cache"].dtype))
    sign = torch.tensor([1.0 if h % 2 == 0 else -1.0 for h in range(G * Hkv)], device=DEV)
    q = 8.0 * sign[None, :, None] * u + 0.1 * t["query"].float()
    t["query"].copy_(q.to(t["query"].dtype))
    import oracle
    ref = oracle_step(oracle, c, oracle_inputs(c, t, range(c.num_seqs)))
    out, _ = gpu_step(c, t, partition_tokens=pt)
    check_attention(to_f64(out), ref, dtype, c.name)


def test_host_argument_errors_launch_nothing():
    c = wl.make_decode_case("args", [10], 4, 2, 128, 16, "bf16", seed=1)
    t = c.materialize(DEV)
    out = torch.empty_like(t["query"])
    bt = torch.as_tensor(c.block_tables, device=DEV)
    lens = torch.as_tensor(c.context_lens, device=DEV)
    with pytest.raises(pa.PAError):  # partition not a multiple of block_size
        pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], bt, lens, c.scale, 10, partition_tokens=20)
    with pytest.raises(pa.PAError):  # workspace too small for a split
        pa.pa_decode(out, t["query"], t["k_cache"], t["v_cache"], bt, lens, c.scale, 5000,
                     partition_tokens=16, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("G", [1, 4, 8])
def test_decode_step_replays_from_a_cuda_graph(G):
    # the step an engine captures once and replays every token: cache write,
    # decode (programmatic dependent launches), split-K reduce
    c = wl.make_decode_case(f"graph_g{G}", [1, 300, 2049, 700, 0], 2 * G, 2, 128, 16, "bf16", seed=70 + G)
    t = c.materialize(DEV)
    slots = torch.as_tensor(c.slot_mapping, device=DEV)
    bt = torch.as_tensor(c.block_tables, device=DEV)
    lens = torch.as_tensor(c.context_lens, device=DEV)
    ws = pa.decode_workspace(t["query"], 2, 16, c.max_context_len, 256)
    out = torch.empty_like(t["query"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step(o):
        pa.pa_reshape_and_cache(t["new_key"], t["new_value"], t["k_cache"], t["v_cache"], slots, d_err=err)
        pa.pa_decode(o, t["query"], t["k_cache"], t["v_cache"], bt, lens, c.scale, c.max_context_len,
                     partition_tokens=256, workspace=ws, d_err=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(out)  # eager warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(out)
    g = torch.Generator(device=DEV).manual_seed(9)
    for i in range(3):
        if i:
            t["query"].copy_(torch.randn(t["query"].shape, generator=g, device=DEV).to(t["query"].dtype))
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        eager = torch.empty_like(out)
        step(eager)
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
        if i == 0:
            assert torch.equal(out, ref)
    assert int(err.item()) == 0


@pytest.mark.parametrize("G,dtype", [(1, "f16"), (8, "bf16")])
def test_hundreds_of_partitions_merge_in_the_reduce(G, dtype):
    # one long sequence in 128-token partitions: the log-sum-exp reduce merges
    # hundreds of partials per head (more than a warp has lanes), beside
    # short sequences that fit one partition and write their output directly
    c = wl.make_decode_case(f"many_parts_g{G}", [60000, 5, 129, 3000], 2 * G, 2, 128, 16, dtype, seed=140 + G)
    parity(c, partition_tokens=128)


@pytest.mark.parametrize("G,Hkv", [(4, 8), (8, 16)])
def test_large_batch_of_short_sequences(G, Hkv):
    # 4096 sequences: tens of thousands of CTAs (units = sequences x kv heads),
    # every sequence against the oracle
    lens = np.random.default_rng(7).integers(1, 65, size=4096)
    c = wl.make_decode_case(f"big_batch_g{G}", lens, G * Hkv, Hkv, 128, 16, "bf16", seed=150 + G)
    parity(c)


def _random_configs(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 4, 8]))
        Hkv = int(rng.integers(1, 5))
        bs = int(rng.choice([8, 16, 32, 64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        B = int(rng.integers(1, 24))
        lens = [int(x) for x in rng.integers(0, 3000, size=B)]
        lens[int(rng.integers(0, B))] = int(rng.integers(1, 4))          # always one very short context
        pt = int(rng.choice([0, bs, 4 * bs, 128 * ((bs + 127) // 128), 1024]))
        out.append((i, D, G, Hkv, bs, dtype, lens, pt))
    return out


@pytest.mark.parametrize("i,D,G,Hkv,bs,dtype,lens,pt", _random_configs(24, 2026))
def test_random_shapes_lengths_and_partitions(i, D, G, Hkv, bs, dtype, lens, pt):
    # seeded random configurations over every supported head_dim, group,
    # block size, dtype and partition length, ragged lengths including empty
    # contexts: both decode kernels against the oracle
    c = wl.make_decode_case(f"rand{i}", lens, G * Hkv, Hkv, D, bs, dtype, seed=200 + i)
    parity(c, partition_tokens=pt)
