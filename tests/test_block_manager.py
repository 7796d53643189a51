"""CPU tests of the native block manager (pa_bm_* in include/pa.h).

What the pages fix ("vLLM PagedAttention chuyen sau", sections "Tuong tu phan
trang bo nho ao", "Co che APC", "Danh gia ty le truy cap APC", FAQ item 5):
  - a sequence of n tokens holds ceil(n/block_size) blocks (the worked
    example: 30 tokens -> 2 blocks, 50 tokens -> 4 at block size 16);
  - growth adds blocks without moving old ones;
  - shared blocks are copied before a diverging write (copy-on-write);
  - a new request's prefix is matched against cached blocks and those
    physical blocks are linked into its table; the hit rate is the share of
    tokens whose blocks were reused;
  - under pressure, least recently used blocks are evicted.
The end-to-end pin: a simulated engine writes each token's K/V (a function of
the whole token prefix, as in a real model) into the slots the manager hands
out, applies its copy pairs, and every live sequence's K/V gathered through
its block table must equal its logical K/V bit for bit; the CPU oracle's
decode over those tables must equal attention over the logical K/V.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl


def test_page_example_block_counts():
    bm = pa.BlockManager(64, 16, prefix_cache=False)
    bm.add_sequence(1, np.arange(30))
    bm.add_sequence(2, np.arange(100, 150))
    assert len(bm.block_table(1)) == 2 == wl.blocks_for(30, 16)
    assert len(bm.block_table(2)) == 4 == wl.blocks_for(50, 16)
    st = bm.stats()
    assert st["used_blocks"] == 6 and st["free_blocks"] == 58
    # blocks are disjoint and every slot lands in the sequence's own table
    assert not set(bm.block_table(1)) & set(bm.block_table(2))


def test_growth_allocates_exactly_at_block_boundaries():
    bm = pa.BlockManager(16, 4, prefix_cache=False)
    slots, cached = bm.add_sequence(7, [1, 2, 3])
    assert cached == 0 and len(bm.block_table(7)) == 1
    first = bm.block_table(7)[0]
    assert list(slots) == [first * 4 + i for i in range(3)]
    seen = list(slots)
    for k in range(3, 13):
        slot, pair = bm.append_token(7, k)
        assert pair is None
        table = bm.block_table(7)
        assert len(table) == wl.blocks_for(k + 1, 4)
        assert slot == table[k // 4] * 4 + k % 4
        assert table[0] == first  # old blocks never move
        seen.append(slot)
    assert len(set(seen)) == len(seen)
    assert bm.seq_len(7) == 13


def test_fork_shares_blocks_and_copy_on_write_isolates_writers():
    bm = pa.BlockManager(32, 16, prefix_cache=False)
    bm.add_sequence(1, np.arange(20))           # block 0 full, block 1 holds 4 tokens
    bm.fork(1, 2)
    bm.fork(1, 3)
    b0, b1 = bm.block_table(1)
    assert bm.refcount(b0) == 3 and bm.refcount(b1) == 3
    # child 2 writes into the shared partial block: copy first
    slot, pair = bm.append_token(2, 99)
    assert pair is not None and pair[0] == b1
    new = pair[1]
    assert bm.block_table(2)[1] == new and slot == new * 16 + 4
    assert bm.refcount(b1) == 2 and bm.refcount(new) == 1
    # child 3 too
    _, pair3 = bm.append_token(3, 98)
    assert pair3 is not None and pair3[0] == b1
    # the parent is now the only holder: it writes in place
    slot1, pair1 = bm.append_token(1, 97)
    assert pair1 is None and slot1 == b1 * 16 + 4
    assert bm.refcount(b0) == 3  # full shared blocks are never copied
    assert bm.stats()["cow_copies"] == 2


def test_free_returns_blocks_and_refcounts():
    bm = pa.BlockManager(8, 4, prefix_cache=False)
    bm.add_sequence(1, np.arange(10))
    bm.fork(1, 2)
    bm.free_sequence(1)
    assert bm.stats()["free_blocks"] == 5  # all still held by 2
    bm.free_sequence(2)
    st = bm.stats()
    assert st["free_blocks"] == 8 and st["used_blocks"] == 0 and st["num_sequences"] == 0
    with pytest.raises(pa.PAError):
        bm.free_sequence(2)


def test_prefix_cache_links_matching_blocks_and_counts_hits():
    bm = pa.BlockManager(64, 4)
    prefix = list(range(12))                    # three full blocks
    s1, c1 = bm.add_sequence(1, prefix + [50, 51])
    assert c1 == 0
    s2, c2 = bm.add_sequence(2, prefix + [60, 61, 62, 63, 64])
    assert c2 == 12 and list(s2[:12]) == [-1] * 12
    t1, t2 = bm.block_table(1), bm.block_table(2)
    assert list(t1[:3]) == list(t2[:3]) and t1[3] != t2[3]
    for b in t1[:3]:
        assert bm.refcount(b) == 2
    st = bm.stats()
    assert st["hit_tokens"] == 12 and st["query_tokens"] == 14 + 17
    assert st["hit_rate"] == pytest.approx(12 / 31)
    # a prompt diverging inside the second block reuses only the first
    _, c3 = bm.add_sequence(3, prefix[:6] + [77] * 6)
    assert c3 == 4
    # released cached blocks stay reusable
    bm.free_sequence(1)
    bm.free_sequence(2)
    bm.free_sequence(3)
    assert bm.stats()["cached_free_blocks"] > 0
    _, c4 = bm.add_sequence(4, prefix + [1])
    assert c4 == 12


def test_blocks_filled_by_decode_join_the_cache():
    bm = pa.BlockManager(32, 4)
    bm.add_sequence(1, [1, 2, 3])
    for tok in (4, 5, 6, 7, 8):
        bm.append_token(1, tok)
    _, cached = bm.add_sequence(2, [1, 2, 3, 4, 5, 6, 7, 8, 9])
    assert cached == 8


def test_eviction_takes_least_recently_released_leaves():
    bm = pa.BlockManager(6, 2)
    bm.add_sequence(1, [1, 2, 3, 4])            # A=[1,2], B=[3,4] under A
    bm.add_sequence(2, [9, 8, 7, 6])            # C=[9,8], D=[7,6] under C
    bm.free_sequence(1)                         # released: B, A
    bm.free_sequence(2)                         # then D, C
    st = bm.stats()
    assert st["cached_free_blocks"] == 4 and st["free_blocks"] == 2
    # 4 blocks: the 2 free ones, then the oldest released leaves B and A
    bm.add_sequence(3, [40, 41, 42, 43, 44, 45, 46, 47])
    assert bm.stats()["evictions"] == 2
    _, c = bm.add_sequence(4, [9, 8, 7, 6])     # C and D survived
    assert c == 4
    with pytest.raises(pa.PAError) as e:        # A and B are gone, and nothing is left to evict
        bm.add_sequence(5, [1, 2, 3, 4])
    assert e.value.status == pa.capi.PA_ERR_NO_BLOCKS


def test_exhaustion_leaves_the_manager_unchanged():
    bm = pa.BlockManager(4, 4, prefix_cache=True)
    bm.add_sequence(1, np.arange(12))
    before = bm.stats()
    with pytest.raises(pa.PAError) as e:
        bm.add_sequence(2, np.arange(100, 108))
    assert e.value.status == pa.capi.PA_ERR_NO_BLOCKS
    after = bm.stats()
    for k in ("free_blocks", "cached_free_blocks", "used_blocks", "num_sequences"):
        assert before[k] == after[k]
    with pytest.raises(pa.PAError):
        bm.seq_len(2)


def test_bad_arguments():
    with pytest.raises(ValueError):
        pa.BlockManager(0, 16)
    bm = pa.BlockManager(4, 4)
    bm.add_sequence(1, [1])
    with pytest.raises(pa.PAError):
        bm.add_sequence(1, [2])                 # duplicate id
    with pytest.raises(pa.PAError):
        bm.fork(5, 6)                           # unknown parent
    with pytest.raises(pa.PAError):
        bm.append_token(9, 1)


# ---------------------------------------------------------------- simulation

def _kv_of(prefix, D, salt):
    """K or V row of the last token of ``prefix``: a deterministic function of
    the whole prefix (as the K/V of a real model is), fp16 bit patterns."""
    h = 1469598103934665603 ^ salt
    for t in prefix:
        h = ((h ^ (int(t) & 0xFFFFFFFF)) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    rng = np.random.Generator(np.random.PCG64(h))
    return rng.standard_normal(D).astype(np.float16).view(np.uint16)


def _simulate(seed, prefix_cache, steps=160, num_blocks=40, bs=4, D=8):
    rng = np.random.Generator(np.random.PCG64(seed))
    bm = pa.BlockManager(num_blocks, bs, prefix_cache=prefix_cache)
    kc = np.zeros((num_blocks, 1, bs, D), np.uint16)
    vc = np.zeros_like(kc)
    tokens = {}
    next_id = 0
    prompts = [list(rng.integers(0, 5, size=int(rng.integers(1, 14)))) for _ in range(6)]

    def write(seq, slot):
        pre = tokens[seq]
        b, o = divmod(slot, bs)
        kc[b, 0, o] = _kv_of(pre, D, 1)
        vc[b, 0, o] = _kv_of(pre, D, 2)

    for _ in range(steps):
        op = rng.integers(0, 10)
        live = sorted(tokens)
        try:
            if op < 3 or not live:
                base = prompts[int(rng.integers(0, len(prompts)))]
                toks = base + list(rng.integers(0, 5, size=int(rng.integers(0, 6))))
                slots, cached = bm.add_sequence(next_id, toks)
                tokens[next_id] = []
                for i, t in enumerate(toks):
                    tokens[next_id].append(int(t))
                    if i >= cached:
                        assert slots[i] >= 0
                        write(next_id, int(slots[i]))
                    else:
                        assert slots[i] == -1
                next_id += 1
            elif op < 4:
                parent = live[int(rng.integers(0, len(live)))]
                bm.fork(parent, next_id)
                tokens[next_id] = list(tokens[parent])
                next_id += 1
            elif op < 9:
                s = live[int(rng.integers(0, len(live)))]
                t = int(rng.integers(0, 5))
                slot, pair = bm.append_token(s, t)
                if pair is not None:
                    assert oracle.copy_blocks(kc, vc, np.array([pair], np.int64)) == 0
                tokens[s].append(t)
                write(s, slot)
                assert bm.refcount(slot // bs) == 1  # a written block is never shared
            else:
                s = live[int(rng.integers(0, len(live)))]
                bm.free_sequence(s)
                del tokens[s]
        except pa.PAError as e:
            assert e.status == pa.capi.PA_ERR_NO_BLOCKS
        # invariants
        st = bm.stats()
        assert st["free_blocks"] + st["cached_free_blocks"] + st["used_blocks"] == num_blocks
        held = {}
        for s in tokens:
            for b in bm.block_table(s):
                held[int(b)] = held.get(int(b), 0) + 1
            assert bm.seq_len(s) == len(tokens[s])
        for b, n in held.items():
            assert bm.refcount(b) == n
    return bm, kc, vc, tokens


@pytest.mark.parametrize("prefix_cache", [True, False])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_simulated_engine_reads_back_every_sequence(seed, prefix_cache):
    bm, kc, vc, tokens = _simulate(seed, prefix_cache)
    bs, D = 4, 8
    for s, toks in tokens.items():
        table = bm.block_table(s)
        for i in range(len(toks)):
            b, o = int(table[i // bs]), i % bs
            assert np.array_equal(kc[b, 0, o], _kv_of(toks[:i + 1], D, 1))
            assert np.array_equal(vc[b, 0, o], _kv_of(toks[:i + 1], D, 2))
    st = bm.stats()
    if prefix_cache:
        assert st["hit_tokens"] > 0
    assert st["cow_copies"] > 0


def test_oracle_decode_over_manager_tables_equals_logical_attention():
    bm, kc, vc, tokens = _simulate(11, True, steps=150)
    seqs = [s for s in sorted(tokens) if tokens[s]]
    bs, D = 4, 8
    tables = bm.tables(seqs)
    lens = np.array([len(tokens[s]) for s in seqs], np.int32)
    rng = np.random.Generator(np.random.PCG64(5))
    q = rng.standard_normal((len(seqs), 1, D)).astype(np.float16).view(np.uint16)
    out = oracle.decode(q, kc, vc, tables, lens, 0.35, "f16", num_threads=2)
    for i, s in enumerate(seqs):
        K = np.stack([_kv_of(tokens[s][:j + 1], D, 1) for j in range(lens[i])]).view(np.float16).astype(np.float64)
        V = np.stack([_kv_of(tokens[s][:j + 1], D, 2) for j in range(lens[i])]).view(np.float16).astype(np.float64)
        z = 0.35 * K @ q[i, 0].view(np.float16).astype(np.float64)
        p = np.exp(z - z.max())
        ref = (p @ V) / p.sum()
        assert np.allclose(out[i, 0], ref, rtol=0, atol=1e-12)
