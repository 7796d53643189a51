"""Pins for the CPU oracle, checked against things other than itself.

* the 16-bit decoders against numpy's own float16 / float32 conversions for
  every bit pattern;
* the worked block-table example printed on the page "vLLM PagedAttention
  chuyen sau" (first code listing: 30 tokens -> blocks 10, 25; 50 tokens ->
  blocks 3, 7, 12, 18 at block_size 16), stored in tests/golden;
* special cases that reduce to a library routine: unpaged attention equals
  ``torch.nn.functional.scaled_dot_product_attention`` in float64 (with
  ``enable_gqa`` for grouped heads, and an explicit causal mask for a chunk);
* closed forms: one token -> its V row exactly; equal keys or a zero query ->
  the mean of V;
* the pages' invariants: physical placement does not matter, shared prefix
  blocks equal private copies, copy-on-write isolates the writer.

Several tests also plant a plausible mistake on the CPU and check that the
pin would have caught it.
"""
import json
import math
import os
import zlib

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from paged_kv_cache_224_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NP16 = {"f16": np.float16}


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(wl.TORCH_DTYPES[dtype])
    return wl.bits(t)


def bits_to_f64(b: np.ndarray, dtype: str) -> np.ndarray:
    # numpy/torch conversions -- independent of the oracle's decoder
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(wl.TORCH_DTYPES[dtype])
    return t.to(torch.float64).numpy()


def paged_from_contiguous(rng, K, V, tables_lens, block_size, num_blocks, dtype):
    """Scatter contiguous per-sequence K/V ([L][Hkv][D] float arrays) into a
    random pool through explicit tables, using plain indexing."""
    Hkv, D = K[0].shape[1], K[0].shape[2]
    kc = to_bits(rng.standard_normal((num_blocks, Hkv, block_size, D)), dtype)
    vc = to_bits(rng.standard_normal((num_blocks, Hkv, block_size, D)), dtype)
    for (table, L), k, v in zip(tables_lens, K, V):
        kb, vb = to_bits(k, dtype), to_bits(v, dtype)
        for t in range(L):
            blk, off = table[t // block_size], t % block_size
            kc[blk, :, off, :] = kb[t]
            vc[blk, :, off, :] = vb[t]
    return kc, vc


def sdpa_reference(q_bits, K_bits, V_bits, scale, dtype, mask=None):
    """Library attention, float64: q [Hq][n_q][D], K/V [L][Hkv][D] bits."""
    q = torch.from_numpy(bits_to_f64(q_bits, dtype))
    K = torch.from_numpy(bits_to_f64(K_bits, dtype)).permute(1, 0, 2)
    V = torch.from_numpy(bits_to_f64(V_bits, dtype)).permute(1, 0, 2)
    gqa = q.shape[0] != K.shape[0]
    out = F.scaled_dot_product_attention(q[None], K[None], V[None], attn_mask=mask, scale=scale,
                                         enable_gqa=gqa)
    return out[0].numpy()


# ------------------------------------------------------------------ decoders

def test_f16_decoder_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode_bits(pats, "f16")
    want = pats.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_decoder_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode_bits(pats, "bf16")
    with np.errstate(invalid="ignore"):
        want = (pats.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# ------------------------------------------------- the page's worked example

def test_page_block_table_example(oracle_mod):
    ex = json.load(open(os.path.join(GOLDEN, "page_block_table_example.json")))
    bs = ex["block_size"]
    for s in ex["sequences"]:
        assert wl.blocks_for(s["tokens"], bs) == s["blocks"] == len(s["table"])
    # Place the two sequences exactly where the page puts them and check that
    # the oracle's gather-then-attend equals library attention on the
    # unpaged rows.
    rng = np.random.default_rng(7)
    Hkv, G, D = 2, 2, 64
    lens = [s["tokens"] for s in ex["sequences"]]
    tables = [s["table"] for s in ex["sequences"]]
    NB = max(max(t) for t in tables) + 1
    K = [rng.standard_normal((L, Hkv, D)) for L in lens]
    V = [rng.standard_normal((L, Hkv, D)) for L in lens]
    kc, vc = paged_from_contiguous(rng, K, V, list(zip(tables, lens)), bs, NB, "f16")
    bt = np.full((2, 4), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    q = to_bits(rng.standard_normal((2, Hkv * G, D)), "f16")
    scale = 1 / math.sqrt(D)
    got = oracle_mod.decode(q, kc, vc, bt, np.array(lens, np.int32), scale, "f16")
    for i in range(2):
        want = sdpa_reference(q[i][:, None, :], to_bits(K[i], "f16"), to_bits(V[i], "f16"), scale, "f16")
        np.testing.assert_allclose(got[i], want[:, 0, :], rtol=1e-12, atol=1e-13)
    # token 17 of the 50-token sequence is logical block 1 -> physical block 7, offset 1
    assert np.array_equal(kc[7, :, 1, :], to_bits(K[1][17], "f16"))


def test_tiny_workload_block_counts():
    c = wl.tiny_case()
    need = [wl.blocks_for(L, 16) for L in c.context_lens]
    assert need == [2, 4, 2, 4] and sum(need) == 12
    assert c.num_blocks == 64
    used = np.concatenate([c.block_tables[s, :n] for s, n in enumerate(need)])
    assert len(set(used.tolist())) == 12 and used.min() >= 0 and used.max() < 64
    # unused table entries stay -1
    for s, n in enumerate(need):
        assert (c.block_tables[s, n:] == -1).all()
    # internal fragmentation: < one block per sequence
    assert c.internal_waste_tokens() == sum(n * 16 - L for n, L in zip(need, c.context_lens))
    assert c.internal_waste_tokens() < 16 * c.num_seqs


# ------------------------------------------- library routine on random cases

CASES = [
    # (G, Hkv, D, bs, dtype, lens)
    (1, 3, 64, 16, "f16", [1, 16, 17, 40]),
    (2, 2, 128, 16, "bf16", [5, 33, 64]),
    (4, 2, 64, 32, "f16", [31, 32, 33, 100]),
    (8, 1, 128, 32, "bf16", [2, 65, 96]),
    (4, 2, 128, 8, "f16", [9, 24]),
]


@pytest.mark.parametrize("G,Hkv,D,bs,dtype,lens", CASES)
def test_decode_equals_library_attention(oracle_mod, G, Hkv, D, bs, dtype, lens):
    rng = np.random.default_rng(zlib.crc32(repr((G, Hkv, D, bs, dtype)).encode()))
    need = [wl.blocks_for(L, bs) for L in lens]
    NB = sum(need) + 5
    perm = rng.permutation(NB)
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n].tolist())
        at += n
    K = [rng.standard_normal((L, Hkv, D)) for L in lens]
    V = [rng.standard_normal((L, Hkv, D)) for L in lens]
    kc, vc = paged_from_contiguous(rng, K, V, list(zip(tables, lens)), bs, NB, dtype)
    bt = np.full((len(lens), max(need)), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    Hq = G * Hkv
    q = to_bits(rng.standard_normal((len(lens), Hq, D)), dtype)
    scale = 1 / math.sqrt(D)
    got = oracle_mod.decode(q, kc, vc, bt, np.array(lens, np.int32), scale, dtype)
    for i in range(len(lens)):
        want = sdpa_reference(q[i][:, None, :], to_bits(K[i], dtype), to_bits(V[i], dtype), scale, dtype)
        np.testing.assert_allclose(got[i], want[:, 0, :], rtol=1e-11, atol=1e-12)
    # planted mistake: mapping query head h to kv head h % Hkv instead of
    # h // G must disagree with the library (caught by this pin)
    if G > 1 and Hkv > 1:
        wrong = np.stack([bits_to_f64(q[0], dtype)[h] for h in range(Hq)])
        kv_of = [h % Hkv for h in range(Hq)]
        Kc = bits_to_f64(to_bits(K[0], dtype), dtype)
        Vc = bits_to_f64(to_bits(V[0], dtype), dtype)
        rows = []
        for h in range(Hq):
            z = scale * Kc[:, kv_of[h], :] @ wrong[h]
            p = np.exp(z - z.max())
            rows.append(p @ Vc[:, kv_of[h], :] / p.sum())
        assert not np.allclose(np.stack(rows), got[0], atol=1e-6)


def test_oracle_threads_identical(oracle_mod):
    c = wl.make_decode_case("t", [3, 70, 128, 1, 45], 8, 2, 64, 16, "bf16", seed=5)
    t = c.materialize("cpu")
    args = (wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"]), c.block_tables,
            c.context_lens, c.scale, c.dtype)
    a = oracle_mod.decode(*args, num_threads=1)
    b = oracle_mod.decode(*args, num_threads=4)
    assert np.array_equal(a, b)


# ------------------------------------------------------------ closed forms

def test_single_token_returns_its_value_row(oracle_mod):
    c = wl.make_decode_case("t", [1, 1], 4, 2, 128, 16, "bf16", seed=11)
    t = c.materialize("cpu")
    out = oracle_mod.decode(wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"]),
                            c.block_tables, c.context_lens, c.scale, c.dtype)
    vc = bits_to_f64(wl.bits(t["v_cache"]), "bf16")
    for s in range(2):
        blk = c.block_tables[s, 0]
        for h in range(4):
            assert np.array_equal(out[s, h], vc[blk, h // 2, 0])


def test_equal_keys_or_zero_query_give_mean_value(oracle_mod):
    rng = np.random.default_rng(3)
    L, Hkv, D, bs = 37, 1, 64, 16
    key_row = rng.standard_normal(D)
    K = [np.broadcast_to(key_row, (L, Hkv, D)).copy()]
    V = [rng.standard_normal((L, Hkv, D))]
    table = [5, 0, 3]
    kc, vc = paged_from_contiguous(rng, K, V, [(table, L)], bs, 6, "f16")
    bt = np.array([table], np.int32)
    q = to_bits(rng.standard_normal((1, 1, D)), "f16")
    vmean = bits_to_f64(to_bits(V[0], "f16"), "f16").mean(axis=0)[0]
    out = oracle_mod.decode(q, kc, vc, bt, np.array([L], np.int32), 0.125, "f16")
    np.testing.assert_allclose(out[0, 0], vmean, rtol=1e-13, atol=1e-14)
    # zero query, random keys: uniform weights again
    kc2, vc2 = paged_from_contiguous(rng, [rng.standard_normal((L, Hkv, D))], V, [(table, L)], bs, 6, "f16")
    out = oracle_mod.decode(np.zeros((1, 1, D), np.uint16), kc2, vc2, bt, np.array([L], np.int32), 0.125, "f16")
    np.testing.assert_allclose(out[0, 0], vmean, rtol=1e-13, atol=1e-14)
    # planted mistake: off-by-one on the length (attending L-1 rows) is caught
    short = bits_to_f64(to_bits(V[0], "f16"), "f16")[:L - 1].mean(axis=0)[0]
    assert not np.allclose(short, out[0, 0], atol=1e-6)


def test_zero_length_gives_zeros(oracle_mod):
    c = wl.make_decode_case("t", [0, 5], 2, 2, 64, 16, "f16", seed=2)
    t = c.materialize("cpu")
    out = oracle_mod.decode(wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"]),
                            c.block_tables, c.context_lens, c.scale, c.dtype)
    assert (out[0] == 0).all() and np.abs(out[1]).sum() > 0


# ------------------------------------------------------------- invariants

def test_physical_permutation_invariance(oracle_mod):
    c = wl.make_decode_case("t", [30, 50, 17, 64], 8, 4, 64, 16, "f16", seed=13, num_blocks=40)
    t = c.materialize("cpu")
    q, kc, vc = wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    a = oracle_mod.decode(q, kc, vc, c.block_tables, c.context_lens, c.scale, c.dtype)
    pi = np.random.default_rng(1).permutation(c.num_blocks)      # block b moves to pi[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    bt2 = np.where(c.block_tables >= 0, pi[np.maximum(c.block_tables, 0)], -1).astype(np.int32)
    b = oracle_mod.decode(q, kc2, vc2, bt2, c.context_lens, c.scale, c.dtype)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("G", [2, 4, 8])
def test_grouped_heads_equal_mha_with_kv_heads_repeated(oracle_mod, G):
    # the textbook reduction: query head h of a group-of-G model attends to kv
    # head h // G, i.e. to the same rows as an MHA model whose pool holds
    # each kv head G times in a row (a wrong head map, e.g. h % Hkv, breaks it)
    Hkv = 2
    c = wl.make_decode_case("gqa", [30, 50, 17, 64], G * Hkv, Hkv, 64, 16, "bf16", seed=17 + G)
    t = c.materialize("cpu")
    q, kc, vc = wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    gqa = oracle_mod.decode(q, kc, vc, c.block_tables, c.context_lens, c.scale, c.dtype)
    kc_rep = np.ascontiguousarray(np.repeat(kc, G, axis=1))   # [NB][Hkv*G][bs][D]
    vc_rep = np.ascontiguousarray(np.repeat(vc, G, axis=1))
    mha = oracle_mod.decode(q, kc_rep, vc_rep, c.block_tables, c.context_lens, c.scale, c.dtype)
    assert np.array_equal(gqa, mha)


def test_shared_prefix_equals_private_copies(oracle_mod):
    c = wl.make_shared_prefix_case("t", num_prompts=2, samples=3, prefix_len=40, max_tail=20,
                                   num_heads=2, head_dim=64, block_size=16, dtype="f16", seed=4)
    t = c.materialize("cpu")
    q, kc, vc = wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert oracle_mod.copy_blocks(kc, vc, c.cow_pairs) == 0
    nk, nv = wl.bits(t["new_key"]), wl.bits(t["new_value"])
    assert oracle_mod.reshape_and_cache(nk, nv, kc, vc, c.slot_mapping, c.block_size) == 0
    shared = oracle_mod.decode(q, kc, vc, c.block_tables, c.context_lens, c.scale, c.dtype)
    assert c.refcounts.max() == 3
    # give every sequence private copies of every block it references
    rows = []
    bt2 = np.full_like(c.block_tables, -1)
    for s in range(c.num_seqs):
        for j in range(wl.blocks_for(c.context_lens[s], c.block_size)):
            bt2[s, j] = len(rows)
            rows.append(c.block_tables[s, j])
    kc2, vc2 = kc[np.array(rows)].copy(), vc[np.array(rows)].copy()
    private = oracle_mod.decode(q, kc2, vc2, bt2, c.context_lens, c.scale, c.dtype)
    assert np.array_equal(shared, private)


def test_copy_on_write_isolates_the_writer(oracle_mod):
    c = wl.make_shared_prefix_case("t", num_prompts=1, samples=4, prefix_len=24, max_tail=0,
                                   num_heads=2, head_dim=64, block_size=16, dtype="bf16", seed=9)
    t = c.materialize("cpu")
    q, kc, vc = wl.bits(t["query"]), wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    assert c.cow_pairs.shape == (3, 2)
    assert oracle_mod.copy_blocks(kc, vc, c.cow_pairs) == 0
    for src, dst in c.cow_pairs:
        assert np.array_equal(kc[dst], kc[src]) and np.array_equal(vc[dst], vc[src])
    before = oracle_mod.decode(q, kc, vc, c.block_tables, c.context_lens, c.scale, c.dtype)
    # sample 0 writes its 25th token into its private copy of the partial block
    lens = c.context_lens.copy()
    lens[0] += 1
    slot = np.array([c.block_tables[0, 1] * 16 + 8], np.int64)
    rng = np.random.default_rng(0)
    nk = to_bits(rng.standard_normal((1, 2, 64)), "bf16")
    assert oracle_mod.reshape_and_cache(nk, nk, kc, vc, slot, 16) == 0
    after = oracle_mod.decode(q, kc, vc, c.block_tables, lens, c.scale, c.dtype)
    assert np.array_equal(before[1:], after[1:])
    assert not np.array_equal(before[0], after[0])


def test_reshape_and_cache_places_new_token_at_last_position(oracle_mod):
    c = wl.make_decode_case("t", [30, 50, 17, 64, 0], 4, 4, 64, 16, "f16", seed=21, num_blocks=64)
    t = c.materialize("cpu")
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    nk, nv = wl.bits(t["new_key"]), wl.bits(t["new_value"])
    assert c.num_new_tokens == 4          # the empty sequence gets no token
    kc0 = kc.copy()
    slots = np.concatenate([c.slot_mapping, [-1, -5]])   # padding slots write nothing
    nk2 = np.concatenate([nk, nk[:2]])
    nv2 = np.concatenate([nv, nv[:2]])
    assert oracle_mod.reshape_and_cache(nk2, nv2, kc, vc, slots, 16) == 0
    for i, s in enumerate(c.new_token_seq):
        L = c.context_lens[s]
        blk = c.block_tables[s, (L - 1) // 16]
        assert np.array_equal(kc[blk, :, (L - 1) % 16], nk[i])
        assert np.array_equal(vc[blk, :, (L - 1) % 16], nv[i])
    changed = np.argwhere((kc != kc0).any(axis=(1, 3)))
    assert len(changed) <= 4 * 4
    # a slot past the pool is skipped and counted
    assert oracle_mod.reshape_and_cache(nk[:1], nv[:1], kc, vc, np.array([64 * 16]), 16) == 1


def test_copy_blocks_rejects_conflicting_pairs(oracle_mod):
    rng = np.random.default_rng(0)
    kc = rng.integers(0, 65535, size=(8, 2, 16, 64), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(8, 2, 16, 64), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[0, 1],    # fine
                      [2, 2],    # src == dst
                      [3, 4],    # dst 4 twice
                      [5, 4],
                      [6, 0],    # dst 0 is a src
                      [7, 9]],   # dst out of pool
                     np.int64)
    assert oracle_mod.copy_blocks(kc, vc, pairs) == 5
    assert np.array_equal(kc[1], k0[0]) and np.array_equal(vc[1], v0[0])
    for b in (0, 2, 3, 4, 5, 6, 7):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])


# ---------------------------------------------------------- chunked prefill

@pytest.mark.parametrize("P,C,G,Hkv,bs,dtype", [(40, 9, 2, 2, 16, "bf16"), (0, 17, 4, 1, 32, "f16"),
                                                (64, 16, 1, 2, 16, "f16")])
def test_prefill_chunk_equals_masked_library_attention(oracle_mod, P, C, G, Hkv, bs, dtype):
    case = wl.make_prefill_case("t", P, C, G * Hkv, Hkv, 64, bs, dtype, seed=P + C)
    t = case.materialize("cpu")
    kc, vc = wl.bits(t["k_cache"]), wl.bits(t["v_cache"])
    nk, nv = wl.bits(t["new_key"]), wl.bits(t["new_value"])
    assert oracle_mod.reshape_and_cache(nk, nv, kc, vc, case.slot_mapping, bs) == 0
    q = wl.bits(t["query"])
    got = oracle_mod.prefill_chunk(q, kc, vc, case.block_table, P, case.scale, dtype)
    # unpaged rows 0..P+C-1 by plain indexing
    pos = np.arange(P + C)
    blk = case.block_table[pos // bs]
    Kc = kc[blk, :, pos % bs, :]
    Vc = vc[blk, :, pos % bs, :]
    mask = torch.from_numpy(np.arange(P + C)[None, :] <= (P + np.arange(C))[:, None])
    want = sdpa_reference(q.transpose(1, 0, 2), Kc, Vc, case.scale, dtype, mask=mask)
    np.testing.assert_allclose(got, want.transpose(1, 0, 2), rtol=1e-11, atol=1e-12)
    # a one-row chunk reduces to decode at context P+1
    lens = np.array([P + 1], np.int32)
    dec = oracle_mod.decode(q[:1], kc, vc, case.block_table[None, :], lens, case.scale, dtype)
    np.testing.assert_allclose(dec[0], got[0], rtol=1e-13, atol=1e-14)
