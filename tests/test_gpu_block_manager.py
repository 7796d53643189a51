"""The block manager drives the GPU kernels through several engine steps.

Prompts with common prefixes (prefix-cache hits), forked samples (shared
blocks, copy-on-write on their first decode token) and per-step growth: each
step the manager's copy pairs go to pa_copy_blocks, its slots to
pa_reshape_and_cache, its tables to pa_decode.  The same copy pairs and
slots are replayed on the CPU oracle's own pool (oracle.copy_blocks,
oracle.reshape_and_cache), so the oracle's decode over the manager's tables
is the checker: the GPU output must match it within the attention tolerance,
and the GPU pool must equal the oracle's pool bit for bit.  Every token's K/V
is also a function of its whole token prefix, so each sequence's attention is
recomputed a second way from its logical token list alone, with no pool, and
the GPU pool must hold each sequence's K/V at the positions its table names.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_224_gb300 as pa
from paged_kv_cache_224_gb300 import workload as wl
from tests.helpers import check_attention, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
BS, HKV, G, D = 16, 2, 2, 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def kv_row(prefix, salt):
    """[Hkv][D] fp16 K (salt 1) or V (salt 2) of the last token of prefix."""
    h = 1469598103934665603 ^ salt
    for t in prefix:
        h = ((h ^ (int(t) & 0xFFFFFFFF)) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    rng = np.random.Generator(np.random.PCG64(h))
    return rng.standard_normal((HKV, D)).astype(np.float16)


def logical_attention(tokens, q, scale):
    K = np.stack([kv_row(tokens[:j + 1], 1) for j in range(len(tokens))]).astype(np.float64)  # [L][Hkv][D]
    V = np.stack([kv_row(tokens[:j + 1], 2) for j in range(len(tokens))]).astype(np.float64)
    out = np.zeros((HKV * G, D))
    for h in range(HKV * G):
        kvh = h // G
        z = scale * K[:, kvh, :] @ q[h].astype(np.float64)
        p = np.exp(z - z.max())
        out[h] = (p @ V[:, kvh, :]) / p.sum()
    return out


def test_block_manager_drives_the_kernels():
    rng = np.random.Generator(np.random.PCG64(2024))
    nb = 256
    bm = pa.BlockManager(nb, BS, prefix_cache=True)
    kc = torch.zeros((nb, HKV, BS, D), dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    ko, vo = wl.bits(kc), wl.bits(vc)  # the oracle's pool, updated by the oracle's own cache calls
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tokens = {}

    def write(seq_slots):
        """K/V rows of (seq, position, slot) triples into the pool on the GPU."""
        if not seq_slots:
            return
        k = np.stack([kv_row(tokens[s][:i + 1], 1) for s, i, _ in seq_slots])
        v = np.stack([kv_row(tokens[s][:i + 1], 2) for s, i, _ in seq_slots])
        sl = np.array([sl for _, _, sl in seq_slots], np.int64)
        pa.pa_reshape_and_cache(torch.as_tensor(k, device=DEV), torch.as_tensor(v, device=DEV), kc, vc,
                                torch.as_tensor(sl, device=DEV), d_err=err)
        assert oracle.reshape_and_cache(k.view(np.uint16), v.view(np.uint16), ko, vo, sl, BS) == 0

    p0 = list(rng.integers(0, 1000, size=100))
    prompts = {0: p0, 1: p0[:64] + list(rng.integers(0, 1000, size=16)), 2: list(rng.integers(0, 1000, size=37))}
    prompts[3] = list(prompts[2])
    hits = {}
    batch = []
    for sid, toks in prompts.items():
        slots, cached = bm.add_sequence(sid, toks)
        hits[sid] = cached
        tokens[sid] = [int(t) for t in toks]
        batch += [(sid, i, int(slots[i])) for i in range(cached, len(toks))]
    write(batch)
    assert hits == {0: 0, 1: 64, 2: 0, 3: 32}
    for child in (10, 11, 12):
        bm.fork(0, child)
        tokens[child] = list(tokens[0])

    scale = 1.0 / np.sqrt(D)
    for step in range(20):
        pairs, batch = [], []
        for sid in sorted(tokens):
            t = int(rng.integers(0, 1000))
            slot, pair = bm.append_token(sid, t)
            tokens[sid].append(t)
            if pair is not None:
                pairs.append(pair)
            batch.append((sid, len(tokens[sid]) - 1, slot))
        if step == 0:
            assert len(pairs) == 3  # the samples' first tokens land in copies of the shared partial block
        if pairs:
            pa.pa_copy_blocks(kc, vc, torch.as_tensor(pairs, dtype=torch.int64, device=DEV), d_err=err)
            assert oracle.copy_blocks(ko, vo, np.array(pairs, np.int64)) == 0
        write(batch)
        if step in (0, 7, 19):
            seqs = sorted(tokens)
            lens = [len(tokens[s]) for s in seqs]
            tables = bm.tables(seqs)
            bt = torch.as_tensor(tables, device=DEV)
            q = torch.as_tensor(rng.standard_normal((len(seqs), HKV * G, D)).astype(np.float16), device=DEV)
            out = torch.full_like(q, float("nan"))
            pa.pa_decode(out, q, kc, vc, bt, torch.as_tensor(lens, dtype=torch.int32, device=DEV), scale,
                         max(lens), d_err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert np.array_equal(wl.bits(kc), ko) and np.array_equal(wl.bits(vc), vo)
            ref = oracle.decode(wl.bits(q), ko, vo, np.ascontiguousarray(tables, np.int32),
                                np.array(lens, np.int32), scale, "f16", num_threads=8)
            check_attention(to_f64(out), ref, "f16", f"step {step} vs oracle")
            qh = q.cpu().numpy()
            logical = np.stack([logical_attention(tokens[s], qh[i], scale) for i, s in enumerate(seqs)])
            check_attention(to_f64(out), logical, "f16", f"step {step} vs logical attention")
    # the pool holds every sequence's K/V where its table says, bit for bit
    kh, vh = kc.cpu().numpy(), vc.cpu().numpy()
    for s, toks in tokens.items():
        table = bm.block_table(s)
        for i in range(len(toks)):
            b, o = int(table[i // BS]), i % BS
            assert np.array_equal(kh[b, :, o], kv_row(toks[:i + 1], 1))
            assert np.array_equal(vh[b, :, o], kv_row(toks[:i + 1], 2))
    st = bm.stats()
    assert st["cow_copies"] == 3 and st["hit_tokens"] == 96
