"""Shared test helpers: tolerances, oracle input extraction, comparisons."""
from __future__ import annotations

import math

import numpy as np
import torch

from paged_kv_cache_224_gb300 import workload as wl

# Max abs error bounds for attention outputs, fp32 accumulation.
TOL = {"f16": 2e-3, "bf16": 1e-2}
MANTISSA = {"f16": 10, "bf16": 7}


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of ``dtype`` at |ref| (the error of one
    correct rounding of the exact result)."""
    a = np.maximum(np.abs(ref), 2.0 ** -14)
    e = np.floor(np.log2(a))
    return 0.5 * 2.0 ** (e - MANTISSA[dtype])


def check_attention(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> dict:
    """|got - ref| <= TOL[dtype] everywhere, except where even a correctly
    rounded result cannot meet it (|ref| large enough that half an ulp of the
    output dtype exceeds TOL); there the bound is that half ulp plus fp32
    accumulation slack.  Returns error statistics."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    floor = half_ulp(ref, dtype) * (1 + 2.0 ** -6) + 1e-5 * np.maximum(1.0, np.abs(ref))
    bound = np.maximum(TOL[dtype], floor)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements over bound, max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return {"max_err": float(err.max()), "over_tol_within_rounding": int((err > TOL[dtype]).sum())}


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_inputs(case: wl.DecodeCase, tensors: dict, seqs) -> dict:
    """Host copies, for the oracle, of everything sequences ``seqs`` touch,
    taken from the ORIGINAL input tensors (before any kernel ran), with the
    pool compacted to just the blocks involved and all ids remapped.

    Includes the copy-on-write sources of those sequences and the new tokens
    that belong to them, so the oracle replays the whole step itself.
    """
    seqs = [int(s) for s in seqs]
    bs = case.block_size
    blocks = []
    for s in seqs:
        n = wl.blocks_for(int(case.context_lens[s]), bs)
        blocks.extend(int(b) for b in case.block_tables[s, :n])
    dsts = set(blocks)
    pairs = [(int(a), int(b)) for a, b in case.cow_pairs if int(b) in dsts]
    blocks.extend(a for a, _ in pairs)
    uniq = sorted(set(blocks))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.as_tensor(uniq, dtype=torch.long, device=tensors["k_cache"].device)
    kc = wl.bits(tensors["k_cache"].index_select(0, idx))
    vc = wl.bits(tensors["v_cache"].index_select(0, idx))
    mb = max(1, max(wl.blocks_for(int(case.context_lens[s]), bs) for s in seqs))
    bt = np.full((len(seqs), mb), -1, np.int32)
    for i, s in enumerate(seqs):
        n = wl.blocks_for(int(case.context_lens[s]), bs)
        bt[i, :n] = [remap[int(b)] for b in case.block_tables[s, :n]]
    sel = np.isin(case.new_token_seq, seqs)
    tok = np.nonzero(sel)[0]
    slots = case.slot_mapping[tok]
    new_slots = np.array([remap[int(x) // bs] * bs + int(x) % bs for x in slots], np.int64)
    tidx = torch.as_tensor(tok, dtype=torch.long, device=tensors["new_key"].device)
    nk = wl.bits(tensors["new_key"].index_select(0, tidx))
    nv = wl.bits(tensors["new_value"].index_select(0, tidx))
    sidx = torch.as_tensor(seqs, dtype=torch.long, device=tensors["query"].device)
    q = wl.bits(tensors["query"].index_select(0, sidx))
    cp = np.array([(remap[a], remap[b]) for a, b in pairs], np.int64).reshape(-1, 2)
    return dict(k_cache=kc, v_cache=vc, block_tables=bt, context_lens=case.context_lens[seqs].copy(),
                query=q, new_key=nk, new_value=nv, slot_mapping=new_slots, cow_pairs=cp)


def oracle_step(oracle, case: wl.DecodeCase, inp: dict, threads: int = 8) -> np.ndarray:
    """Replay copy-on-write, cache write and decode on the oracle."""
    kc, vc = inp["k_cache"], inp["v_cache"]
    assert oracle.copy_blocks(kc, vc, inp["cow_pairs"]) == 0
    assert oracle.reshape_and_cache(inp["new_key"], inp["new_value"], kc, vc, inp["slot_mapping"],
                                    case.block_size) == 0
    return oracle.decode(inp["query"], kc, vc, inp["block_tables"], inp["context_lens"], case.scale,
                         case.dtype, num_threads=threads)


def sample_seqs(case: wl.DecodeCase, k: int, seed: int = 0) -> list:
    """k sequences: the shortest, the longest, and random others."""
    lens = case.context_lens
    rng = np.random.default_rng(seed)
    pick = {int(lens.argmin()), int(lens.argmax())}
    others = rng.permutation(case.num_seqs)
    for s in others:
        if len(pick) >= min(k, case.num_seqs):
            break
        pick.add(int(s))
    return sorted(pick)


def scale_for(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
