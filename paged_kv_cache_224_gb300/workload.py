"""Seeded synthetic inputs for the paged-KV path.

This module draws inputs only: context lengths, a host-side block allocation
(block tables, slot mappings, copy-on-write pairs) and N(0,1) query / cache
values.  It contains none of the attention arithmetic, so both the CUDA path
and the CPU oracle can consume what it produces.

Recipe (the same for every workload):
  * integers (lengths, tail lengths, the block permutation) come from
    ``numpy.random.Generator(PCG64(seed))``;
  * values come from ``torch.Generator(device).manual_seed(seed)`` as
    ``torch.randn`` in the element dtype (N(0,1), round-to-nearest-even),
    drawn in the order k_cache, v_cache, query, new_key, new_value;
  * the physical pool holds ``ceil(1.25 * blocks needed)`` blocks unless a
    workload fixes it; physical blocks are handed out in the order of a
    seeded permutation, so a sequence's blocks are scattered across the pool;
  * every pool slot is filled with N(0,1) values, including slots no sequence
    owns, so a kernel that reads past a context length sees garbage;
  * unused block-table entries are -1, which a correct kernel never reads;
  * ``context_lens`` counts the newly written token, which sits at position
    L-1 of its sequence.

Cache layout: ``[num_blocks][num_kv_heads][block_size][head_dim]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def blocks_for(tokens: int, block_size: int) -> int:
    """Physical blocks a sequence of ``tokens`` tokens occupies (ceiling)."""
    return -(-int(tokens) // int(block_size))


@dataclasses.dataclass
class DecodeCase:
    """One decode step: metadata on the host, values as torch tensors."""
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    context_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray          # int32 [B][MB], unused = -1
    slot_mapping: np.ndarray          # int64 [T] slots of the new tokens
    new_token_seq: np.ndarray         # int64 [T] which sequence each new token belongs to
    new_token_pos: np.ndarray         # int64 [T] its position in that sequence
    cow_pairs: np.ndarray             # int64 [n][2] (src, dst) copy-on-write pairs, maybe empty
    refcounts: np.ndarray             # int32 [NB] how many tables reference each block
    seed: int
    tensors: dict = dataclasses.field(default_factory=dict)
    group_size: int = 1               # consecutive sequences sharing a prefix (parallel sampling)
    shared_blocks: int = 0            # full blocks every table of a group starts with

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes of one decode: each valid row once per kv head, K and V."""
        el = 2
        return int(self.context_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim * el

    def unique_kv_bytes(self) -> int:
        """KV bytes counting each referenced physical row once (shared blocks once)."""
        el = 2
        seen = {}
        for s in range(self.num_seqs):
            L = int(self.context_lens[s])
            for j in range(blocks_for(L, self.block_size)):
                blk = int(self.block_tables[s, j])
                rows = min(self.block_size, L - j * self.block_size)
                seen[blk] = max(seen.get(blk, 0), rows)
        return sum(seen.values()) * 2 * self.num_kv_heads * self.head_dim * el

    def decode_bytes(self) -> int:
        """Algorithmic bytes of one decode call: KV rows + Q + out + tables + lens."""
        el = 2
        q = self.num_seqs * self.num_heads * self.head_dim * el
        tables = sum(blocks_for(int(L), self.block_size) for L in self.context_lens) * 4
        return self.kv_bytes() + 2 * q + tables + 4 * self.num_seqs

    def reshape_bytes(self) -> int:
        """Bytes of one cache write: new K/V rows read and written, slots read."""
        el = 2
        row = self.num_kv_heads * self.head_dim * el
        return self.num_new_tokens * (4 * row + 8)

    def copy_bytes(self) -> int:
        el = 2
        blk = self.num_kv_heads * self.block_size * self.head_dim * el
        return int(self.cow_pairs.shape[0]) * 2 * 2 * blk + int(self.cow_pairs.size) * 8

    def internal_waste_tokens(self) -> int:
        """Slots allocated but unused at the end of each sequence's last block."""
        return int(sum(blocks_for(int(L), self.block_size) * self.block_size - int(L)
                       for L in self.context_lens))

    def materialize(self, device="cpu", pool_fill: Optional[float] = None) -> dict:
        """Draw the value tensors on ``device`` (seeded) and return them.

        ``pool_fill`` replaces every pool slot with this constant before the
        real rows are drawn -- used to plant NaN garbage in unowned slots.
        """
        g = torch.Generator(device=device)
        g.manual_seed(self.seed)
        dt = TORCH_DTYPES[self.dtype]
        NB, Hkv, bs, D = self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim
        shape = (NB, Hkv, bs, D)
        kc = torch.randn(shape, generator=g, device=device, dtype=dt)
        vc = torch.randn(shape, generator=g, device=device, dtype=dt)
        if pool_fill is not None:
            owned = torch.zeros(NB, dtype=torch.bool)
            for s in range(self.num_seqs):
                n = blocks_for(int(self.context_lens[s]), bs)
                owned[torch.as_tensor(self.block_tables[s, :n], dtype=torch.long)] = True
            unowned = (~owned).nonzero().flatten().to(device)
            kc[unowned] = pool_fill
            vc[unowned] = pool_fill
            # slots past the length inside owned last blocks
            for s in range(self.num_seqs):
                L = int(self.context_lens[s])
                if L % bs:
                    blk = int(self.block_tables[s, L // bs])
                    kc[blk, :, L % bs:, :] = pool_fill
                    vc[blk, :, L % bs:, :] = pool_fill
        q = torch.randn((self.num_seqs, self.num_heads, D), generator=g, device=device, dtype=dt)
        T = self.num_new_tokens
        nk = torch.randn((T, Hkv, D), generator=g, device=device, dtype=dt)
        nv = torch.randn((T, Hkv, D), generator=g, device=device, dtype=dt)
        self.tensors = dict(k_cache=kc, v_cache=vc, query=q, new_key=nk, new_value=nv)
        return self.tensors


def _scatter_tables(rng, lens: Sequence[int], block_size: int, num_blocks: Optional[int],
                    pool_factor: float):
    need = [blocks_for(L, block_size) for L in lens]
    total = int(sum(need))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * total)))
    if total > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {total}")
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(1, max(need) if need else 1)
    tables = np.full((len(lens), mb), -1, dtype=np.int32)
    at = 0
    for s, n in enumerate(need):
        tables[s, :n] = perm[at:at + n]
        at += n
    return tables, num_blocks


def _slots_of(tables, seqs, positions, block_size):
    seqs = np.asarray(seqs, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    blk = tables[seqs, positions // block_size].astype(np.int64)
    return blk * block_size + positions % block_size


def make_decode_case(name: str, lens: Sequence[int], num_heads: int, num_kv_heads: int,
                     head_dim: int, block_size: int, dtype: str, seed: int,
                     num_blocks: Optional[int] = None, pool_factor: float = 1.25,
                     tables: Optional[np.ndarray] = None) -> DecodeCase:
    """A decode step: every sequence with L > 0 gets one new token at position L-1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = [int(L) for L in lens]
    if tables is None:
        tables, num_blocks = _scatter_tables(rng, lens, block_size, num_blocks, pool_factor)
    else:
        tables = np.asarray(tables, dtype=np.int32)
        assert num_blocks is not None
    live = [s for s, L in enumerate(lens) if L > 0]
    pos = [lens[s] - 1 for s in live]
    slots = _slots_of(tables, live, pos, block_size) if live else np.zeros(0, np.int64)
    refc = np.zeros(num_blocks, dtype=np.int32)
    for s, L in enumerate(lens):
        for j in range(blocks_for(L, block_size)):
            refc[tables[s, j]] += 1
    return DecodeCase(name=name, num_seqs=len(lens), num_heads=num_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                      num_blocks=int(num_blocks), dtype=dtype, scale=1.0 / math.sqrt(head_dim),
                      context_lens=np.asarray(lens, dtype=np.int32), block_tables=tables,
                      slot_mapping=np.asarray(slots, dtype=np.int64),
                      new_token_seq=np.asarray(live, dtype=np.int64),
                      new_token_pos=np.asarray(pos, dtype=np.int64),
                      cow_pairs=np.zeros((0, 2), dtype=np.int64), refcounts=refc, seed=seed)


def make_shared_prefix_case(name: str, num_prompts: int, samples: int, prefix_len: int,
                            max_tail: int, num_heads: int, head_dim: int, block_size: int,
                            dtype: str, seed: int, pool_factor: float = 1.25,
                            num_kv_heads: Optional[int] = None) -> DecodeCase:
    """Parallel sampling: each prompt's prefix blocks are referenced by all its samples.

    The partial last prefix block (if any) is copy-on-write: samples
    0..samples-2 each get a private copy (a (src, dst) pair), the last sample
    keeps the original.  Every sample then grows a tail of U{0..max_tail}
    tokens, written through ``slot_mapping``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    bs = block_size
    full = prefix_len // bs
    partial = prefix_len % bs
    prefix_blocks = blocks_for(prefix_len, bs)
    B = num_prompts * samples
    tails = rng.integers(0, max_tail + 1, size=B)
    lens = [prefix_len + int(t) for t in tails]
    # blocks each sample needs beyond the shared prefix blocks
    own = []
    for s in range(B):
        k = s % samples
        n_after = blocks_for(lens[s], bs) - prefix_blocks
        cow = 1 if (partial and k < samples - 1) else 0
        own.append(cow + n_after)
    total = num_prompts * prefix_blocks + int(sum(own))
    num_blocks = int(math.ceil(pool_factor * total))
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(blocks_for(L, bs) for L in lens)
    tables = np.full((B, mb), -1, dtype=np.int32)
    pairs = []
    at = 0
    for p in range(num_prompts):
        shared = perm[at:at + prefix_blocks]
        at += prefix_blocks
        for k in range(samples):
            s = p * samples + k
            tables[s, :prefix_blocks] = shared
            if partial and k < samples - 1:
                dst = perm[at]
                at += 1
                pairs.append((int(shared[-1]), int(dst)))
                tables[s, prefix_blocks - 1] = dst
            n_after = blocks_for(lens[s], bs) - prefix_blocks
            tables[s, prefix_blocks:prefix_blocks + n_after] = perm[at:at + n_after]
            at += n_after
    seqs, pos = [], []
    for s in range(B):
        for t in range(prefix_len, lens[s]):
            seqs.append(s)
            pos.append(t)
    slots = _slots_of(tables, seqs, pos, bs) if seqs else np.zeros(0, np.int64)
    refc = np.zeros(num_blocks, dtype=np.int32)
    for s in range(B):
        for j in range(blocks_for(lens[s], bs)):
            refc[tables[s, j]] += 1
    return DecodeCase(name=name, num_seqs=B, num_heads=num_heads,
                      num_kv_heads=num_heads if num_kv_heads is None else num_kv_heads,
                      head_dim=head_dim, block_size=bs, num_blocks=num_blocks, dtype=dtype,
                      scale=1.0 / math.sqrt(head_dim),
                      context_lens=np.asarray(lens, dtype=np.int32), block_tables=tables,
                      slot_mapping=np.asarray(slots, dtype=np.int64),
                      new_token_seq=np.asarray(seqs, dtype=np.int64),
                      new_token_pos=np.asarray(pos, dtype=np.int64),
                      cow_pairs=np.asarray(pairs, dtype=np.int64).reshape(-1, 2),
                      refcounts=refc, seed=seed, group_size=samples, shared_blocks=full)


@dataclasses.dataclass
class PrefillCase:
    """One chunked-prefill step: a chunk of C query rows after P cached tokens."""
    name: str
    prefix_len: int
    chunk_len: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    block_table: np.ndarray      # int32 [ceil((P+C)/bs)]
    slot_mapping: np.ndarray     # int64 [C] slots of the chunk's tokens
    seed: int
    tensors: dict = dataclasses.field(default_factory=dict)

    def flops(self) -> int:
        """Algorithmic flops: 2*D for QK and 2*D for PV per visible (row, key, head)."""
        P, C = self.prefix_len, self.chunk_len
        pairs = C * P + C * (C + 1) // 2
        return 4 * self.head_dim * pairs * self.num_heads

    def kv_bytes(self) -> int:
        return (self.prefix_len + self.chunk_len) * 2 * self.num_kv_heads * self.head_dim * 2

    def materialize(self, device="cpu", pool_fill: Optional[float] = None) -> dict:
        """Draw the value tensors on ``device`` (seeded) and return them.

        ``pool_fill`` replaces every slot past position P+C-1 (unowned blocks
        and the tail of the last block) with this constant -- NaN garbage.
        """
        g = torch.Generator(device=device)
        g.manual_seed(self.seed)
        dt = TORCH_DTYPES[self.dtype]
        shape = (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)
        kc = torch.randn(shape, generator=g, device=device, dtype=dt)
        vc = torch.randn(shape, generator=g, device=device, dtype=dt)
        if pool_fill is not None:
            bs, end = self.block_size, self.prefix_len + self.chunk_len
            owned = torch.zeros(self.num_blocks, dtype=torch.bool)
            owned[torch.as_tensor(self.block_table, dtype=torch.long)] = True
            unowned = (~owned).nonzero().flatten().to(device)
            kc[unowned] = pool_fill
            vc[unowned] = pool_fill
            if end % bs:
                blk = int(self.block_table[end // bs])
                kc[blk, :, end % bs:, :] = pool_fill
                vc[blk, :, end % bs:, :] = pool_fill
        C = self.chunk_len
        q = torch.randn((C, self.num_heads, self.head_dim), generator=g, device=device, dtype=dt)
        nk = torch.randn((C, self.num_kv_heads, self.head_dim), generator=g, device=device, dtype=dt)
        nv = torch.randn((C, self.num_kv_heads, self.head_dim), generator=g, device=device, dtype=dt)
        self.tensors = dict(k_cache=kc, v_cache=vc, query=q, new_key=nk, new_value=nv)
        return self.tensors


def make_prefill_case(name: str, prefix_len: int, chunk_len: int, num_heads: int,
                      num_kv_heads: int, head_dim: int, block_size: int, dtype: str, seed: int,
                      pool_factor: float = 1.25) -> PrefillCase:
    rng = np.random.Generator(np.random.PCG64(seed))
    n = blocks_for(prefix_len + chunk_len, block_size)
    num_blocks = max(1, int(math.ceil(pool_factor * n)))
    table = rng.permutation(num_blocks)[:n].astype(np.int32)
    pos = np.arange(prefix_len, prefix_len + chunk_len, dtype=np.int64)
    slots = table[pos // block_size].astype(np.int64) * block_size + pos % block_size
    return PrefillCase(name=name, prefix_len=prefix_len, chunk_len=chunk_len, num_heads=num_heads,
                       num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                       num_blocks=num_blocks, dtype=dtype, scale=1.0 / math.sqrt(head_dim),
                       block_table=table, slot_mapping=slots, seed=seed)


@dataclasses.dataclass
class PrefillBatchCase:
    """Several sequences' prompt chunks in one step, over one shared pool."""
    name: str
    prefix_lens: np.ndarray      # int32 [n]
    chunk_lens: np.ndarray       # int32 [n]
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    block_tables: np.ndarray     # int32 [n][MB], unused = -1
    slot_mapping: np.ndarray     # int64 [sum(chunk_lens)] slots of the chunks' tokens, in row order
    seed: int
    tensors: dict = dataclasses.field(default_factory=dict)

    def flops(self) -> int:
        tot = 0
        for P, C in zip(self.prefix_lens.tolist(), self.chunk_lens.tolist()):
            tot += C * P + C * (C + 1) // 2
        return 4 * self.head_dim * tot * self.num_heads

    def materialize(self, device="cpu") -> dict:
        g = torch.Generator(device=device)
        g.manual_seed(self.seed)
        dt = TORCH_DTYPES[self.dtype]
        shape = (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)
        kc = torch.randn(shape, generator=g, device=device, dtype=dt)
        vc = torch.randn(shape, generator=g, device=device, dtype=dt)
        R = int(self.chunk_lens.sum())
        q = torch.randn((R, self.num_heads, self.head_dim), generator=g, device=device, dtype=dt)
        nk = torch.randn((R, self.num_kv_heads, self.head_dim), generator=g, device=device, dtype=dt)
        nv = torch.randn((R, self.num_kv_heads, self.head_dim), generator=g, device=device, dtype=dt)
        self.tensors = dict(k_cache=kc, v_cache=vc, query=q, new_key=nk, new_value=nv)
        return self.tensors


def make_prefill_batch_case(name: str, prefix_lens, chunk_lens, num_heads: int, num_kv_heads: int,
                            head_dim: int, block_size: int, dtype: str, seed: int,
                            pool_factor: float = 1.25) -> PrefillBatchCase:
    rng = np.random.Generator(np.random.PCG64(seed))
    P = np.asarray(prefix_lens, dtype=np.int32)
    C = np.asarray(chunk_lens, dtype=np.int32)
    need = [blocks_for(int(p + c), block_size) for p, c in zip(P, C)]
    num_blocks = max(1, int(math.ceil(pool_factor * sum(need))))
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(1, max(need))
    tables = np.full((len(P), mb), -1, dtype=np.int32)
    at = 0
    slots = []
    for i, n in enumerate(need):
        tables[i, :n] = perm[at:at + n]
        at += n
        pos = np.arange(P[i], P[i] + C[i], dtype=np.int64)
        slots.append(tables[i][pos // block_size].astype(np.int64) * block_size + pos % block_size)
    return PrefillBatchCase(name=name, prefix_lens=P, chunk_lens=C, num_heads=num_heads,
                            num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                            num_blocks=num_blocks, dtype=dtype, scale=1.0 / math.sqrt(head_dim),
                            block_tables=tables, slot_mapping=np.concatenate(slots) if slots else
                            np.zeros(0, np.int64), seed=seed)


@dataclasses.dataclass
class MixedCase:
    """One continuous-batching step over one pool: prompt chunks of some
    sequences (prefill) and one new token for each of the others (decode)."""
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    context_lens: np.ndarray     # int32 [B] decode sequences, new token included
    decode_tables: np.ndarray    # int32 [B][MB]
    prefix_lens: np.ndarray      # int32 [n] prefill sequences
    chunk_lens: np.ndarray       # int32 [n]
    prefill_tables: np.ndarray   # int32 [n][MB]
    slot_mapping: np.ndarray     # int64 [T]: the decode tokens (live sequences, in order), then the chunks' tokens
    seed: int
    tensors: dict = dataclasses.field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    def decode_bytes(self) -> int:
        el = 2
        kv = int(self.context_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim * el
        q = self.num_seqs * self.num_heads * self.head_dim * el
        tables = sum(blocks_for(int(L), self.block_size) for L in self.context_lens) * 4
        return kv + 2 * q + tables + 4 * self.num_seqs

    def prefill_flops(self) -> int:
        tot = sum(C * P + C * (C + 1) // 2 for P, C in zip(self.prefix_lens.tolist(), self.chunk_lens.tolist()))
        return 4 * self.head_dim * tot * self.num_heads

    def materialize(self, device="cpu", pool_fill: Optional[float] = None) -> dict:
        """``pool_fill`` replaces every pool slot past each sequence's context
        (decode: position L-1; prompt chunk: P+C-1) and every unused block with
        this constant (e.g. NaN: nothing past a context may reach an output)."""
        g = torch.Generator(device=device)
        g.manual_seed(self.seed)
        dt = TORCH_DTYPES[self.dtype]
        Hq, Hkv, D = self.num_heads, self.num_kv_heads, self.head_dim
        kc = torch.randn((self.num_blocks, Hkv, self.block_size, D), generator=g, device=device, dtype=dt)
        vc = torch.randn((self.num_blocks, Hkv, self.block_size, D), generator=g, device=device, dtype=dt)
        if pool_fill is not None:
            bs = self.block_size
            owned = torch.zeros((self.num_blocks, bs), dtype=torch.bool)
            ends = [(self.decode_tables[i], int(L)) for i, L in enumerate(self.context_lens)]
            ends += [(self.prefill_tables[i], int(P + C)) for i, (P, C) in
                     enumerate(zip(self.prefix_lens.tolist(), self.chunk_lens.tolist()))]
            for table, end in ends:
                for j in range(blocks_for(end, bs)):
                    owned[int(table[j]), :min(bs, end - j * bs)] = True
            mask = (~owned).to(device)[:, None, :, None].expand_as(kc)
            kc[mask] = pool_fill
            vc[mask] = pool_fill
        dq = torch.randn((self.num_seqs, Hq, D), generator=g, device=device, dtype=dt)
        pq = torch.randn((int(self.chunk_lens.sum()), Hq, D), generator=g, device=device, dtype=dt)
        T = int(self.slot_mapping.shape[0])
        nk = torch.randn((T, Hkv, D), generator=g, device=device, dtype=dt)
        nv = torch.randn((T, Hkv, D), generator=g, device=device, dtype=dt)
        self.tensors = dict(k_cache=kc, v_cache=vc, decode_query=dq, prefill_query=pq, new_key=nk, new_value=nv)
        return self.tensors


def make_mixed_case(name: str, context_lens, prefix_lens, chunk_lens, num_heads: int, num_kv_heads: int,
                    head_dim: int, block_size: int, dtype: str, seed: int, pool_factor: float = 1.25) -> MixedCase:
    rng = np.random.Generator(np.random.PCG64(seed))
    L = np.asarray(context_lens, dtype=np.int32)
    P = np.asarray(prefix_lens, dtype=np.int32)
    C = np.asarray(chunk_lens, dtype=np.int32)
    tables, num_blocks = _scatter_tables(rng, [int(x) for x in L] + [int(p + c) for p, c in zip(P, C)],
                                         block_size, None, pool_factor)
    dt_, pt_ = tables[:len(L)], tables[len(L):]
    live = [s for s in range(len(L)) if L[s] > 0]
    slots = [_slots_of(dt_, live, [int(L[s]) - 1 for s in live], block_size)]
    for i in range(len(P)):
        pos = np.arange(P[i], P[i] + C[i], dtype=np.int64)
        slots.append(pt_[i][pos // block_size].astype(np.int64) * block_size + pos % block_size)
    return MixedCase(name=name, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                     block_size=block_size, num_blocks=num_blocks, dtype=dtype, scale=1.0 / math.sqrt(head_dim),
                     context_lens=L, decode_tables=dt_, prefix_lens=P, chunk_lens=C, prefill_tables=pt_,
                     slot_mapping=np.concatenate(slots).astype(np.int64), seed=seed)


# ---------------------------------------------------------------- workloads
# The five workloads, named by what they are.  Seeds are 1000 + index.

def tiny_case() -> DecodeCase:
    """4 sequences of {30, 50, 17, 64} tokens, 4/4 heads, D=64, fp16, bs=16, 64 blocks."""
    return make_decode_case("tiny_mha_d64_fp16", [30, 50, 17, 64], num_heads=4, num_kv_heads=4,
                            head_dim=64, block_size=16, dtype="f16", seed=1000, num_blocks=64)


def opt13b_case(seed: int = 1001) -> DecodeCase:
    """OPT-13B-shaped MHA: 64 sequences, L ~ U{128..2048}, 40/40 heads, D=128, fp16."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    lens = rng.integers(128, 2048 + 1, size=64)
    return make_decode_case("opt13b_mha_b64_fp16", lens, num_heads=40, num_kv_heads=40,
                            head_dim=128, block_size=16, dtype="f16", seed=seed)


def llama_gqa_case(seed: int = 1002, num_seqs: int = 256) -> DecodeCase:
    """LLaMA-style GQA: 256 sequences, L ~ U{1..4096}, 32/8 heads, D=128, bf16, bs=16."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    lens = rng.integers(1, 4096 + 1, size=num_seqs)
    return make_decode_case("llama_gqa_b256_bf16", lens, num_heads=32, num_kv_heads=8,
                            head_dim=128, block_size=16, dtype="bf16", seed=seed)


def shared_prefix_case(seed: int = 1003) -> DecodeCase:
    """32 prompts x 8 samples sharing a 1000-token prefix, tails U{0..512}, 40 heads, fp16."""
    return make_shared_prefix_case("shared_prefix_32x8_fp16", num_prompts=32, samples=8,
                                   prefix_len=1000, max_tail=512, num_heads=40, head_dim=128,
                                   block_size=16, dtype="f16", seed=seed)


def long_context_case(block_size: int = 16, seed: int = 1004) -> DecodeCase:
    """8 sequences, L ~ U{32768..131072}, 64/8 heads, D=128, bf16, bs 16 or 32."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    lens = rng.integers(32768, 131072 + 1, size=8)
    return make_decode_case(f"long_context_b8_bs{block_size}_bf16", lens, num_heads=64,
                            num_kv_heads=8, head_dim=128, block_size=block_size, dtype="bf16",
                            seed=seed)


def chunked_prefill_case(seed: int = 1004) -> PrefillCase:
    """One 512-token chunk over an 8192-token paged prefix, 64/8 heads, D=128, bf16."""
    return make_prefill_case("prefill_p8192_c512_bf16", prefix_len=8192, chunk_len=512,
                             num_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
                             dtype="bf16", seed=seed)


def prefill_batch_case(seed: int = 1005) -> PrefillBatchCase:
    """Continuous-batching prefill: 8 prompt chunks of mixed sizes after mixed
    prefixes, LLaMA-style 64/8 heads, bf16, block size 16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chunks = [512, 1024, 256, 2048, 512, 128, 1024, 512]
    prefixes = [int(x) for x in rng.integers(0, 16384, size=len(chunks))]
    return make_prefill_batch_case("prefill_batch8_bf16", prefixes, chunks, 64, 8, 128, 16, "bf16", seed=seed)


def mixed_case(seed: int = 1006) -> MixedCase:
    """A continuous-batching step of a 64/8-head model (D=128, bf16, bs 16):
    one 512-token prompt chunk after an 8192-token prefix, and 256 decoding
    sequences with L ~ U{1..4096}."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    lens = rng.integers(1, 4096 + 1, size=256)
    return make_mixed_case("mixed_p8192_c512_b256_bf16", lens, [8192], [512], 64, 8, 128, 16, "bf16", seed=seed)


def bits(t: torch.Tensor) -> np.ndarray:
    """16-bit element tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
