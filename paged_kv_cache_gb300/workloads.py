"""Seeded synthetic workloads for paged attention.

This module only *generates inputs*: bf16 Q/K/V rows drawn from N(0, 1),
block tables filled from a shuffled free list, sequence lengths, and initial
pool bytes.  It holds none of the attention arithmetic and none of the cache
addressing: filling the pool is the job of ``pa_write_kv`` (GPU) or of the
oracle's scatter (CPU), so the two sides never share a layout helper.

The five named workloads follow the configurations the library is measured on:

* ``tiny_case``: 1 sequence of 40 tokens, 8 q heads / 2 kv heads, d 64, a pool
  of 16 pages, table = the first 3 entries of a seeded permutation; prefill
  of rows 0..39, then one token written at position 40 and a decode of 41.
* ``llama_prefill_case``: Llama-3.2-1B attention shapes (32/8 heads, d 64), prompts of
  17 and 512 tokens, 2 GiB pool of 65536 pages, table [2][16][128], K/V written
  at layers 0 and 15.
* ``uniform_decode_case``: 64 sequences, lengths uniform in [128, 2048], fragmented pool
  of 65536 pages.
* ``long_prefill_case``: 4 x 8192 causal prefill, (32/8, d 64) or (16/4, d 128), 512
  shuffled pages per sequence from a 65536-page pool.
* ``lognormal_decode_case``: 256 sequences, lengths round(LogNormal(ln 1024, 1.0)) clipped
  to [1, 16384], 4 GiB pool of 131072 pages; c-1 tokens preloaded, then one
  new token written at position c-1 and a decode of length c.

Default seeds: 1000 (tiny), 1001 (Llama prompts), 1002 (64-sequence decode),
1003 (long prefill), 1004 (256-sequence decode).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

TOKENS_PER_PAGE = 16


@dataclass
class Geometry:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_layers: int
    num_slots: int
    max_blocks_per_seq: int
    num_blocks: int

    @property
    def kv_dim(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def page_bytes(self) -> int:
        # K[16][KV_DIM] then V[16][KV_DIM], 2 bytes each
        return 2 * TOKENS_PER_PAGE * self.kv_dim * 2

    @property
    def pool_bytes(self) -> int:
        return self.num_blocks * self.page_bytes

    def as_tuple(self):
        return (self.num_q_heads, self.num_kv_heads, self.head_dim, self.n_layers,
                self.num_slots, self.max_blocks_per_seq, self.num_blocks)


@dataclass
class KVWrite:
    """One ``pa_write_kv`` call: rows k/v [n][KV_DIM] (bf16 bits) to (slot, pos)."""
    layer: int
    tok_slot: np.ndarray
    tok_pos: np.ndarray
    k: np.ndarray
    v: np.ndarray


@dataclass
class Case:
    name: str
    geom: Geometry
    scale: float
    layer: int                       # layer read by the attention call
    slots: np.ndarray                # [B] slot of each sequence
    lens: np.ndarray                 # [B] tokens attended (prefill: prompt length; decode: seq_len)
    block_table: np.ndarray          # [num_slots][n_layers][max_blocks] int32
    writes: List[KVWrite]            # K/V rows to scatter before attending
    q: np.ndarray                    # prefill [T][Hq][d] / decode [B][Hq][d], bf16 bits
    kind: str                        # "prefill" | "decode"
    pool_fill: str = "random"        # initial pool bytes: "random" | "nan" | "zero"
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.lens.shape[0])

    @property
    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.batch + 1, np.int32)
        cu[1:] = np.cumsum(self.lens)
        return cu

    @property
    def total_tokens(self) -> int:
        return int(self.lens.sum())

    @property
    def max_len(self) -> int:
        return int(self.lens.max()) if self.batch else 0


# ------------------------------------------------------------- RoPE tables

def rope_tables(max_pos: int, head_dim: int, base: float = 500000.0):
    """cos / sin tables [max_pos][head_dim/2] fp32 of the usual RoPE angles
    pos * base^(-2i/head_dim) (input data for the RoPE calls; the pages'
    program fills such tables once at start-up and the kernel only reads
    them).  base 500000 is the Llama-3 family's value."""
    half = head_dim // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# ---------------------------------------------------------------- helpers

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, 1) samples rounded to bf16, generated in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


class FreeList:
    """Host page allocator: a list of free physical pages, taken from the back.

    Mirrors the free-list discipline of the pages (pop_back to allocate,
    push_back to release); ``shuffle`` scatters pages across the pool so that
    logically adjacent pages are physically far apart (a fragmented cache).
    """

    def __init__(self, num_blocks: int, rng: Optional[np.random.Generator] = None,
                 shuffle: bool = True):
        ids = np.arange(num_blocks, dtype=np.int64)
        if shuffle and rng is not None:
            rng.shuffle(ids)
        self._free = ids.tolist()

    def pop(self) -> int:
        if not self._free:
            raise MemoryError("page pool exhausted")
        return int(self._free.pop())

    def push(self, blk: int) -> None:
        self._free.append(int(blk))

    def __len__(self):
        return len(self._free)


def empty_table(geom: Geometry) -> np.ndarray:
    return np.full((geom.num_slots, geom.n_layers, geom.max_blocks_per_seq), -1, np.int32)


def assign_pages(table: np.ndarray, free: FreeList, slot: int, layer: int, n_tokens: int) -> None:
    """Gives (slot, layer) a physical page for every logical page of n_tokens."""
    for lb in range((n_tokens + TOKENS_PER_PAGE - 1) // TOKENS_PER_PAGE):
        if table[slot, layer, lb] < 0:
            table[slot, layer, lb] = free.pop()


def release_slot(table: np.ndarray, free: FreeList, slot: int) -> None:
    """Returns every page of a slot (all layers) to the free list, resetting to -1."""
    for layer in range(table.shape[1]):
        for lb in range(table.shape[2]):
            if table[slot, layer, lb] >= 0:
                free.push(int(table[slot, layer, lb]))
                table[slot, layer, lb] = -1


def initial_pool(geom: Geometry, fill: str, seed: int) -> np.ndarray:
    """Pool bytes before any write: random bytes, all-0xFF (bf16 NaN) or zeros."""
    n = geom.pool_bytes
    if fill == "nan":
        return np.full(n, 0xFF, np.uint8)
    if fill == "zero":
        return np.zeros(n, np.uint8)
    rng = np.random.default_rng(seed + 7777)
    return rng.integers(0, 256, n, dtype=np.uint8)


def prompt_writes(geom: Geometry, rng, slots, lens, layers) -> List[KVWrite]:
    """K/V rows for every prompt token, one write call per layer."""
    writes = []
    T = int(np.sum(lens))
    tok_slot = np.repeat(np.asarray(slots, np.int32), lens).astype(np.int32)
    tok_pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lens]) if T else \
        np.zeros(0, np.int32)
    for layer in layers:
        k = normal_bf16(rng, (T, geom.kv_dim))
        v = normal_bf16(rng, (T, geom.kv_dim))
        writes.append(KVWrite(layer, tok_slot, tok_pos, k, v))
    return writes


# ------------------------------------------------------------ generic cases

def make_prefill_case(name, geom: Geometry, lens, seed: int, scale=None, layers=(0,),
                      attend_layer=None, pool_fill="random", slots=None,
                      shuffle_pages=True) -> Case:
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    B = lens.shape[0]
    slots = np.arange(B, dtype=np.int32) if slots is None else np.asarray(slots, np.int32)
    table = empty_table(geom)
    free = FreeList(geom.num_blocks, rng, shuffle=shuffle_pages)
    for layer in layers:
        for b in range(B):
            assign_pages(table, free, int(slots[b]), layer, int(lens[b]))
    writes = prompt_writes(geom, rng, slots, lens, layers)
    q = normal_bf16(rng, (int(lens.sum()), geom.num_q_heads, geom.head_dim))
    scale = 1.0 / np.sqrt(geom.head_dim) if scale is None else scale
    layer = layers[-1] if attend_layer is None else attend_layer
    return Case(name, geom, float(scale), layer, slots, lens, table, writes, q, "prefill",
                pool_fill, seed)


def make_chunked_case(name, geom: Geometry, prefix_lens, chunk_lens, seed: int, scale=None, layer=0,
                      pool_fill="random", slots=None, shuffle_pages=True) -> Case:
    """Prefill of query chunks over a cached prefix: sequence b already holds
    prefix_lens[b] tokens (one write, as an earlier step left them) and then
    scatters its chunk of chunk_lens[b] new tokens (a second write) before the
    attention call; q holds the chunks' rows only.  extra["prefix"] = prefix_lens."""
    rng = np.random.default_rng(seed)
    pre = np.asarray(prefix_lens, np.int32)
    lens = np.asarray(chunk_lens, np.int32)
    B = lens.shape[0]
    slots = np.arange(B, dtype=np.int32) if slots is None else np.asarray(slots, np.int32)
    table = empty_table(geom)
    free = FreeList(geom.num_blocks, rng, shuffle=shuffle_pages)
    for b in range(B):
        assign_pages(table, free, int(slots[b]), layer, int(pre[b] + lens[b]))
    writes = []
    for first, count in ((np.zeros(B, np.int32), pre), (pre, lens)):
        T = int(np.sum(count))
        tok_slot = np.repeat(slots, count).astype(np.int32)
        tok_pos = (np.concatenate([np.arange(f, f + c, dtype=np.int32) for f, c in zip(first, count)])
                   if T else np.zeros(0, np.int32))
        writes.append(KVWrite(layer, tok_slot, tok_pos, normal_bf16(rng, (T, geom.kv_dim)),
                              normal_bf16(rng, (T, geom.kv_dim))))
    q = normal_bf16(rng, (int(lens.sum()), geom.num_q_heads, geom.head_dim))
    scale = 1.0 / np.sqrt(geom.head_dim) if scale is None else scale
    return Case(name, geom, float(scale), layer, slots, lens, table, writes, q, "chunked", pool_fill, seed,
                extra={"prefix": pre})


def make_decode_case(name, geom: Geometry, lens, seed: int, scale=None, layer=0,
                     pool_fill="random", slots=None, shuffle_pages=True,
                     split_last_write=True) -> Case:
    """Decode case: the first len-1 tokens are preloaded, the last one is a
    separate write (the new token), then a decode of length len."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    B = lens.shape[0]
    slots = np.arange(B, dtype=np.int32) if slots is None else np.asarray(slots, np.int32)
    table = empty_table(geom)
    free = FreeList(geom.num_blocks, rng, shuffle=shuffle_pages)
    for b in range(B):
        assign_pages(table, free, int(slots[b]), layer, int(lens[b]))
    if split_last_write:
        pre = np.maximum(lens - 1, 0)
        writes = prompt_writes(geom, rng, slots, pre, [layer])
        has_new = lens > 0
        new_slot = slots[has_new]
        new_pos = (lens[has_new] - 1).astype(np.int32)
        n_new = int(has_new.sum())
        writes.append(KVWrite(layer, new_slot.astype(np.int32), new_pos,
                              normal_bf16(rng, (n_new, geom.kv_dim)),
                              normal_bf16(rng, (n_new, geom.kv_dim))))
    else:
        writes = prompt_writes(geom, rng, slots, lens, [layer])
    q = normal_bf16(rng, (B, geom.num_q_heads, geom.head_dim))
    scale = 1.0 / np.sqrt(geom.head_dim) if scale is None else scale
    return Case(name, geom, float(scale), layer, slots, lens, table, writes, q, "decode",
                pool_fill, seed)


# -------------------------------------------------------- named workloads

def tiny_case(seed: int = 1000, pool_fill: str = "nan"):
    """Returns (prefill_case, decode_case) sharing one table: 40-token prefill,
    then the token at position 40 and a decode of length 41."""
    geom = Geometry(8, 2, 64, 1, 1, 4, 16)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(16).astype(np.int32)
    table = empty_table(geom)
    table[0, 0, :3] = perm[:3]
    lens = np.array([40], np.int32)
    slots = np.array([0], np.int32)
    writes = prompt_writes(geom, rng, slots, lens, [0])
    q = normal_bf16(rng, (40, 8, 64))
    pre = Case("tiny_prefill", geom, 0.125, 0, slots, lens, table, writes, q, "prefill",
               pool_fill, seed)
    new = KVWrite(0, np.array([0], np.int32), np.array([40], np.int32),
                  normal_bf16(rng, (1, geom.kv_dim)), normal_bf16(rng, (1, geom.kv_dim)))
    qd = normal_bf16(rng, (1, 8, 64))
    dec = Case("tiny_decode", geom, 0.125, 0, slots, np.array([41], np.int32), table,
               writes + [new], qd, "decode", pool_fill, seed)
    return pre, dec


def llama_prefill_case(seed: int = 1001, pool_fill: str = "random", attend_layer: int = 15):
    geom = Geometry(32, 8, 64, 16, 2, 128, 65536)
    return make_prefill_case("llama_prefill_case", geom, [17, 512], seed, scale=0.125, layers=(0, 15),
                             attend_layer=attend_layer, pool_fill=pool_fill)


def uniform_decode_lens(seed: int = 1002, batch: int = 64):
    rng = np.random.default_rng(seed)
    return rng.integers(128, 2048, size=batch, endpoint=True).astype(np.int32)


def uniform_decode_case(seed: int = 1002, pool_fill: str = "random", batch: int = 64):
    geom = Geometry(32, 8, 64, 1, batch, 128, 65536)
    return make_decode_case("uniform_decode_case", geom, uniform_decode_lens(seed, batch), seed + 1, scale=0.125,
                            pool_fill=pool_fill)


def long_prefill_geometry(variant: str = "d64") -> Geometry:
    if variant == "d64":
        return Geometry(32, 8, 64, 1, 4, 512, 65536)
    if variant == "d128":
        return Geometry(16, 4, 128, 1, 4, 512, 65536)
    raise ValueError(variant)


def long_prefill_case(variant: str = "d64", seed: int = 1003, pool_fill: str = "random", batch: int = 4,
            seqlen: int = 8192):
    geom = long_prefill_geometry(variant)
    return make_prefill_case("long_prefill_case_" + variant, geom, [seqlen] * batch, seed,
                             scale=1.0 / np.sqrt(geom.head_dim), layers=(0,), pool_fill=pool_fill)


def lognormal_decode_lens(seed: int = 1004, batch: int = 256):
    rng = np.random.default_rng(seed)
    c = np.round(rng.lognormal(mean=np.log(1024.0), sigma=1.0, size=batch))
    return np.clip(c, 1, 16384).astype(np.int32)


def lognormal_decode_case(seed: int = 1004, pool_fill: str = "random", batch: int = 256):
    geom = Geometry(32, 8, 64, 1, batch, 1024, 131072)
    return make_decode_case("lognormal_decode_case", geom, lognormal_decode_lens(seed, batch), seed + 1, scale=0.125,
                            pool_fill=pool_fill)
