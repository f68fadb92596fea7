"""Seeded synthetic inputs for the paged KV-cache hot path.

This module is shared by the tests, the bench and the smoke check. It feeds both the CUDA
library and the CPU oracle, so it holds none of the method's arithmetic: it draws values,
lengths and block placements, and it builds the integer bookkeeping (block tables, slot
mappings, cu_seqlens) that an engine's block manager would hand to the attention layer.

Where the inputs come from (pages: "nano-vLLM Part 4", section 3, the prefill/decode table
and the per-rank tensors list; "mini-vLLM", the paged pool of 16-token blocks):

* a KV pool is a preallocated set of fixed-size token blocks, one pool for K and one for V,
  laid out ``[num_blocks, block_size, Hkv, D]``;
* a block table lists, per sequence, the physical block IDs holding its tokens in order;
  unused entries are -1;
* a slot mapping gives, per new token, its physical slot ``block_id * block_size + offset``;
  -1 marks a padding token that is not stored;
* decode feeds one new token per sequence, at position ``context_len - 1``;
* prefill feeds packed prompts delimited by ``cu_seqlens_q``; with a cached prefix of P
  tokens, ``cu_seqlens_k`` counts ``P + q_len`` keys per sequence.

Values are standard normal draws, rounded once to fp16 or bf16 and handed around as the
raw 16-bit patterns (``uint16``), so both sides start from the same bits.

The five named workloads mirror the five configurations of the paged-decode benchmark:
``tiny``, ``qwen25_05b_decode``, ``qwen3_06b_decode``, ``prefill_prefix`` and
``longtail_decode``. A sixth, ``qwen25_prefill``, is the prefill of the Qwen2.5-0.5B head shape
(14/2 heads, head dim 64, 16-token blocks) with the same prompt mix as ``prefill_prefix``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "DecodeCase", "PrefillCase", "BlockAllocator", "CONFIGS", "normal_bits",
    "decode_case", "prefill_case", "make", "lengths",
]

F16, BF16 = "f16", "bf16"

# ---------------------------------------------------------------------------------------
# Values
# ---------------------------------------------------------------------------------------

_CHUNK = 1 << 23  # elements per generator stream; fixed so a seed gives the same bits anywhere


def _to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 draws once to the storage format; return the raw 16-bit patterns."""
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32)
        # round to nearest, ties to even, on the 16 bits that are dropped (inputs are finite)
        return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def normal_bits(n: int, dtype: str, seed: int, stream: int = 0, threads: int | None = None) -> np.ndarray:
    """``n`` standard normal values as fp16/bf16 bit patterns.

    The array is filled in chunks of ``_CHUNK`` elements, each from its own child of
    ``SeedSequence([seed, stream])``, so the result depends only on (n, dtype, seed, stream)
    and not on the thread count.
    """
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks == 0:
        return out
    children = np.random.SeedSequence([seed, stream]).spawn(nchunks)

    def fill(c: int) -> None:
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.default_rng(children[c])
        out[lo:hi] = _to_bits(g.standard_normal(hi - lo, dtype=np.float32), dtype)

    if threads is None:
        threads = min(os.cpu_count() or 1, 32)
    if nchunks == 1 or threads <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(min(threads, nchunks)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


# ---------------------------------------------------------------------------------------
# Block bookkeeping (a test-side stand-in for an engine's block manager)
# ---------------------------------------------------------------------------------------

class BlockAllocator:
    """Free list of physical block IDs with reference counts.

    The free list starts as a seeded permutation of ``range(num_blocks)`` so that sequences
    land on scattered physical blocks, as they do in a pool that has been in use for a while.
    ``alloc`` pops from the front; ``share`` bumps the count of a block that a second sequence
    reuses (a cached prefix); ``free`` drops a count and returns the block at zero.
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator | None = None):
        self.num_blocks = int(num_blocks)
        order = np.arange(self.num_blocks) if rng is None else rng.permutation(self.num_blocks)
        self.free_list = [int(b) for b in order]
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)

    @property
    def num_free(self) -> int:
        return len(self.free_list)

    def alloc(self, n: int) -> list[int]:
        if n > len(self.free_list):
            raise MemoryError(f"pool exhausted: want {n}, have {len(self.free_list)}")
        ids, self.free_list = self.free_list[:n], self.free_list[n:]
        for b in ids:
            self.refcount[b] = 1
        return ids

    def share(self, ids: list[int]) -> None:
        for b in ids:
            if self.refcount[b] <= 0:
                raise ValueError(f"block {b} is not allocated")
            self.refcount[b] += 1

    def free(self, ids: list[int]) -> None:
        for b in ids:
            if self.refcount[b] <= 0:
                raise ValueError(f"double free of block {b}")
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free_list.append(b)


def _table(rows: list[list[int]], width: int) -> np.ndarray:
    bt = np.full((len(rows), max(width, 1)), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        bt[i, : len(r)] = r
    return bt


def _slot(table_row: np.ndarray, pos: int, block_size: int) -> int:
    return int(table_row[pos // block_size]) * block_size + pos % block_size


# ---------------------------------------------------------------------------------------
# Cases
# ---------------------------------------------------------------------------------------

@dataclass
class DecodeCase:
    """One decode layer-step: store one new K/V row per sequence, then attend over the pool."""
    name: str
    dtype: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    scale: float
    q: np.ndarray             # uint16 [B, Hq, D]
    k_new: np.ndarray         # uint16 [B, Hkv, D]  the step's new key row per sequence
    v_new: np.ndarray         # uint16 [B, Hkv, D]
    k_cache: np.ndarray       # uint16 [num_blocks, block_size, Hkv, D]  before the store
    v_cache: np.ndarray
    block_tables: np.ndarray  # int32 [B, max_blocks_per_seq], -1 padded
    context_lens: np.ndarray  # int32 [B], counts the new token
    slot_mapping: np.ndarray  # int32 [B], slot of position context_len - 1 (-1: not stored)
    seed: int = 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


@dataclass
class PrefillCase:
    """One prefill layer-step: store the prompts' K/V, then varlen causal attention."""
    name: str
    dtype: str
    S: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    scale: float
    prefix_len: int            # -1: a prefix length per sequence (k_lens - q_lens)
    q: np.ndarray              # uint16 [Tq, Hq, D]
    k: np.ndarray              # uint16 [Tq, Hkv, D]  new tokens only
    v: np.ndarray
    k_cache: np.ndarray        # uint16 [num_blocks, block_size, Hkv, D], prefix blocks filled
    v_cache: np.ndarray
    cu_seqlens_q: np.ndarray   # int32 [S+1]
    cu_seqlens_k: np.ndarray   # int32 [S+1]
    block_tables: np.ndarray   # int32 [S, max_blocks_per_seq]
    slot_mapping: np.ndarray   # int32 [Tq]
    refcount: np.ndarray       # int64 [num_blocks]
    seed: int = 0

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)

    @property
    def k_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_k)

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max(initial=0))

    @property
    def max_seqlen_k(self) -> int:
        return int(self.k_lens.max(initial=0))

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def _pool(num_blocks: int, block_size: int, Hkv: int, D: int, dtype: str, seed: int, stream: int):
    n = num_blocks * block_size * Hkv * D
    return normal_bits(n, dtype, seed, stream).reshape(num_blocks, block_size, Hkv, D)


def decode_case(*, B: int, Hq: int, Hkv: int, D: int, block_size: int, dtype: str,
                context_lens, num_blocks: int | None = None, pool_factor: float = 1.25,
                placement: str = "shuffled", max_blocks_per_seq: int | None = None,
                seed: int = 0, name: str = "custom", pad_slots: int = 0) -> DecodeCase:
    """Build a decode step.

    ``placement`` is ``"shuffled"`` (each sequence takes its blocks in turn from a shuffled
    free list), ``"interleaved"`` (sequences grow one block at a time in round-robin order
    from a shuffled free list, so every sequence's blocks are scattered among the others') or
    ``"identity"`` (block IDs handed out in increasing order). ``pad_slots`` > 0 marks that
    many trailing sequences as padding: their new token has slot -1 and is not stored.
    """
    rng = np.random.default_rng([seed, 1])
    ctx = np.asarray(context_lens, dtype=np.int64)
    assert ctx.shape == (B,)
    nblk = [(int(c) + block_size - 1) // block_size for c in ctx]
    total = sum(nblk)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * total))
    alloc = BlockAllocator(num_blocks, None if placement == "identity" else rng)
    rows: list[list[int]] = [[] for _ in range(B)]
    if placement == "interleaved":
        for j in range(max(nblk, default=0)):
            for i in range(B):
                if j < nblk[i]:
                    rows[i] += alloc.alloc(1)
    else:
        for i in range(B):
            rows[i] = alloc.alloc(nblk[i])
    width = max_blocks_per_seq if max_blocks_per_seq is not None else max(max(nblk, default=0), 1)
    bt = _table(rows, width)

    slots = np.full(B, -1, dtype=np.int32)
    for i in range(B - pad_slots):
        if ctx[i] > 0:
            slots[i] = _slot(bt[i], int(ctx[i]) - 1, block_size)

    q = normal_bits(B * Hq * D, dtype, seed, 10).reshape(B, Hq, D)
    k_new = normal_bits(B * Hkv * D, dtype, seed, 11).reshape(B, Hkv, D)
    v_new = normal_bits(B * Hkv * D, dtype, seed, 12).reshape(B, Hkv, D)
    k_cache = _pool(num_blocks, block_size, Hkv, D, dtype, seed, 13)
    v_cache = _pool(num_blocks, block_size, Hkv, D, dtype, seed, 14)
    return DecodeCase(name=name, dtype=dtype, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                      num_blocks=num_blocks, scale=1.0 / math.sqrt(D), q=q, k_new=k_new,
                      v_new=v_new, k_cache=k_cache, v_cache=v_cache, block_tables=bt,
                      context_lens=ctx.astype(np.int32), slot_mapping=slots, seed=seed)


def prefill_case(*, q_lens, prefix_len, Hq: int, Hkv: int, D: int, block_size: int,
                 dtype: str, pool_factor: float = 1.25, num_blocks: int | None = None,
                 shared_prefix: bool = True, seed: int = 0, name: str = "custom") -> PrefillCase:
    """Build a prefill step over packed prompts.

    Every sequence s has ``prefix_len`` tokens already in the pool followed by ``q_lens[s]``
    new tokens. With ``shared_prefix`` the prefix must be whole blocks and all sequences point
    at the same prefix blocks (one allocation, its refcount raised once per extra sharer), the
    way a prefix cache reuses full blocks of a common system prompt. The new tokens' slots
    follow the prefix in each sequence's own blocks. ``prefix_len`` may also be one length per
    sequence (private prefixes): a sequence with one new token and a prefix of n - 1 is a decode
    row of a mixed prefill + decode batch.
    """
    rng = np.random.default_rng([seed, 1])
    ql = np.asarray(q_lens, dtype=np.int64)
    S = int(ql.shape[0])
    per_seq = np.ndim(prefix_len) > 0
    Ps = (np.asarray(prefix_len, dtype=np.int64) if per_seq
          else np.full(S, int(prefix_len), dtype=np.int64))
    if Ps.shape != (S,) or (Ps < 0).any():
        raise ValueError("prefix_len: one non-negative length, or one per sequence")
    if per_seq:
        shared_prefix = False
    P = -1 if per_seq else int(prefix_len)
    if shared_prefix and P % block_size:
        raise ValueError("a shared prefix must be a whole number of blocks")
    kl = ql + Ps
    nblk = [(int(k) + block_size - 1) // block_size for k in kl]
    npre = P // block_size if shared_prefix else 0
    total = (npre + sum(n - npre for n in nblk)) if shared_prefix else sum(nblk)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * total))
    alloc = BlockAllocator(num_blocks, rng)
    prefix_ids = alloc.alloc(npre) if shared_prefix else []
    rows = []
    for s in range(S):
        if shared_prefix:
            if s > 0:
                alloc.share(prefix_ids)
            rows.append(prefix_ids + alloc.alloc(nblk[s] - npre))
        else:
            rows.append(alloc.alloc(nblk[s]))
    bt = _table(rows, max(nblk, default=1))

    cu_q = np.zeros(S + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(ql)
    cu_k = np.zeros(S + 1, dtype=np.int32)
    cu_k[1:] = np.cumsum(kl)
    Tq = int(cu_q[-1])
    slots = np.empty(Tq, dtype=np.int32)
    for s in range(S):
        for r in range(int(ql[s])):
            slots[cu_q[s] + r] = _slot(bt[s], int(Ps[s]) + r, block_size)

    q = normal_bits(Tq * Hq * D, dtype, seed, 20).reshape(Tq, Hq, D)
    k = normal_bits(Tq * Hkv * D, dtype, seed, 21).reshape(Tq, Hkv, D)
    v = normal_bits(Tq * Hkv * D, dtype, seed, 22).reshape(Tq, Hkv, D)
    k_cache = _pool(num_blocks, block_size, Hkv, D, dtype, seed, 23)
    v_cache = _pool(num_blocks, block_size, Hkv, D, dtype, seed, 24)
    return PrefillCase(name=name, dtype=dtype, S=S, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                       num_blocks=num_blocks, scale=1.0 / math.sqrt(D), prefix_len=P, q=q, k=k,
                       v=v, k_cache=k_cache, v_cache=v_cache, cu_seqlens_q=cu_q,
                       cu_seqlens_k=cu_k, block_tables=bt, slot_mapping=slots,
                       refcount=alloc.refcount.copy(), seed=seed)


# ---------------------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "decode" | "prefill"
    title: str
    seed: int
    params: dict = field(default_factory=dict)


CONFIGS: dict[str, Workload] = {
    "tiny": Workload(
        "tiny", "decode",
        "Tiny paged decode + store: 4 seqs, ctx {1,17,100,255}, 4/2 heads, D 64, bs 16, "
        "64-block pool, fp16", 0,
        dict(B=4, Hq=4, Hkv=2, D=64, block_size=16, dtype=F16, num_blocks=64)),
    "qwen25_05b_decode": Workload(
        "qwen25_05b_decode", "decode",
        "Qwen2.5-0.5B-shaped decode: 32 seqs, ctx U[128,2048], 14/2 heads, D 64, bs 16, fp16", 1,
        dict(B=32, Hq=14, Hkv=2, D=64, block_size=16, dtype=F16, pool_factor=1.25)),
    "qwen3_06b_decode": Workload(
        "qwen3_06b_decode", "decode",
        "Qwen3-0.6B-shaped decode: 256 seqs, ctx U[100,4096], 16/8 heads, D 128, bs 256, bf16", 2,
        dict(B=256, Hq=16, Hkv=8, D=128, block_size=256, dtype=BF16, pool_factor=1.25)),
    "prefill_prefix": Workload(
        "prefill_prefix", "prefill",
        "Varlen causal prefill, 64 prompts q U[100,1024], shared 512-token cached prefix, "
        "16/8 heads, D 128, bs 256, bf16", 3,
        dict(S=64, prefix_len=512, Hq=16, Hkv=8, D=128, block_size=256, dtype=BF16)),
    "qwen25_prefill": Workload(
        "qwen25_prefill", "prefill",
        "Qwen2.5-0.5B-shaped varlen causal prefill: 64 prompts q U[100,1024], shared 512-token "
        "cached prefix, 14/2 heads, D 64, bs 16, fp16", 5,
        dict(S=64, prefix_len=512, Hq=14, Hkv=2, D=64, block_size=16, dtype=F16)),
    "longtail_decode": Workload(
        "longtail_decode", "decode",
        "Max-batch long-tail decode: 512 seqs, ctx lognormal(median 2048, sigma 1) clipped "
        "to [1,16384], 16/8 heads, D 128, bs 256, bf16, pool 95% full, interleaved placement", 4,
        dict(B=512, Hq=16, Hkv=8, D=128, block_size=256, dtype=BF16)),
}


def _lengths(name: str, seed: int, n: int | None = None) -> np.ndarray:
    rng = np.random.default_rng([seed, 0])
    if name == "tiny":
        return np.array([1, 17, 100, 255], dtype=np.int64)
    if name == "qwen25_05b_decode":
        return rng.integers(128, 2048, size=n or 32, endpoint=True)
    if name == "qwen3_06b_decode":
        return rng.integers(100, 4096, size=n or 256, endpoint=True)
    if name in ("prefill_prefix", "qwen25_prefill"):
        return rng.integers(100, 1024, size=n or 64, endpoint=True)
    if name == "longtail_decode":
        x = rng.lognormal(mean=math.log(2048.0), sigma=1.0, size=n or 512)
        return np.clip(np.rint(x), 1, 16384).astype(np.int64)
    raise KeyError(name)


def lengths(name: str, seed: int | None = None, n: int | None = None) -> np.ndarray:
    """The per-sequence lengths (contexts, or prompt lengths) of a named workload, without
    building its pools: what ``make(name, seed, n)`` would use."""
    return _lengths(name, CONFIGS[name].seed if seed is None else seed, n)


def make(name: str, seed: int | None = None, n: int | None = None):
    """Build one of the five named workloads (``n`` overrides the sequence count)."""
    w = CONFIGS[name]
    seed = w.seed if seed is None else seed
    p = dict(w.params)
    lens = _lengths(name, seed, n)
    if w.kind == "prefill":
        p.pop("S", None)
        return prefill_case(q_lens=lens, seed=seed, name=name, **p)
    p["B"] = len(lens)
    if name == "longtail_decode":
        bs = p["block_size"]
        need = int(sum((int(c) + bs - 1) // bs for c in lens))
        p["num_blocks"] = math.ceil(need / 0.95)
        return decode_case(context_lens=lens, seed=seed, name=name, placement="interleaved",
                           max_blocks_per_seq=16384 // bs, **p)
    if name == "qwen3_06b_decode":
        return decode_case(context_lens=lens, seed=seed, name=name,
                           max_blocks_per_seq=4096 // p["block_size"], **p)
    if name == "qwen25_05b_decode":
        return decode_case(context_lens=lens, seed=seed, name=name,
                           max_blocks_per_seq=2048 // p["block_size"], **p)
    return decode_case(context_lens=lens, seed=seed, name=name, **p)
