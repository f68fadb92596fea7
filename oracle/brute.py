"""Brute-force contiguous attention in numpy fp64.

TEST INFRASTRUCTURE (see the package docstring): a second, independent statement of scaled
dot-product attention with grouped-query heads, used to pin the paged C oracle on small
inputs. It knows nothing about blocks: callers hand it K and V rows already in sequence order.

Definition (pages: "mini-vLLM", grouped-query attention; prompts attending causally to
themselves; "nano-vLLM Part 4", section 3, prefill and decode rows): for query row r and query
head h, with kv head h // G,

    o[r, h] = softmax_j(scale * q[r, h] . k[j, h // G]) @ v[:, h // G]

over keys j < N, or j <= N - M + r under the causal mask (M query rows are the last M
positions of the N keys).
"""
from __future__ import annotations

import numpy as np


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """fp16 / bf16 storage bits to float64 via numpy's own float types."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
              causal: bool = False) -> np.ndarray:
    """q [M, Hq, D], k and v [N, Hkv, D] (float64) -> o [M, Hq, D]."""
    M, Hq, D = q.shape
    N, Hkv, _ = k.shape
    G = Hq // Hkv
    if N == 0:
        return np.zeros_like(q)
    kk = np.repeat(k, G, axis=1)                       # kv head g serves q heads gG .. gG+G-1
    vv = np.repeat(v, G, axis=1)
    s = np.einsum("mhd,nhd->hmn", q, kk) * scale       # [Hq, M, N]
    if causal:
        allowed = np.arange(N)[None, :] <= (N - M + np.arange(M))[:, None]
        s = np.where(allowed[None], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("hmn,nhd->mhd", p, vv)


def gather_sequence(cache: np.ndarray, table_row: np.ndarray, n: int) -> np.ndarray:
    """Rows 0..n-1 of one sequence from a pool [NB, bs, Hkv, D], in order, via numpy indexing."""
    bs = cache.shape[1]
    pos = np.arange(n)
    return cache[np.asarray(table_row)[pos // bs], pos % bs]
