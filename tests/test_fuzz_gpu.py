"""Seeded random shapes against the fp64 oracle: decode (two calls and the fused call) and prefill.

Each case draws a group size 1..8, D 64 or 128, a dtype, a block size (powers of two and odd
sizes), a batch with some empty sequences, and context lengths that land anywhere inside a tile
(64 rows, or 128 on the D = 64 tensor-core path) so partial tiles, the new token's spare row and
boxes of every height meet. Block placement alternates between shuffled and interleaved. The
cases are small enough for the oracle to check every row.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, DecodeRun, bits, err_buf, f64, i32, max_abs, to_dev, workspace

pytestmark = pytest.mark.gpu

BLOCK_SIZES = (1, 2, 3, 4, 5, 8, 16, 24, 32, 64, 128, 256)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _decode_case(seed):
    rng = np.random.default_rng([seed, 77])
    G = int(rng.integers(1, 9))
    Hkv = int(rng.choice([1, 2, 3]))
    D = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    bs = int(rng.choice(BLOCK_SIZES))
    B = int(rng.integers(1, 40))
    lens = rng.integers(1, 700, size=B)
    lens[rng.random(B) < 0.1] = 0
    # some lengths right at a tile edge or one past it
    edge = rng.random(B) < 0.3
    lens[edge] = rng.choice([63, 64, 65, 127, 128, 129, 255, 256, 257], size=int(edge.sum()))
    placement = "interleaved" if seed % 2 else "shuffled"
    return W.decode_case(B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt,
                         context_lens=lens, seed=seed, placement=placement)


@pytest.mark.parametrize("seed", range(48))
def test_decode_random_shapes(orc, seed):
    c = _decode_case(seed)
    kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    ref = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=c.dtype)
    # store, then decode
    run = DecodeRun(c)
    two = run.step().clone()
    assert int(run.err.item()) == 0
    assert np.array_equal(bits(run.kc), kref) and np.array_equal(bits(run.vc), vref)
    assert max_abs(f64(two), ref) <= TOL[c.dtype]
    # the fused call: same pools, the same output bits
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    out = torch.empty_like(run.q)
    err = err_buf()
    pa.pa_store_decode(out, run.q, run.k_new, run.v_new, kc, vc, run.bt, run.cl, c.scale,
                       workspace=workspace(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size),
                       err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    assert torch.equal(out.view(torch.int16), two.view(torch.int16))


def _prefill_case(seed):
    rng = np.random.default_rng([seed, 91])
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 3, 4]))
    D = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    bs = int(rng.choice([1, 4, 16, 64, 128, 256]))
    S = int(rng.integers(1, 7))
    q_lens = rng.integers(1, 300, size=S)
    prefix = rng.integers(0, 400, size=S)
    prefix[rng.random(S) < 0.3] = 0
    return W.prefill_case(q_lens=q_lens, prefix_len=prefix, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                          dtype=dt, seed=seed)


@pytest.mark.parametrize("seed", range(24))
def test_prefill_random_shapes(orc, seed):
    c = _prefill_case(seed)
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    err = err_buf()
    pa.pa_store_kv(to_dev(c.k, c.dtype), to_dev(c.v, c.dtype), kc, vc, i32(c.slot_mapping), err=err)
    q = to_dev(c.q, c.dtype)
    out = torch.empty_like(q)
    pa.pa_prefill_varlen(out, q, None, None, kc, vc, i32(c.cu_seqlens_q), i32(c.cu_seqlens_k),
                         c.max_seqlen_q, c.max_seqlen_k, i32(c.block_tables), Hkv=c.Hkv,
                         scale=c.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kref, vref = orc.store_kv(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    ref = orc.prefill(c.q, None, None, kref, vref, c.cu_seqlens_q, c.cu_seqlens_k, c.block_tables,
                      Hkv=c.Hkv, block_size=c.block_size, scale=c.scale, dtype=c.dtype)
    assert max_abs(f64(out), ref) <= TOL[c.dtype]
