"""Decode of short contexts: the one-CTA-per-pair kernel against the oracle and against the
persistent kernel on the same inputs.

pa_decode / pa_store_decode take the short-context kernel when no sequence can hold more than 256
positions (the block table's width times the block size), the persistent split kernel otherwise.
Each case runs both: once with a table exactly 256 positions wide, once with the same table
widened by padding columns (entries never read), and both are compared element by element with
the fp64 oracle ("nano-vLLM Part 4" §3, decode over the cached history through the block table;
"mini-vLLM", grouped-query attention).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, bits, err_buf, f64, i32, max_abs, to_dev, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _fused(c, bt, maxb):
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    q = to_dev(c.q, c.dtype)
    out = torch.empty_like(q)
    err = err_buf()
    ws = workspace(c.B, c.Hq, c.Hkv, c.D, maxb, c.block_size)
    pa.pa_store_decode(out, q, to_dev(c.k_new, c.dtype), to_dev(c.v_new, c.dtype), kc, vc, i32(bt),
                       i32(c.context_lens), c.scale, workspace=ws, err=err)
    torch.cuda.synchronize()
    return f64(out), bits(kc), bits(vc), int(err.item())


@pytest.mark.parametrize("G,Hkv,D,dt,bs", [(1, 4, 128, "bf16", 16), (2, 2, 64, "f16", 16),
                                           (4, 2, 128, "bf16", 16), (7, 2, 64, "f16", 16),
                                           (8, 1, 128, "bf16", 4), (3, 2, 64, "bf16", 1),
                                           (5, 3, 64, "f16", 8)])
def test_short_and_persistent_paths_match_oracle(orc, G, Hkv, D, dt, bs):
    rng = np.random.default_rng([G, D, bs])
    ctx = np.concatenate([[1, 256, 255, 17, 128, 129], rng.integers(1, 257, size=5)])
    c = W.decode_case(B=len(ctx), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt,
                      context_lens=ctx, max_blocks_per_seq=256 // bs, seed=G * 10 + bs)
    kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    ref = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=dt)
    wide = np.concatenate([c.block_tables, np.full((c.B, 8), -1, np.int32)], axis=1)
    for bt in (c.block_tables, wide):  # 256 positions: short kernel; wider: persistent kernel
        o, kc, vc, err = _fused(c, bt, bt.shape[1])
        assert err == 0
        assert np.array_equal(kc, kref) and np.array_equal(vc, vref)
        e = max_abs(o, ref)
        assert e <= TOL[dt], (bt.shape[1], e)


def test_short_path_padding_rows_and_bad_entries(orc):
    """Context 0 rows give zeros; a table entry outside the pool masks its positions and raises
    PA_DEVERR_TABLE; a length beyond the table raises PA_DEVERR_LENGTH and zeroes the row."""
    ctx = np.array([0, 40, 40, 20])
    c = W.decode_case(B=4, Hq=14, Hkv=2, D=64, block_size=16, dtype="f16", context_lens=ctx,
                      max_blocks_per_seq=16, seed=3)
    bt = c.block_tables.copy()
    bt[2, 1] = c.num_blocks + 5  # positions 16..31 of sequence 2
    cl = c.context_lens.copy()
    cl[3] = 16 * 16 + 1          # beyond the table
    kc, vc = to_dev(c.k_cache, "f16"), to_dev(c.v_cache, "f16")
    q = to_dev(c.q, "f16")
    out = torch.full_like(q, 3.0)
    err = err_buf()
    pa.pa_decode(out, q, kc, vc, i32(bt), i32(cl), c.scale,
                 workspace=workspace(4, 14, 2, 64, 16, 16), err=err)
    torch.cuda.synchronize()
    o = f64(out)
    assert int(err.item()) & pa.PA_DEVERR_TABLE and int(err.item()) & pa.PA_DEVERR_LENGTH
    assert not o[0].any() and not o[3].any()
    ref = orc.decode(c.q[1:2], c.k_cache, c.v_cache, c.block_tables[1:2], c.context_lens[1:2],
                     scale=c.scale, dtype="f16")
    assert max_abs(o[1:2], ref) <= TOL["f16"]
    assert np.isfinite(o[2]).all()
