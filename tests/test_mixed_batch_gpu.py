"""Mixed prefill + decode batches in one varlen launch.

A decode row is a sequence with one new token whose n - 1 earlier tokens are in the pool, so a
batch that mixes decode rows with prompts (with or without a cached prefix) is one call of
pa_prefill_varlen with a block table, after the store of every new row. (nano-vLLM Part 4 §3
and the smzdm deep dive "调度与内存" run prefill and decode as separate steps; mini-vLLM's
section on batching names the one-token-per-sequence decode row.) The launch is compared with the
fp64 oracle element by element, and its decode rows also with pa_decode on the same pools.
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


def _mixed_case(Hq, Hkv, D, bs, dt, seed):
    rng = np.random.default_rng([seed, 7])
    n_dec = 9
    dec_ctx = rng.integers(1, 1500, size=n_dec)
    # prompts around the 64/128-row tiles, with no, short, block-aligned and long prefixes
    pre_q = [37, 128, 129, 300, 64]
    pre_p = [0, 17, 4 * bs, 700, 1]
    q_lens = np.concatenate([np.ones(n_dec, np.int64), pre_q])
    prefix = np.concatenate([dec_ctx - 1, pre_p])
    order = rng.permutation(len(q_lens))  # decode rows interleaved with the prompts
    c = W.prefill_case(q_lens=q_lens[order], prefix_len=prefix[order], Hq=Hq, Hkv=Hkv, D=D,
                       block_size=bs, dtype=dt, seed=seed)
    return c, np.flatnonzero(q_lens[order] == 1)


@pytest.mark.parametrize("Hq,Hkv,D,bs,dt", [(16, 8, 128, 16, "bf16"), (16, 8, 128, 256, "bf16"),
                                            (14, 2, 64, 16, "f16")])
def test_mixed_launch_matches_oracle_and_decode(orc, Hq, Hkv, D, bs, dt):
    c, dec_rows = _mixed_case(Hq, Hkv, D, bs, dt, seed=Hq + D + bs)
    kc, vc = to_dev(c.k_cache, dt), to_dev(c.v_cache, dt)
    err = err_buf()
    pa.pa_store_kv(to_dev(c.k, dt), to_dev(c.v, dt), kc, vc, i32(c.slot_mapping), err=err)
    q = to_dev(c.q, dt)
    out = torch.empty_like(q)
    bt = i32(c.block_tables)
    pa.pa_prefill_varlen(out, q, None, None, kc, vc, i32(c.cu_seqlens_q), i32(c.cu_seqlens_k),
                         c.max_seqlen_q, c.max_seqlen_k, bt, Hkv=Hkv, scale=c.scale, err=err)
    # the decode rows alone through pa_decode, on the same pools
    rows_q = c.cu_seqlens_q[dec_rows]
    ctx = (c.cu_seqlens_k[dec_rows + 1] - c.cu_seqlens_k[dec_rows]).astype(np.int32)
    qd = q[torch.as_tensor(rows_q, device=q.device, dtype=torch.long)].contiguous()
    outd = torch.empty_like(qd)
    btd = i32(c.block_tables[dec_rows])
    ws = workspace(len(dec_rows), Hq, Hkv, D, c.block_tables.shape[1], bs)
    pa.pa_decode(outd, qd, kc, vc, btd, i32(ctx), c.scale, workspace=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    kref, vref = orc.store_kv(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    ref = orc.prefill(c.q, None, None, kref, vref, c.cu_seqlens_q, c.cu_seqlens_k,
                      c.block_tables, Hkv=Hkv, block_size=bs, scale=c.scale, dtype=dt)
    e = max_abs(f64(out), ref)
    assert e <= TOL[dt], e
    ed = max_abs(f64(outd), ref[rows_q])
    assert ed <= TOL[dt], ed
    # and the decode oracle agrees with the varlen oracle on those rows (same definition)
    refd = orc.decode(c.q[rows_q], kref, vref, c.block_tables[dec_rows], ctx, scale=c.scale,
                      dtype=dt)
    assert max_abs(refd, ref[rows_q]) <= 1e-12
