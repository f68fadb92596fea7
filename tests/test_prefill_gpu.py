"""pa_prefill_varlen on the GPU against the fp64 oracle.

Covers the pool path (prefix cached, block table given, new rows stored first) and the packed
path (no table), causal and not, ragged prompt lengths around the 64/128-row tiles, both
dtypes, D 64/128 and several group sizes; every row of the full prefill_prefix workload.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, bits, err_buf, f64, i32, max_abs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _run_pool(c, causal=True):
    """Store the new rows, then prefill through the block table; returns (out, pools, err)."""
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    err = err_buf()
    pa.pa_store_kv(to_dev(c.k, c.dtype), to_dev(c.v, c.dtype), kc, vc, i32(c.slot_mapping), err=err)
    q = to_dev(c.q, c.dtype)
    out = torch.empty_like(q)
    pa.pa_prefill_varlen(out, q, None, None, kc, vc, i32(c.cu_seqlens_q), i32(c.cu_seqlens_k),
                         c.max_seqlen_q, c.max_seqlen_k, i32(c.block_tables), Hkv=c.Hkv,
                         scale=c.scale, causal=causal, err=err)
    torch.cuda.synchronize()
    return out, kc, vc, err


def _ref_pool(orc, c, causal=True, seqs=None):
    kc, vc = orc.store_kv(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping)
    if seqs is None:
        return orc.prefill(c.q, None, None, kc, vc, c.cu_seqlens_q, c.cu_seqlens_k,
                           c.block_tables, Hkv=c.Hkv, block_size=c.block_size, scale=c.scale,
                           dtype=c.dtype, causal=causal), kc, vc
    outs = []
    for s in seqs:
        a, b = c.cu_seqlens_q[s], c.cu_seqlens_q[s + 1]
        kl = c.cu_seqlens_k[s + 1] - c.cu_seqlens_k[s]
        outs.append(orc.prefill(c.q[a:b], None, None, kc, vc, np.array([0, b - a], np.int32),
                                np.array([0, kl], np.int32), c.block_tables[s:s + 1], Hkv=c.Hkv,
                                block_size=c.block_size, scale=c.scale, dtype=c.dtype,
                                causal=causal))
    return outs, kc, vc


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("P,bs", [(0, 16), (16, 16), (512, 256), (48, 16), (5, 1)])
def test_pool_path(orc, P, bs, causal):
    shared = P % bs == 0
    c = W.prefill_case(q_lens=[1, 63, 64, 65, 130], prefix_len=P, Hq=8, Hkv=4, D=128,
                       block_size=bs, dtype="bf16", shared_prefix=shared, seed=P + bs)
    out, kc, vc, err = _run_pool(c, causal)
    ref, kref, vref = _ref_pool(orc, c, causal)
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    e = max_abs(f64(out), ref)
    assert e <= TOL["bf16"], e
    assert int(err.item()) == 0


@pytest.mark.parametrize("G,D,dt", [(1, 64, "f16"), (2, 128, "f16"), (7, 64, "bf16"),
                                    (4, 128, "bf16"), (8, 64, "f16"), (3, 128, "bf16"),
                                    (5, 64, "f16")])
def test_packed_path(orc, G, D, dt):
    Hkv = 2
    q_lens = [3, 64, 100, 129]
    c = W.prefill_case(q_lens=q_lens, prefix_len=0, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=16,
                       dtype=dt, seed=G)
    q = to_dev(c.q, dt)
    out = torch.empty_like(q)
    err = err_buf()
    pa.pa_prefill_varlen(out, q, to_dev(c.k, dt), to_dev(c.v, dt), None, None,
                         i32(c.cu_seqlens_q), i32(c.cu_seqlens_q), c.max_seqlen_q, c.max_seqlen_q,
                         None, Hkv=Hkv, scale=c.scale, err=err)
    torch.cuda.synchronize()
    ref = orc.prefill(c.q, c.k, c.v, None, None, c.cu_seqlens_q, c.cu_seqlens_q, None, Hkv=Hkv,
                      block_size=16, scale=c.scale, dtype=dt)
    e = max_abs(f64(out), ref)
    assert e <= TOL[dt], e
    assert int(err.item()) == 0


@pytest.mark.parametrize("bs", [16, 4])
def test_pool_path_qwen25_head_shape(orc, bs):
    """The Qwen2.5-0.5B head shape (14 query / 2 kv heads, head dim 64: groups of 7, one pair
    with a single head) with a cached prefix; 16-token blocks take the tcgen05 kernel, 4-token
    blocks the mma.sync one."""
    c = W.prefill_case(q_lens=[1, 63, 64, 65, 130, 257], prefix_len=48, Hq=14, Hkv=2, D=64,
                       block_size=bs, dtype="f16", seed=40 + bs)
    out, kc, vc, err = _run_pool(c)
    ref, kref, vref = _ref_pool(orc, c)
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    e = max_abs(f64(out), ref)
    assert e <= TOL["f16"], e
    assert int(err.item()) == 0


def test_prefix_equals_recompute_on_gpu(orc):
    """The cached-prefix result matches the oracle's full recomputation of prefix + prompt."""
    c = W.prefill_case(q_lens=[40, 90], prefix_len=64, Hq=4, Hkv=2, D=64, block_size=16,
                       dtype="f16", seed=11)
    out, _, _, _ = _run_pool(c)
    kc, vc = orc.store_kv(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping)
    for s in range(2):
        kl = int(c.cu_seqlens_k[s + 1] - c.cu_seqlens_k[s])
        pos = np.arange(kl)
        ks = kc[c.block_tables[s][pos // 16], pos % 16]
        vs = vc[c.block_tables[s][pos // 16], pos % 16]
        a, b = c.cu_seqlens_q[s], c.cu_seqlens_q[s + 1]
        # queries for the prefix rows are irrelevant to the tail rows; use zeros
        qfull = np.concatenate([np.zeros((64, 4, 64), np.uint16), c.q[a:b]])
        full = orc.prefill(qfull, ks, vs, None, None, np.array([0, kl], np.int32),
                           np.array([0, kl], np.int32), None, Hkv=2, block_size=16,
                           scale=c.scale, dtype="f16")
        assert max_abs(f64(out[a:b]), full[64:]) <= TOL["f16"]


def test_bad_lengths_are_flagged_and_zeroed():
    c = W.prefill_case(q_lens=[10, 20], prefix_len=16, Hq=4, Hkv=2, D=64, block_size=16,
                       dtype="f16", seed=12)
    cu_k = c.cu_seqlens_k.copy()
    cu_k[1] = cu_k[0] + 5          # sequence 0: k_len 5 < q_len 10
    kc, vc = to_dev(c.k_cache, "f16"), to_dev(c.v_cache, "f16")
    q = to_dev(c.q, "f16")
    out = torch.full_like(q, 7.0)
    err = err_buf()
    pa.pa_prefill_varlen(out, q, None, None, kc, vc, i32(c.cu_seqlens_q), i32(cu_k),
                         c.max_seqlen_q, c.max_seqlen_k, i32(c.block_tables), Hkv=2,
                         scale=c.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_LENGTH
    assert out[:10].eq(0).all()


def test_empty_is_noop():
    q = torch.empty(0, 4, 64, dtype=torch.float16, device="cuda")
    kv = torch.empty(0, 2, 64, dtype=torch.float16, device="cuda")
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill_varlen(q, q, kv, kv, None, None, cu, cu, 0, 0, None, Hkv=2, scale=0.1)
    torch.cuda.synchronize()


@pytest.fixture(scope="module")
def full_prefill(orc):
    """The prefill_prefix workload (64 prompts, 512-token shared prefix) in the launch
    configuration the bench times: store, then prefill, once on the GPU; the oracle's own scatter
    gives the pools its reference attends over."""
    c = W.make("prefill_prefix")
    out, kc, vc, err = _run_pool(c)
    kref, vref = orc.store_kv(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping)
    return c, f64(out), bits(kc), bits(vc), int(err.item()), kref, vref


def test_full_prefill_workload_store_and_errors(full_prefill):
    c, o, kc, vc, err, kref, vref = full_prefill
    assert err == 0
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)
    assert np.isfinite(o).all()


@pytest.mark.parametrize("part", range(4))
def test_full_prefill_workload_every_prompt(orc, full_prefill, part):
    """Every output row of all 64 prompts against the fp64 oracle, a quarter of the prompts per
    case (the work items go out largest first across the whole launch, so any prompt may be
    split over several CTAs)."""
    c, o, _, _, _, kref, vref = full_prefill
    s0, s1 = 16 * part, 16 * (part + 1)
    a, b = int(c.cu_seqlens_q[s0]), int(c.cu_seqlens_q[s1])
    ka = int(c.cu_seqlens_k[s0])
    ref = orc.prefill(c.q[a:b], None, None, kref, vref, c.cu_seqlens_q[s0:s1 + 1] - a,
                      c.cu_seqlens_k[s0:s1 + 1] - ka, c.block_tables[s0:s1], Hkv=c.Hkv,
                      block_size=c.block_size, scale=c.scale, dtype=c.dtype)
    e = max_abs(o[a:b], ref)
    assert e <= TOL["bf16"], e


@pytest.fixture(scope="module")
def full_qwen25_prefill(orc):
    """The qwen25_prefill workload (the Qwen2.5-0.5B head shape: 64 prompts, 512-token shared
    prefix, 14/2 heads, head dim 64, 16-token blocks, fp16) in the bench's launch configuration."""
    c = W.make("qwen25_prefill")
    out, kc, vc, err = _run_pool(c)
    kref, vref = orc.store_kv(c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping)
    return c, f64(out), bits(kc), bits(vc), int(err.item()), kref, vref


def test_full_qwen25_prefill_store_and_errors(full_qwen25_prefill):
    c, o, kc, vc, err, kref, vref = full_qwen25_prefill
    assert err == 0
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)
    assert np.isfinite(o).all()


@pytest.mark.parametrize("part", range(4))
def test_full_qwen25_prefill_every_prompt(orc, full_qwen25_prefill, part):
    """Every output row of all 64 prompts of the Qwen2.5-shaped prefill against the oracle."""
    c, o, _, _, _, kref, vref = full_qwen25_prefill
    s0, s1 = 16 * part, 16 * (part + 1)
    a, b = int(c.cu_seqlens_q[s0]), int(c.cu_seqlens_q[s1])
    ka = int(c.cu_seqlens_k[s0])
    ref = orc.prefill(c.q[a:b], None, None, kref, vref, c.cu_seqlens_q[s0:s1 + 1] - a,
                      c.cu_seqlens_k[s0:s1 + 1] - ka, c.block_tables[s0:s1], Hkv=c.Hkv,
                      block_size=c.block_size, scale=c.scale, dtype=c.dtype)
    e = max_abs(o[a:b], ref)
    assert e <= TOL["f16"], e


def test_max_seqlen_k_only_orders_the_work(orc):
    """max_seqlen_k sizes the bands of prompts the work goes out in (and nothing else): 0, 1, the
    true bound and a huge value give bit-identical outputs (every item's arithmetic is the same
    whichever CTA takes it), equal to the oracle."""
    c = W.prefill_case(q_lens=[5, 130, 300, 64, 200, 17, 129, 256, 1, 77], prefix_len=256, Hq=16,
                       Hkv=8, D=128, block_size=256, dtype="bf16", seed=77)
    kc, vc = to_dev(c.k_cache, "bf16"), to_dev(c.v_cache, "bf16")
    pa.pa_store_kv(to_dev(c.k, "bf16"), to_dev(c.v, "bf16"), kc, vc, i32(c.slot_mapping))
    q = to_dev(c.q, "bf16")
    outs = []
    for hint in (c.max_seqlen_k, 0, 1, 1 << 30):
        out = torch.empty_like(q)
        err = err_buf()
        pa.pa_prefill_varlen(out, q, None, None, kc, vc, i32(c.cu_seqlens_q), i32(c.cu_seqlens_k),
                             c.max_seqlen_q, hint, i32(c.block_tables), Hkv=c.Hkv, scale=c.scale,
                             err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(bits(out))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    ref, _, _ = _ref_pool(orc, c)
    o = f64(torch.from_numpy(outs[0].view(np.int16)).view(torch.bfloat16))
    assert max_abs(o, ref) <= TOL["bf16"]
