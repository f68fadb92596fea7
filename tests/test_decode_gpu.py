"""pa_decode on the GPU against the fp64 oracle (store first, as one decode layer step).

Every case is compared element by element, the full-size workloads too (the launch
configuration the bench times: 32, 256 and 512 sequences). Tolerance: max-abs 2e-3 (fp16),
1e-2 (bf16), compared in fp64.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, DecodeRun, bits, err_buf, f64, i32, max_abs, to_dev, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _reference(orc, c, kc_bits, vc_bits, rows=None):
    if rows is None:
        return orc.decode(c.q, kc_bits, vc_bits, c.block_tables, c.context_lens, scale=c.scale,
                          dtype=c.dtype)
    return orc.decode(c.q[rows], kc_bits, vc_bits, c.block_tables[rows], c.context_lens[rows],
                      scale=c.scale, dtype=c.dtype)


def _check_full(orc, c):
    run = DecodeRun(c)
    out = f64(run.step())
    kc_ref, vc_ref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(run.kc), kc_ref) and np.array_equal(bits(run.vc), vc_ref)
    ref = _reference(orc, c, kc_ref, vc_ref)
    e = max_abs(out, ref)
    assert e <= TOL[c.dtype], e
    assert int(run.err.item()) == 0
    return e


def test_tiny_config(orc):
    _check_full(orc, W.make("tiny"))


@pytest.mark.parametrize("name,n", [("qwen25_05b_decode", 6), ("qwen3_06b_decode", 5),
                                    ("longtail_decode", 7)])
def test_shrunken_configs_elementwise(orc, name, n):
    _check_full(orc, W.make(name, n=n))


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("D,dt", [(64, "f16"), (128, "bf16")])
def test_group_sizes(orc, G, D, dt):
    Hkv = 2
    lens = [1, 63, 64, 65, 200, 700]
    c = W.decode_case(B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=16, dtype=dt,
                      context_lens=lens, seed=G)
    _check_full(orc, c)


# small groups (fp32 pipes, unswizzled tiles) and large groups (tensor-core fragments, swizzled
# 64-column halves): the block size sets the TMA box height, 1 row up to 64
@pytest.mark.parametrize("Hq,Hkv,D,dt", [(8, 4, 128, "bf16"), (14, 2, 64, "f16"), (16, 2, 128, "bf16")])
@pytest.mark.parametrize("bs", [1, 3, 4, 16, 64, 256])
def test_block_sizes(orc, bs, Hq, Hkv, D, dt):
    lens = [1, 2, bs, bs + 1, 129, 511, 1000]
    c = W.decode_case(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs, dtype=dt,
                      context_lens=lens, seed=bs, placement="interleaved")
    _check_full(orc, c)


@pytest.mark.parametrize("Hq", [4, 14])
def test_zero_context_and_padding_rows(orc, Hq):
    lens = [0, 5, 0, 300]
    c = W.decode_case(B=4, Hq=Hq, Hkv=2, D=64, block_size=16, dtype="f16", context_lens=lens,
                      seed=3, pad_slots=0)
    run = DecodeRun(c)
    out = f64(run.step())
    assert not out[0].any() and not out[2].any()
    kc_ref, vc_ref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert max_abs(out, _reference(orc, c, kc_ref, vc_ref)) <= TOL["f16"]


@pytest.mark.parametrize("Hq,Hkv", [(6, 3), (24, 3)])
def test_single_token_returns_its_value(orc, Hq, Hkv):
    c = W.decode_case(B=3, Hq=Hq, Hkv=Hkv, D=128, block_size=256, dtype="bf16",
                      context_lens=[1, 1, 1], seed=4)
    out = f64(DecodeRun(c).step())
    v = (c.v_new.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    G = Hq // Hkv
    for h in range(Hq):
        assert np.array_equal(out[:, h], v[:, h // G])


def test_max_context(orc):
    # one sequence at the longest context the long-tail workload allows (16384)
    c = W.decode_case(B=2, Hq=16, Hkv=8, D=128, block_size=256, dtype="bf16",
                      context_lens=[16384, 9000], seed=5, placement="interleaved")
    _check_full(orc, c)


def test_batch_equals_alone():
    c = W.make("qwen3_06b_decode", n=6)
    run = DecodeRun(c)
    batched = run.step().clone()
    for i in (0, 3, 5):
        out = torch.empty(1, c.Hq, c.D, dtype=run.q.dtype, device="cuda")
        pa.pa_decode(out, run.q[i:i + 1].contiguous(), run.kc, run.vc, run.bt[i:i + 1].contiguous(),
                     run.cl[i:i + 1].contiguous(), c.scale,
                     workspace=workspace(1, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size))
        torch.cuda.synchronize()
        # the split plan depends on the batch size, so only the summation order may differ
        assert max_abs(f64(out[0]), f64(batched[i])) <= TOL[c.dtype]


@pytest.mark.parametrize("Hq", [4, 14])
def test_invalid_table_entry_is_flagged_and_masked(orc, Hq):
    c = W.decode_case(B=2, Hq=Hq, Hkv=2, D=64, block_size=16, dtype="f16", context_lens=[40, 40],
                      seed=6)
    bt = c.block_tables.copy()
    bt[1, 1] = c.num_blocks + 7          # positions 16..31 of sequence 1 point outside the pool
    run = DecodeRun(c)
    run.bt = i32(bt)
    out = f64(run.step())
    assert int(run.err.item()) & pa.PA_DEVERR_TABLE
    kc_ref, vc_ref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    ref0 = orc.decode(c.q[:1], kc_ref, vc_ref, c.block_tables[:1], c.context_lens[:1],
                      scale=c.scale, dtype=c.dtype)
    assert max_abs(out[:1], ref0) <= TOL["f16"]      # the healthy sequence is untouched
    assert np.isfinite(out[1]).all()


def test_context_longer_than_table_is_flagged_and_zeroed():
    c = W.decode_case(B=2, Hq=4, Hkv=2, D=64, block_size=16, dtype="f16", context_lens=[20, 20],
                      seed=7)
    run = DecodeRun(c)
    run.cl = i32(np.array([20, c.max_blocks_per_seq * 16 + 1]))
    out = f64(run.step())
    assert int(run.err.item()) & pa.PA_DEVERR_LENGTH
    assert not out[1].any()


def test_workspace_too_small_is_refused():
    c = W.make("qwen25_05b_decode", n=4)
    run = DecodeRun(c)
    need = pa.pa_decode_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.pa_decode(run.out, run.q, run.kc, run.vc, run.bt, run.cl, c.scale, workspace=small)
    assert ei.value.status == 5


def test_empty_batch_is_noop():
    q = torch.empty(0, 4, 64, dtype=torch.float16, device="cuda")
    kc = torch.zeros(2, 16, 2, 64, dtype=torch.float16, device="cuda")
    pa.pa_decode(q, q, kc, kc, torch.empty(0, 1, dtype=torch.int32, device="cuda"),
                 torch.empty(0, dtype=torch.int32, device="cuda"), 0.125)
    torch.cuda.synchronize()


def _every_row(orc, c):
    """One launch in the configuration given; every output row against the oracle, which attends
    over the pools its own scatter produced (the GPU's pools must equal them bit for bit)."""
    run = DecodeRun(c)
    out = f64(run.step())
    assert int(run.err.item()) == 0
    kc_ref, vc_ref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(run.kc), kc_ref) and np.array_equal(bits(run.vc), vc_ref)
    ref = _reference(orc, c, kc_ref, vc_ref)
    e = max_abs(out, ref)
    assert e <= TOL[c.dtype], e
    return e


@pytest.mark.parametrize("name", ["qwen25_05b_decode", "qwen3_06b_decode", "longtail_decode"])
def test_full_size_every_row(orc, name):
    """The full-size decode workloads (32, 256 and 512 sequences) in the launch configuration the
    bench times, every sequence and head against the oracle."""
    _every_row(orc, W.make(name))


@pytest.mark.parametrize("G,Hkv,D,bs,dt", [(7, 2, 64, 16, "f16"), (8, 2, 128, 256, "bf16"),
                                           (4, 4, 128, 16, "bf16"), (2, 8, 128, 256, "bf16")])
def test_many_tiles_per_cta_every_row(orc, G, Hkv, D, bs, dt):
    """About a hundred tiles per CTA: the stage ring wraps many times, so every stage passes
    through many barrier phases and, with two producers, each producer's stages alternate with
    the other's. Every row against the oracle; the error word (which a timed-out wait would set)
    stays clear."""
    rng = np.random.default_rng(11)
    lens = rng.integers(100, 4096, size=256, endpoint=True)
    c = W.decode_case(B=256, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt, context_lens=lens,
                      seed=12)
    _every_row(orc, c)


@pytest.mark.parametrize("G,Hkv,D,bs,dt", [(8, 2, 128, 16, "bf16"), (7, 2, 64, 256, "f16")])
def test_batch_larger_than_a_cta_tensor_core_path(orc, G, Hkv, D, bs, dt):
    """More sequences than a CTA has threads (320 on the tensor-core path): the start-up scan
    over the context lengths runs in chunks. Zero-length sequences are mixed in."""
    rng = np.random.default_rng(21)
    lens = rng.integers(1, 600, size=700, endpoint=True)
    lens[rng.choice(700, size=40, replace=False)] = 0
    c = W.decode_case(B=700, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt, context_lens=lens,
                      seed=22)
    run = DecodeRun(c)
    out = f64(run.step())
    assert int(run.err.item()) == 0
    kc_ref, vc_ref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(run.kc), kc_ref) and np.array_equal(bits(run.vc), vc_ref)
    zero = np.flatnonzero(lens == 0)
    assert not out[zero].any()
    assert max_abs(out, _reference(orc, c, kc_ref, vc_ref)) <= TOL[dt]


@pytest.mark.parametrize("G,dt", [(7, "f16"), (4, "bf16")])
def test_two_ctas_per_sm_choice_elementwise(orc, G, dt):
    """D = 64 tensor-core kernels run two CTAs per SM when the table width allows many stages per
    SM (an upper bound: every sequence at the full width). Short real contexts in a wide table
    take that choice while every row stays cheap to check against the oracle; the fused call
    must give the same bits."""
    rng = np.random.default_rng(31)
    lens = rng.integers(1, 300, size=160, endpoint=True)
    c = W.decode_case(B=160, Hq=2 * G, Hkv=2, D=64, block_size=16, dtype=dt, context_lens=lens,
                      seed=32, max_blocks_per_seq=256)
    _check_full(orc, c)
    out, *_ = _fused_step(c)
    run = DecodeRun(c)
    assert torch.equal(out.view(torch.int16), run.step().view(torch.int16))


def _fused_step(c):
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    q = to_dev(c.q, c.dtype)
    out = torch.empty_like(q)
    err = err_buf()
    pa.pa_store_decode(out, q, to_dev(c.k_new, c.dtype), to_dev(c.v_new, c.dtype), kc, vc,
                       i32(c.block_tables), i32(c.context_lens), c.scale,
                       workspace=workspace(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size),
                       err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, kc, vc


@pytest.mark.parametrize("G,Hkv,D,bs,dt,B,lo,hi", [
    (2, 8, 128, 256, "bf16", 64, 2800, 4096),   # one producer, offsets per sequence
    (1, 4, 64, 16, "f16", 240, 1800, 2600),
    (3, 2, 128, 16, "bf16", 280, 2800, 4000),
    (2, 2, 64, 16, "f16", 600, 1200, 2000),     # one producer, offsets per 32 sequences
    (4, 2, 128, 256, "bf16", 128, 2500, 4000),  # tensor-core consumers: equal shares only
    (8, 1, 128, 16, "bf16", 160, 2000, 3000),
    (7, 2, 64, 16, "f16", 256, 1500, 3000),
    (8, 2, 128, 256, "bf16", 700, 600, 1200),
])
def test_dynamic_tail_elementwise(orc, G, Hkv, D, bs, dt, B, lo, hi):
    """Launches of the one-producer kernels (groups up to 3) with enough tiles per CTA split their
    last eighth of tiles into small units that CTAs take from a counter as they finish (beyond one
    CTA's threads of sequences the first tile of every 32nd sequence is kept and a unit's sequence
    is found by one warp-wide read). Unit bounds are closed-form and each unit's arithmetic is the
    same whichever CTA runs it, so the output is checked element by element against the oracle and
    must be bit-identical between the two-call step and the fused call, and between repeated calls;
    the same for the tensor-core kernels at the same sizes, which keep equal shares. Empty
    sequences are mixed in."""
    rng = np.random.default_rng(B + G)
    lens = rng.integers(lo, hi, size=B, endpoint=True)
    lens[rng.choice(B, size=max(1, B // 40), replace=False)] = 0
    c = W.decode_case(B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt, context_lens=lens,
                      seed=B + 7)
    _check_full(orc, c)
    out, kc, vc = _fused_step(c)
    run = DecodeRun(c)
    first = run.step().clone()
    assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    for _ in range(3):  # the same pools again: the store rewrites the same rows
        pa.pa_decode(run.out, run.q, run.kc, run.vc, run.bt, run.cl, c.scale, workspace=run.ws, err=run.err)
        torch.cuda.synchronize()
        assert torch.equal(run.out.view(torch.int16), first.view(torch.int16))
    assert int(run.err.item()) == 0
