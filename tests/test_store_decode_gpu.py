"""pa_store_decode (store + decode in one launch) on the GPU.

The fused call must give exactly what pa_store_kv followed by pa_decode gives (nano-vLLM Part 4
§3: each decode step stores the new token's key and value through the slot mapping, then attends
over the cache): the pools bit for bit, the output within the fp tolerance of the fp64 oracle and
bit for bit equal to the two-call path (the same kernel arithmetic reads the same bits).
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


def _fused(c):
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    q = to_dev(c.q, c.dtype)
    out = torch.empty_like(q)
    err = err_buf()
    ws = workspace(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)
    pa.pa_store_decode(out, q, to_dev(c.k_new, c.dtype), to_dev(c.v_new, c.dtype), kc, vc,
                       i32(c.block_tables), i32(c.context_lens), c.scale, workspace=ws, err=err)
    torch.cuda.synchronize()
    return out, kc, vc, err


def _check(orc, c):
    out, kc, vc, err = _fused(c)
    assert int(err.item()) == 0
    kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    ref = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=c.dtype)
    e = max_abs(f64(out), ref)
    assert e <= TOL[c.dtype], e
    two = DecodeRun(c).step()
    assert torch.equal(out.view(torch.int16), two.view(torch.int16))


def test_tiny(orc):
    _check(orc, W.make("tiny"))


@pytest.mark.parametrize("name,n", [("qwen25_05b_decode", 6), ("qwen3_06b_decode", 5),
                                    ("longtail_decode", 7)])
def test_shrunken_configs(orc, name, n):
    _check(orc, W.make(name, n=n))


@pytest.mark.parametrize("G", [1, 2, 4, 7, 8])
@pytest.mark.parametrize("D,dt,bs", [(64, "f16", 16), (128, "bf16", 256), (128, "bf16", 1)])
def test_group_sizes_and_blocks(orc, G, D, dt, bs):
    lens = [1, 63, 64, 65, 200, 700]
    c = W.decode_case(B=len(lens), Hq=G * 2, Hkv=2, D=D, block_size=bs, dtype=dt,
                      context_lens=lens, seed=G + bs)
    _check(orc, c)


def test_padding_rows_store_nothing(orc):
    lens = [0, 300, 0, 17, 0]
    c = W.decode_case(B=len(lens), Hq=8, Hkv=2, D=128, block_size=16, dtype="bf16",
                      context_lens=lens, seed=5)
    _check(orc, c)
    out, _, _, _ = _fused(c)
    assert torch.all(out[torch.tensor(lens, device=out.device) == 0] == 0)


@pytest.mark.parametrize("name", ["qwen25_05b_decode", "qwen3_06b_decode", "longtail_decode"])
def test_full_size_every_row(orc, name):
    """The bench's step (the fused call) on the full-size decode workloads, in their launch
    configuration: pools bit for bit, every output row against the oracle."""
    c = W.make(name)
    out, kc, vc, err = _fused(c)
    assert int(err.item()) == 0
    kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(kc), kref) and np.array_equal(bits(vc), vref)
    ref = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=c.dtype)
    e = max_abs(f64(out), ref)
    assert e <= TOL[c.dtype], e
