"""pa_store_kv on the GPU against the oracle's scatter: bit-exact, whole pools compared."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import bits, err_buf, i32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _store_and_compare(orc, k, v, kc, vc, slots, dt):
    dk, dv = to_dev(kc, dt), to_dev(vc, dt)
    err = err_buf()
    pa.pa_store_kv(to_dev(k, dt), to_dev(v, dt), dk, dv, i32(slots), err=err)
    torch.cuda.synchronize()
    rk, rv = orc.store_kv(k, v, kc, vc, slots)
    assert np.array_equal(bits(dk), rk)
    assert np.array_equal(bits(dv), rv)
    return int(err.item())


def test_store_tiny(orc):
    c = W.make("tiny")
    assert _store_and_compare(orc, c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping, c.dtype) == 0


def test_store_prefill_workload_full(orc):
    # the whole prefill_prefix step: ~36k new tokens into a 256-token-block pool
    c = W.make("prefill_prefix")
    assert _store_and_compare(orc, c.k, c.v, c.k_cache, c.v_cache, c.slot_mapping, c.dtype) == 0


@pytest.mark.parametrize("bs,Hkv,D,dt", [(1, 1, 8, "f16"), (3, 2, 64, "bf16"), (16, 14, 64, "f16"),
                                         (256, 8, 128, "bf16"), (5, 3, 24, "f16")])
def test_store_shapes_with_padding(orc, bs, Hkv, D, dt):
    rng = np.random.default_rng([bs, Hkv, D])
    NB = 9
    T = min(NB * bs, 37)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[rng.choice(T, size=T // 4, replace=False)] = -1   # padding tokens are skipped
    k = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    kc = rng.integers(0, 1 << 16, size=(NB, bs, Hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(NB, bs, Hkv, D), dtype=np.uint16)
    assert _store_and_compare(orc, k, v, kc, vc, slots, dt) == 0


def test_store_out_of_range_slot_is_flagged_and_skipped():
    NB, bs, Hkv, D = 4, 4, 2, 64
    kc = torch.zeros(NB, bs, Hkv, D, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones(3, Hkv, D, dtype=torch.float16, device="cuda")
    err = err_buf()
    pa.pa_store_kv(k, k, kc, vc, i32(np.array([0, NB * bs, 5])), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_SLOT
    flat = kc.view(NB * bs, -1)
    assert flat[0].eq(1).all() and flat[5].eq(1).all()
    assert int(flat.ne(0).any(dim=1).sum()) == 2


def test_store_empty_is_noop():
    kc = torch.zeros(2, 4, 1, 64, dtype=torch.bfloat16, device="cuda")
    e = torch.empty(0, 1, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_store_kv(e, e, kc, kc.clone(), torch.empty(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert kc.eq(0).all()
