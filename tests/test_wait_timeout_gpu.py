"""A bounded device wait that runs out: the kernel gives up, reports PA_DEVERR_TIMEOUT and returns,
and the CUDA context stays usable.

The probe (tests/native/wait_probe.cu, a test-only library) compiles the library's own mbarrier
wait and give-up path into a one-warp kernel that waits on an mbarrier nothing arrives on. It
issues no asynchronous copy or MMA, so nothing is in flight when the wait gives up. The library's
kernels are never made to time out.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, DecodeRun, f64, max_abs
from tests.native import build_wait_probe

pytestmark = pytest.mark.gpu

LIMIT_NS = 500_000_000  # the library's wait limit (0.5 s)


@pytest.fixture(scope="module")
def probe():
    lib = ctypes.CDLL(str(build_wait_probe()))
    lib.pa_test_wait_probe.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.pa_test_wait_probe.restype = ctypes.c_int
    return lib


def _run(probe, arrive):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream()
    rc = probe.pa_test_wait_probe(err.data_ptr(), int(arrive), elapsed.data_ptr(), stream.cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    return int(err.item()), int(elapsed.item())


def test_wait_that_completes_reports_nothing(probe):
    err, ns = _run(probe, arrive=True)
    assert err == 0
    assert ns < LIMIT_NS // 10


def test_wait_that_runs_out_sets_timeout_and_returns(probe):
    err, ns = _run(probe, arrive=False)
    assert err == pa.PA_DEVERR_TIMEOUT
    assert LIMIT_NS <= ns < 4 * LIMIT_NS
    # the context is still usable: the probe again, and a decode step against the oracle
    assert _run(probe, arrive=True)[0] == 0
    c = W.make("tiny")
    run = DecodeRun(c)
    out = f64(run.step())
    assert int(run.err.item()) == 0
    orc = oracle.get()
    kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    ref = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=c.dtype)
    assert max_abs(out, ref) <= TOL[c.dtype]
