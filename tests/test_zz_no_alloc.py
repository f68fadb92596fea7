"""pa_decode_noalloc through the C ABI on the GPU, against the fp64 oracle and against pa_decode.

pa_decode_noalloc serves callers that cannot allocate device memory (a host framework that owns
every allocation, a process whose device memory is already reserved, a step loop that cannot
afford cudaMalloc's synchronisation): its split-K scratch is a fixed device array inside the
library. Its launch differs from pa_decode's (one unit per CTA, no units handed out as CTAs
finish), so it is checked against the oracle itself, on two calls in a row that share the array.
This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, DecodeRun, bits, f64, max_abs

pytestmark = pytest.mark.gpu


def _case(seed):
    # uses split-K scratch (partials at the SMs' range boundaries) and fits under its limit
    return W.make("qwen3_06b_decode", seed=seed, n=24)


def test_noalloc_matches_oracle_and_decode_on_two_calls_in_a_row():
    orc = oracle.get()
    for seed in (101, 202):
        c = _case(seed)
        # pa_decode's own workspace also holds the units of its dynamic tail; the no-alloc entry
        # keeps the static split, whose partials for this case fit its fixed scratch
        need = pa.pa_decode_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)
        assert need > 0
        run = DecodeRun(c)
        ref = run.step().clone()                 # store + pa_decode with a caller workspace
        kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
        assert np.array_equal(bits(run.kc), kref) and np.array_equal(bits(run.vc), vref)
        exact = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale,
                           dtype=c.dtype)
        out = torch.full_like(run.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_decode_noalloc(out, run.q, run.kc, run.vc, run.bt, run.cl, c.scale, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert max_abs(f64(out), exact) <= TOL[c.dtype]
        assert max_abs(f64(out), f64(ref)) <= TOL[c.dtype]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # groups of 8 query heads at D 128 need more partial-result space than the fixed array
    B, Hq, Hkv, D, maxb, bs = 64, 16, 2, 128, 64, 256
    assert pa.pa_decode_workspace_size(B, Hq, Hkv, D, maxb, bs) > pa.PA_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, bs, Hkv, D, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(B, maxb, dtype=torch.int32, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.pa_decode_noalloc(torch.empty_like(q), q, kc, kc, bt, cl, 0.088)
    assert ei.value.status == 5
