"""pa_decode_noalloc against pa_decode, through the C ABI, on the GPU.

pa_decode_noalloc serves callers that cannot allocate device memory (a host framework that owns
every allocation, a process whose device memory is already reserved, a step loop that cannot
afford cudaMalloc's synchronisation): its split-K scratch is a fixed device array inside the
library. This file is named so that pytest collects it last.
"""
import pytest
import torch

import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, DecodeRun, f64, max_abs

pytestmark = pytest.mark.gpu


def _case(seed):
    # uses split-K scratch (partials at the SMs' range boundaries) and fits under its limit
    return W.make("qwen3_06b_decode", seed=seed, n=24)


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    for seed in (101, 202):
        c = _case(seed)
        # pa_decode's own workspace also holds the units of its dynamic tail; the no-alloc entry
        # keeps the static split, whose partials for this case fit its fixed scratch
        need = pa.pa_decode_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)
        assert need > 0
        run = DecodeRun(c)
        ref = run.step().clone()                 # store + pa_decode with a caller workspace
        out = torch.full_like(run.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_decode_noalloc(out, run.q, run.kc, run.vc, run.bt, run.cl, c.scale, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
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
