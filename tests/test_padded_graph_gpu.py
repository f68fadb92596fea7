"""Decode batches padded to a fixed size and replayed from one captured CUDA graph.

An engine captures one graph per batch-size bucket and fills unused rows with padding (nano-vLLM
Part 4 §3 on CUDA graphs per batch size; smzdm deep dive "GPU执行优化"). A padding row has
context length 0, slot -1 and a table row of -1: the store skips it, the decode writes zeros for
it, and it costs no KV traffic. The graph of store + decode is captured once for a 64-row bucket
and replayed after different real batches (40, 64 and 1 rows) are copied into its input buffers.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_83_gb300 as pa
import workloads as W
from tests.gpu_util import TOL, bits, err_buf, f64, i32, max_abs, to_dev, workspace

pytestmark = pytest.mark.gpu

BUCKET, NB, BS, MAXB = 64, 4096, 16, 64  # 64 rows x 64 blocks fit the pool


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _batch(n_real, seed, Hq, Hkv, D, DT):
    rng = np.random.default_rng([seed, 5])
    ctx = np.zeros(BUCKET, np.int64)
    ctx[:n_real] = rng.integers(1, MAXB * BS, size=n_real)
    return W.decode_case(B=BUCKET, Hq=Hq, Hkv=Hkv, D=D, block_size=BS, dtype=DT, context_lens=ctx,
                         num_blocks=NB, max_blocks_per_seq=MAXB, seed=seed)


# the fp32 consumers (group 2) and the tensor-core ones (the Qwen2.5 head shape, group 7); the
# step as two calls (store, then decode) and as the fused call
@pytest.mark.parametrize("Hq,Hkv,D,DT", [(16, 8, 128, "bf16"), (14, 2, 64, "f16")])
@pytest.mark.parametrize("fused", [False, True])
def test_padded_bucket_graph_replays(orc, Hq, Hkv, D, DT, fused):
    c0 = _batch(BUCKET, 1, Hq, Hkv, D, DT)
    bufs = {"q": to_dev(c0.q, DT), "kn": to_dev(c0.k_new, DT), "vn": to_dev(c0.v_new, DT),
            "kc": to_dev(c0.k_cache, DT), "vc": to_dev(c0.v_cache, DT),
            "bt": i32(c0.block_tables), "cl": i32(c0.context_lens), "sm": i32(c0.slot_mapping)}
    out = torch.empty_like(bufs["q"])
    ws = workspace(BUCKET, Hq, Hkv, D, MAXB, BS)
    err = err_buf()

    def body():
        if fused:
            pa.pa_store_decode(out, bufs["q"], bufs["kn"], bufs["vn"], bufs["kc"], bufs["vc"],
                               bufs["bt"], bufs["cl"], c0.scale, workspace=ws, err=err)
            return
        pa.pa_store_kv(bufs["kn"], bufs["vn"], bufs["kc"], bufs["vc"], bufs["sm"], err=err)
        pa.pa_decode(out, bufs["q"], bufs["kc"], bufs["vc"], bufs["bt"], bufs["cl"], c0.scale,
                     workspace=ws, err=err)

    body()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()

    for n_real, seed in [(40, 2), (BUCKET, 3), (1, 4), (40, 2)]:
        c = _batch(n_real, seed, Hq, Hkv, D, DT)
        src = {"q": c.q, "kn": c.k_new, "vn": c.v_new, "kc": c.k_cache, "vc": c.v_cache}
        for key, a in src.items():
            bufs[key].copy_(to_dev(a, DT))
        for key, a in (("bt", c.block_tables), ("cl", c.context_lens), ("sm", c.slot_mapping)):
            bufs[key].copy_(i32(a))
        out.fill_(float("nan"))
        err.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
        assert np.array_equal(bits(bufs["kc"]), kref) and np.array_equal(bits(bufs["vc"]), vref)
        o = f64(out)
        ref = orc.decode(c.q[:n_real], kref, vref, c.block_tables[:n_real],
                         c.context_lens[:n_real], scale=c.scale, dtype=DT)
        e = max_abs(o[:n_real], ref)
        assert e <= TOL[DT], (n_real, e)
        assert np.all(o[n_real:] == 0.0), n_real  # padding rows: zeros, not stale values


def test_graph_replays_with_and_without_the_dynamic_tail(orc):
    """A graph replays the same launch parameters (the same launch epoch) every time, while the
    real batch in its buffers changes: replays whose tile count turns the dynamic tail on must get
    a fresh ticket counter each time, and a replay that runs equal shares only must not merge the
    tail records an earlier replay left in the workspace."""
    bucket, maxb, bs, nb, Hq, Hkv, D, DT = 128, 64, 16, 8400, 16, 8, 64, "f16"

    def batch(n_real, seed, lo):
        rng = np.random.default_rng([seed, 9])
        ctx = np.zeros(bucket, np.int64)
        ctx[:n_real] = rng.integers(lo, maxb * bs, size=n_real, endpoint=True)
        return W.decode_case(B=bucket, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, dtype=DT, context_lens=ctx,
                             num_blocks=nb, max_blocks_per_seq=maxb, seed=seed)

    c0 = batch(bucket, 11, 700)
    bufs = {"q": to_dev(c0.q, DT), "kn": to_dev(c0.k_new, DT), "vn": to_dev(c0.v_new, DT),
            "kc": to_dev(c0.k_cache, DT), "vc": to_dev(c0.v_cache, DT),
            "bt": i32(c0.block_tables), "cl": i32(c0.context_lens)}
    out = torch.empty_like(bufs["q"])
    ws = workspace(bucket, Hq, Hkv, D, maxb, bs)
    err = err_buf()

    def body():
        pa.pa_store_decode(out, bufs["q"], bufs["kn"], bufs["vn"], bufs["kc"], bufs["vc"], bufs["bt"],
                           bufs["cl"], c0.scale, workspace=ws, err=err)

    body()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    # full batches of long contexts (about 14 k tiles: the tail runs), then a small batch (equal
    # shares), then full batches again; each replay's choice is read back from the workspace
    for n_real, seed, lo in [(bucket, 12, 700), (16, 13, 1), (bucket, 14, 700), (bucket, 15, 900),
                             (8, 16, 1), (bucket, 12, 700)]:
        c = batch(n_real, seed, lo)
        for key, a in (("q", c.q), ("kn", c.k_new), ("vn", c.v_new), ("kc", c.k_cache), ("vc", c.v_cache)):
            bufs[key].copy_(to_dev(a, DT))
        bufs["bt"].copy_(i32(c.block_tables))
        bufs["cl"].copy_(i32(c.context_lens))
        out.fill_(float("nan"))
        err.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # the replay took the path it was meant to exercise: the kernel's own choice, read back
        tail = pa.pa_decode_debug_tail_units(ws, bucket, Hq, Hkv, D, maxb, bs)
        assert (tail > 0) if n_real == bucket else (tail == 0), (n_real, tail)
        kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
        assert np.array_equal(bits(bufs["kc"]), kref) and np.array_equal(bits(bufs["vc"]), vref)
        o = f64(out)
        ref = orc.decode(c.q[:n_real], kref, vref, c.block_tables[:n_real], c.context_lens[:n_real],
                         scale=c.scale, dtype=DT)
        assert max_abs(o[:n_real], ref) <= TOL[DT]
        assert not o[n_real:].any()  # padding rows are zero
