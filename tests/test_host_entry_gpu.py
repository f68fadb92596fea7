"""pa_store_decode_host: the decode layer step with its inputs and output in host memory.

The library stages q, the new K/V rows, the block tables and the context lengths into its
workspace, runs the fused store + decode on the device pools and copies the output back, all on
one stream. The pools it leaves and the output it returns must be bit-identical to the device
call's, and both must match the fp64 oracle within the decode tolerance.
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


def _host(bits_arr, dt, pin):
    t = torch.from_numpy(np.ascontiguousarray(bits_arr).view(np.int16).copy())
    t = t.view(torch.float16 if dt == "f16" else torch.bfloat16)
    return t.pin_memory() if pin else t


def _host_i32(a, pin):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32).copy())
    return t.pin_memory() if pin else t


def _host_step(c, pin, stream=None):
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    q = _host(c.q, c.dtype, pin)
    out = torch.empty(q.shape, dtype=q.dtype)
    out = out.pin_memory() if pin else out
    n = pa.pa_store_decode_host_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq,
                                               c.block_size)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda:0")
    err = err_buf()
    pa.pa_store_decode_host(out, q, _host(c.k_new, c.dtype, pin), _host(c.v_new, c.dtype, pin), kc, vc,
                            _host_i32(c.block_tables, pin), _host_i32(c.context_lens, pin), c.scale,
                            workspace=ws, err=err, stream=stream)
    if stream is None:
        torch.cuda.current_stream().synchronize()
    else:
        stream.synchronize()
    assert int(err.item()) == 0
    return out, kc, vc


def _device_step(c):
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


SHAPES = [  # (G, Hkv, D, block size, dtype): fp32 consumers, both tensor-core widths, odd blocks
    (2, 8, 128, 256, "bf16"),
    (7, 2, 64, 16, "f16"),
    (8, 2, 128, 64, "bf16"),
    (1, 3, 64, 5, "f16"),
]


@pytest.mark.parametrize("G,Hkv,D,bs,dt", SHAPES)
@pytest.mark.parametrize("pin", [True, False])
def test_host_entry_matches_device_call_and_oracle(orc, G, Hkv, D, bs, dt, pin):
    rng = np.random.default_rng([G, D, bs])
    lens = rng.integers(0, 600, size=23)
    lens[3] = 0
    lens[5] = 1
    c = W.decode_case(B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt,
                      context_lens=lens, seed=int(G * 100 + D + bs))
    out_h, kc_h, vc_h = _host_step(c, pin)
    out_d, kc_d, vc_d = _device_step(c)
    assert torch.equal(kc_h.view(torch.int16), kc_d.view(torch.int16))
    assert torch.equal(vc_h.view(torch.int16), vc_d.view(torch.int16))
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
    kref, vref = orc.store_kv(c.k_new, c.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(kc_h), kref) and np.array_equal(bits(vc_h), vref)
    ref = orc.decode(c.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=c.dtype)
    assert max_abs(f64(out_h), ref) <= TOL[c.dtype]


def _packed_inputs(c, pin=True):
    """The five inputs as views of one host buffer at the library's packed offsets."""
    offs, n = pa.pa_store_decode_host_layout(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq)
    buf = torch.zeros(n, dtype=torch.uint8)
    buf = buf.pin_memory() if pin else buf
    views = []
    for o, arr, dt in zip(offs, (c.q, c.k_new, c.v_new, c.block_tables, c.context_lens),
                          (c.dtype, c.dtype, c.dtype, "i32", "i32")):
        src = (_host_i32(arr, False) if dt == "i32" else _host(arr, dt, False))
        nb = src.numel() * src.element_size()
        v = buf[o:o + nb].view(src.dtype).view(src.shape)
        v.copy_(src)
        views.append(v)
    return views


@pytest.mark.parametrize("G,Hkv,D,bs,dt", SHAPES[:2])
@pytest.mark.parametrize("pin", [True, False])
def test_host_entry_packed_inputs(orc, G, Hkv, D, bs, dt, pin):
    """Packed inputs move in one transfer: pulled by a kernel when the buffer is page-locked and
    mapped, by the copy engine when it is pageable. Either way the same bits as the device call;
    repeated steps with new inputs in the same buffers must not see the previous step's bytes."""
    lens = np.random.default_rng(G + D).integers(0, 900, size=37)
    c = W.decode_case(B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt,
                      context_lens=lens, seed=3 + G)
    q, kn, vn, bt, cl = _packed_inputs(c, pin)
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    out = torch.empty(q.shape, dtype=q.dtype)
    out = out.pin_memory() if pin else out
    n = pa.pa_store_decode_host_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda:0")
    err = err_buf()
    pa.pa_store_decode_host(out, q, kn, vn, kc, vc, bt, cl, c.scale, workspace=ws, err=err)
    torch.cuda.current_stream().synchronize()
    assert int(err.item()) == 0
    out_d, kc_d, vc_d = _device_step(c)
    assert torch.equal(out.view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc_d.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc_d.view(torch.int16))
    # a second step through the same host buffers with new query rows and new K/V rows
    c2 = W.decode_case(B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, dtype=dt,
                       context_lens=lens, seed=50 + G)
    q.copy_(_host(c2.q, dt, False))
    kn.copy_(_host(c2.k_new, dt, False))
    vn.copy_(_host(c2.v_new, dt, False))
    kc2, vc2 = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    pa.pa_store_decode_host(out, q, kn, vn, kc2, vc2, bt, cl, c.scale, workspace=ws, err=err)
    torch.cuda.current_stream().synchronize()
    assert int(err.item()) == 0
    kref, vref = orc.store_kv(c2.k_new, c2.v_new, c.k_cache, c.v_cache, c.slot_mapping)
    assert np.array_equal(bits(kc2), kref) and np.array_equal(bits(vc2), vref)
    ref = orc.decode(c2.q, kref, vref, c.block_tables, c.context_lens, scale=c.scale, dtype=dt)
    assert max_abs(f64(out), ref) <= TOL[dt]


def test_host_entry_on_a_side_stream(orc):
    c = W.decode_case(B=9, Hq=16, Hkv=2, D=128, block_size=16, dtype="bf16",
                      context_lens=[0, 1, 15, 16, 17, 300, 64, 65, 1000], seed=5)
    s = torch.cuda.Stream()
    out_h, kc_h, _ = _host_step(c, True, stream=s)
    out_d, kc_d, _ = _device_step(c)
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(kc_h.view(torch.int16), kc_d.view(torch.int16))


def test_host_entry_rejects_device_tensors():
    c = W.decode_case(B=2, Hq=4, Hkv=2, D=64, block_size=16, dtype="f16", context_lens=[3, 4], seed=1)
    kc, vc = to_dev(c.k_cache, c.dtype), to_dev(c.v_cache, c.dtype)
    q = to_dev(c.q, c.dtype)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(ValueError):
        pa.pa_store_decode_host(torch.empty_like(q), q, to_dev(c.k_new, c.dtype), to_dev(c.v_new, c.dtype),
                                kc, vc, i32(c.block_tables), i32(c.context_lens), c.scale, workspace=ws)
