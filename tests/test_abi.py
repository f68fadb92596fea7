"""The C-ABI library without a GPU: it loads, exports every entry point that include/pa.h
declares, and its host-side argument checks return the documented status codes before any
CUDA work (no kernel is launched by these calls)."""
import ctypes
import re
from pathlib import Path

import pytest

import paged_kv_cache_83_gb300 as pa
from paged_kv_cache_83_gb300 import binding

ROOT = Path(__file__).resolve().parents[1]


def declared_functions():
    text = (ROOT / "include" / "pa.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not binding.LIB_PATH.exists():
        from paged_kv_cache_83_gb300 import build
        build.build()
    return pa.load()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("pa_store_kv", "pa_decode", "pa_store_decode", "pa_prefill_varlen", "pa_decode_workspace_size",
              "pa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value
    assert set(binding.EXPORTS) <= set(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(0) == b"ok"


# A non-null, 16-byte aligned dummy address. Every call below that passes FAKE is built to fail a
# host-side check (or to be an empty no-op), so no kernel ever launches on it.
FAKE = 1 << 20


def test_store_kv_host_checks(lib):
    args = [FAKE, FAKE, FAKE, FAKE, FAKE]
    assert lib.pa_store_kv(*args, 4, 8, 16, 2, 64, 7, None, None) == 3        # dtype
    assert lib.pa_store_kv(*args, -1, 8, 16, 2, 64, 0, None, None) == 2       # T < 0
    assert lib.pa_store_kv(*args, 4, 8, 0, 2, 64, 0, None, None) == 2         # block_size 0
    assert lib.pa_store_kv(*args, 4, 8, 16, 2, 60, 0, None, None) == 4        # D % 8
    assert lib.pa_store_kv(*args, 0, 8, 16, 2, 64, 0, None, None) == 0        # empty: no-op
    assert lib.pa_store_kv(None, FAKE, FAKE, FAKE, FAKE, 4, 8, 16, 2, 64, 0, None, None) == 1
    assert lib.pa_store_kv(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 4, 8, 16, 2, 64, 0, None, None) == 4


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, maxb=4, cl=FAKE, B=2, Hq=4, Hkv=2, D=64,
             bs=16, nb=8, scale=0.125, dt=0, ws=None, wsb=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_decode(*a.values())


def test_decode_host_checks(lib):
    assert _decode(lib, dt=2) == 3
    assert _decode(lib, Hq=5) == 2          # Hq % Hkv
    assert _decode(lib, Hq=18) == 4         # group of 9
    assert _decode(lib, D=96) == 4
    assert _decode(lib, bs=0) == 2
    assert _decode(lib, B=0) == 0           # empty batch: no-op
    assert _decode(lib, q=None) == 1
    assert _decode(lib, bt=None) == 1
    assert _decode(lib, out=FAKE + 8) == 4  # misaligned
    need = lib.pa_decode_workspace_size(2, 4, 2, 64, 4, 16)
    if need:
        assert _decode(lib, ws=None, wsb=0) == 5
        assert _decode(lib, ws=FAKE, wsb=need - 1) == 5


def _prefill(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, cq=FAKE, ck=FAKE, S=2, tq=16, tk=16,
             mq=8, mk=8, bt=FAKE, maxb=2, Hq=4, Hkv=2, D=128, bs=16, nb=8, scale=0.1, causal=1, dt=1,
             err=None, stream=None)
    a.update(kw)
    return lib.pa_prefill_varlen(*a.values())


def test_prefill_host_checks(lib):
    assert _prefill(lib, dt=9) == 3
    assert _prefill(lib, S=-1) == 2
    assert _prefill(lib, causal=2) == 2
    assert _prefill(lib, D=80) == 4
    assert _prefill(lib, S=0) == 0
    assert _prefill(lib, mq=0) == 0
    assert _prefill(lib, kc=None) == 1               # table given, pool missing
    assert _prefill(lib, bt=None, k=None) == 1       # packed keys missing
    assert _prefill(lib, cq=None) == 1
    assert _prefill(lib, bs=0) == 2
    assert _prefill(lib, tq=-1) == 2
    assert _prefill(lib, tq=0) == 0                   # no query rows: no-op


def test_workspace_size_rules(lib):
    assert lib.pa_decode_workspace_size(0, 4, 2, 64, 4, 16) == 0
    assert lib.pa_decode_workspace_size(2, 4, 3, 64, 4, 16) == 0      # invalid heads
    small = lib.pa_decode_workspace_size(2, 4, 2, 64, 4, 16)
    big = lib.pa_decode_workspace_size(2, 4, 2, 64, 400, 16)
    assert big >= small


def _store_decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kn=FAKE, vn=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, maxb=4, cl=FAKE, B=2,
             Hq=4, Hkv=2, D=64, bs=16, nb=8, scale=0.125, dt=0, ws=None, wsb=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_store_decode(*a.values())


def test_store_decode_host_checks(lib):
    assert _store_decode(lib, dt=2) == 3
    assert _store_decode(lib, Hq=5) == 2
    assert _store_decode(lib, D=96) == 4
    assert _store_decode(lib, bs=0) == 2
    assert _store_decode(lib, B=0) == 0           # empty batch: no-op
    assert _store_decode(lib, kn=None) == 1
    assert _store_decode(lib, vc=None) == 1
    assert _store_decode(lib, vn=FAKE + 8) == 4   # misaligned new rows
    need = lib.pa_decode_workspace_size(2, 4, 2, 64, 4, 16)
    if need:
        assert _store_decode(lib, ws=None, wsb=0) == 5


def _store_decode_host(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kn=FAKE, vn=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, maxb=4, cl=FAKE, B=2,
             Hq=4, Hkv=2, D=64, bs=16, nb=8, scale=0.125, dt=0, ws=None, wsb=0, err=None, stream=None)
    a.update(kw)
    return lib.pa_store_decode_host(*a.values())


def test_store_decode_host_entry_checks(lib):
    # every case below returns before the first copy is queued
    assert _store_decode_host(lib, dt=2) == 3
    assert _store_decode_host(lib, Hq=5) == 2
    assert _store_decode_host(lib, D=96) == 4
    assert _store_decode_host(lib, bs=0) == 2
    assert _store_decode_host(lib, B=0) == 0          # empty batch: no-op, nothing copied
    assert _store_decode_host(lib, q=None) == 1
    assert _store_decode_host(lib, out=None) == 1
    assert _store_decode_host(lib, kc=None) == 1
    assert _store_decode_host(lib, bt=None) == 1      # a table width without a table
    assert _store_decode_host(lib, ws=None, wsb=0) == 5
    need = lib.pa_store_decode_host_workspace_size(2, 4, 2, 64, 4, 16)
    assert _store_decode_host(lib, ws=FAKE, wsb=need - 1) == 5
    assert _store_decode_host(lib, ws=FAKE + 128, wsb=need) == 5   # staged regions need 256-byte alignment


def test_store_decode_host_workspace_covers_staging(lib):
    B, Hq, Hkv, D, maxb, bs = 3, 8, 2, 128, 5, 16
    need = lib.pa_store_decode_host_workspace_size(B, Hq, Hkv, D, maxb, bs)
    staged = B * Hq * D * 2 * 2 + B * Hkv * D * 2 * 2 + B * maxb * 4 + B * 4
    assert need >= staged + lib.pa_decode_workspace_size(B, Hq, Hkv, D, maxb, bs)
    assert need % 256 == 0
    assert lib.pa_store_decode_host_workspace_size(0, Hq, Hkv, D, maxb, bs) == 0
    assert lib.pa_store_decode_host_workspace_size(B, 5, Hkv, D, maxb, bs) == 0


def test_store_decode_host_layout(lib):
    B, Hq, Hkv, D, maxb = 5, 16, 8, 128, 7
    offs, n = binding.pa_store_decode_host_layout(B, Hq, Hkv, D, maxb)
    sizes = [B * Hq * D * 2, B * Hkv * D * 2, B * Hkv * D * 2, B * maxb * 4, B * 4]
    assert offs[0] == 0 and all(o % 256 == 0 for o in offs)
    for i in range(4):  # in order, each region clear of the next
        assert offs[i] + sizes[i] <= offs[i + 1]
    assert n == offs[4] + sizes[4]
    assert lib.pa_store_decode_host_layout(B, Hq, Hkv, D, maxb, None) == n
    assert binding.pa_store_decode_host_layout(0, Hq, Hkv, D, maxb) == (None, 0)
    assert binding.pa_store_decode_host_layout(B, 5, Hkv, D, maxb) == (None, 0)


def test_workspace_units_rules(lib):
    """The decode workspace holds one unit per CTA, plus up to eight per CTA of the dynamic tail
    for group sizes up to 3 when the batch has at most 9216 sequences and its table could hold
    enough tiles; the static scheme's size does not depend on the batch."""
    ws = lib.pa_decode_workspace_size
    # group of 8: equal shares only, whatever the batch and table
    assert ws(8, 16, 2, 128, 64, 256) == ws(256, 16, 2, 128, 64, 256) == ws(256, 16, 2, 128, 1, 1)
    # group of 2: a table too narrow for the tail, a wide one, and a batch beyond 9216 sequences
    static = ws(256, 16, 8, 128, 1, 1)
    wide = ws(256, 16, 8, 128, 64, 256)
    assert 8.0 < wide / static < 10.0
    assert ws(10000, 16, 8, 128, 64, 256) == static
    assert ws(9216, 16, 8, 128, 64, 256) == wide
