"""CPU oracle for the paged KV-cache hot path: the plain definition, in fp64.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference leg may import this package. The CUDA library (``paged_kv_cache_83_gb300``)
never imports it, and the two share no code.

Two independent implementations live here:

* ``pa_oracle.c`` (built into ``_build/liboracle.so``, called through ``ctypes``): the naive
  scatter, and paged attention that walks the block table row by row, decodes every 16-bit
  value to double from the format's definition, and takes the softmax in one pass per query
  row. OpenMP spreads (sequence, head) pairs over the host cores.
* ``brute.py``: contiguous attention in numpy fp64 on already-gathered K/V, used to pin the
  C oracle on small inputs.

The C oracle follows the pages' statement of the three operations (see the header of
``pa_oracle.c`` for the passages and the readings taken where they are silent).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from pathlib import Path

import numpy as np

from . import brute  # noqa: F401  (re-exported)

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "pa_oracle.c"
BUILD_DIR = HERE / "_build"
LIB_PATH = BUILD_DIR / "liboracle.so"

F16, BF16 = 0, 1
_DT = {"f16": F16, "bf16": BF16}

ERRORS = {-1: "bad argument", -2: "slot outside the pool or reused", -3: "block table entry out of range",
          -4: "length outside the contract", -5: "out of memory"}


def build(source: Path = SOURCE, out: Path = LIB_PATH, defines: tuple[str, ...] = ()) -> Path:
    """Compile the C oracle with the host compiler (plain -O2, IEEE semantics, OpenMP)."""
    out.parent.mkdir(parents=True, exist_ok=True)
    cc = os.environ.get("CC") or shutil.which("gcc") or "cc"
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = [cc, "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           *[f"-D{d}" for d in defines], str(source), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one build of ``pa_oracle.c``."""

    def __init__(self, path: Path | str = LIB_PATH):
        path = Path(path)
        if path == LIB_PATH and (not path.exists() or path.stat().st_mtime < SOURCE.stat().st_mtime):
            build()
        self.path = path
        lib = ctypes.CDLL(str(path))
        P, I, D_ = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.oracle_store_kv.argtypes = [P, P, P, P, P, I, I, I, I, I]
        lib.oracle_decode.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, D_, I, I]
        lib.oracle_prefill.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, D_, I, I, I]
        lib.oracle_bits_to_double.argtypes = [P, P, ctypes.c_longlong, I]
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = D_
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D_
        lib.oracle_max_threads.restype = I
        for f in (lib.oracle_store_kv, lib.oracle_decode, lib.oracle_prefill):
            f.restype = I
        self.lib = lib

    # --- helpers -------------------------------------------------------------------------
    @staticmethod
    def _p(a: np.ndarray | None):
        return None if a is None else a.ctypes.data

    @staticmethod
    def _check(rc: int, what: str) -> None:
        if rc != 0:
            raise ValueError(f"oracle {what}: {ERRORS.get(rc, rc)}")

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def bits_to_double(self, bits: np.ndarray, dtype: str) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.oracle_bits_to_double(self._p(bits), self._p(out), bits.size, _DT[dtype])
        return out

    # --- the three operations --------------------------------------------------------------
    def store_kv(self, k, v, k_cache, v_cache, slot_mapping):
        """Return copies of the pools after scattering k, v rows to their slots."""
        k = np.ascontiguousarray(k, np.uint16)
        v = np.ascontiguousarray(v, np.uint16)
        kc = np.array(k_cache, dtype=np.uint16, order="C", copy=True)
        vc = np.array(v_cache, dtype=np.uint16, order="C", copy=True)
        sm = np.ascontiguousarray(slot_mapping, np.int32)
        NB, bs, Hkv, D = kc.shape
        T = sm.shape[0]
        assert k.shape == (T, Hkv, D) and v.shape == (T, Hkv, D)
        self._check(self.lib.oracle_store_kv(self._p(k), self._p(v), self._p(kc), self._p(vc),
                                             self._p(sm), T, NB, bs, Hkv, D), "store_kv")
        return kc, vc

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, *, scale: float,
               dtype: str, threads: int = 0) -> np.ndarray:
        """fp64 [B, Hq, D] decode attention output."""
        q = np.ascontiguousarray(q, np.uint16)
        kc = np.ascontiguousarray(k_cache, np.uint16)
        vc = np.ascontiguousarray(v_cache, np.uint16)
        bt = np.ascontiguousarray(block_tables, np.int32)
        cl = np.ascontiguousarray(context_lens, np.int32)
        B, Hq, D = q.shape
        NB, bs, Hkv, D2 = kc.shape
        assert D2 == D and bt.shape[0] == B and cl.shape == (B,)
        out = np.zeros((B, Hq, D), dtype=np.float64)
        self._check(self.lib.oracle_decode(self._p(out), self._p(q), self._p(kc), self._p(vc),
                                           self._p(bt), bt.shape[1], self._p(cl), B, Hq, Hkv, D,
                                           bs, NB, float(scale), _DT[dtype], int(threads)),
                    "decode")
        return out

    def prefill(self, q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, *,
                Hkv: int, block_size: int, scale: float, dtype: str, causal: bool = True,
                threads: int = 0) -> np.ndarray:
        """fp64 [Tq, Hq, D] varlen prefill output. With ``block_tables`` the keys come from the
        pools; without it from the packed ``k``, ``v`` rows indexed by ``cu_seqlens_k``."""
        q = np.ascontiguousarray(q, np.uint16)
        Tq, Hq, D = q.shape
        k = None if k is None else np.ascontiguousarray(k, np.uint16)
        v = None if v is None else np.ascontiguousarray(v, np.uint16)
        kc = None if k_cache is None else np.ascontiguousarray(k_cache, np.uint16)
        vc = None if v_cache is None else np.ascontiguousarray(v_cache, np.uint16)
        cq = np.ascontiguousarray(cu_seqlens_q, np.int32)
        ck = np.ascontiguousarray(cu_seqlens_k, np.int32)
        bt = None if block_tables is None else np.ascontiguousarray(block_tables, np.int32)
        S = cq.shape[0] - 1
        NB = 0 if kc is None else kc.shape[0]
        maxb = 0 if bt is None else bt.shape[1]
        out = np.zeros((Tq, Hq, D), dtype=np.float64)
        self._check(self.lib.oracle_prefill(self._p(out), self._p(q), self._p(k), self._p(v),
                                            self._p(kc), self._p(vc), self._p(cq), self._p(ck),
                                            S, self._p(bt), maxb, Hq, Hkv, D, block_size, NB,
                                            float(scale), int(bool(causal)), _DT[dtype],
                                            int(threads)), "prefill")
        return out


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
