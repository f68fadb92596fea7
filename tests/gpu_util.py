"""Helpers shared by the GPU parity tests: host<->device marshalling and the tolerances."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_83_gb300 as pa

# max-abs tolerance on unit-variance inputs, compared in fp64 against the oracle
TOL = {"f16": 2e-3, "bf16": 1e-2}


def dev():
    return torch.device("cuda:0")


def to_dev(bits: np.ndarray, dt: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev())
    return t.view(torch.float16 if dt == "f16" else torch.bfloat16)


def i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def err_buf() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=dev())


def workspace(B, Hq, Hkv, D, maxb, bs) -> torch.Tensor:
    n = pa.pa_decode_workspace_size(B, Hq, Hkv, D, maxb, bs)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=dev())


class DecodeRun:
    """A decode case resident on the GPU: store then decode, as one layer step."""

    def __init__(self, c):
        self.c = c
        self.kc = to_dev(c.k_cache, c.dtype)
        self.vc = to_dev(c.v_cache, c.dtype)
        self.q = to_dev(c.q, c.dtype)
        self.k_new = to_dev(c.k_new, c.dtype)
        self.v_new = to_dev(c.v_new, c.dtype)
        self.bt = i32(c.block_tables)
        self.cl = i32(c.context_lens)
        self.sm = i32(c.slot_mapping)
        self.ws = workspace(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)
        self.out = torch.empty_like(self.q)
        self.err = err_buf()

    def step(self):
        pa.pa_store_kv(self.k_new, self.v_new, self.kc, self.vc, self.sm, err=self.err)
        pa.pa_decode(self.out, self.q, self.kc, self.vc, self.bt, self.cl, self.c.scale,
                     workspace=self.ws, err=self.err)
        torch.cuda.synchronize()
        return self.out


def max_abs(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.max(np.abs(a - b))) if a.size else 0.0
