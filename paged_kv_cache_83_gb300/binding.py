"""Python binding of the C ABI in ``include/pa.h`` (argument marshalling only).

Each function takes torch CUDA tensors, checks their dtype / shape / contiguity, and calls the
entry point of the same name in ``_build/libpagedattn.so`` with raw device pointers and the
current CUDA stream. Every step of the computation runs in the library's kernels; there is no
fallback: if the library is missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "_build" / "libpagedattn.so"

PA_F16, PA_BF16 = 0, 1
PA_DEVERR_SLOT, PA_DEVERR_TABLE, PA_DEVERR_LENGTH, PA_DEVERR_TIMEOUT = 1, 2, 4, 8
EXPORTS = ("pa_store_kv", "pa_decode_workspace_size", "pa_decode", "pa_store_decode",
           "pa_store_decode_host", "pa_store_decode_host_workspace_size", "pa_store_decode_host_layout",
           "pa_prefill_varlen", "pa_decode_noalloc", "pa_decode_debug_tail_units", "pa_status_string", "pa_bm_create",
           "pa_bm_destroy", "pa_bm_allocate", "pa_bm_can_allocate", "pa_bm_append",
           "pa_bm_release", "pa_bm_block_table", "pa_bm_num_tokens", "pa_bm_num_free",
           "pa_bm_refcount")
PA_DECODE_NOALLOC_SCRATCH_BYTES = 1 << 20

_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")
        self.status = status


def load(path: Path | str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = Path(path)
    if not path.exists():
        raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_83_gb300.build.build()")
    lib = ctypes.CDLL(str(path))
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pa_store_kv.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.pa_store_kv.restype = I
    lib.pa_decode_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.pa_decode_workspace_size.restype = Z
    lib.pa_decode.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, P, Z, P, P]
    lib.pa_decode.restype = I
    lib.pa_store_decode.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, P, Z, P, P]
    lib.pa_store_decode.restype = I
    lib.pa_store_decode_host.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, P, Z, P, P]
    lib.pa_store_decode_host.restype = I
    lib.pa_store_decode_host_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.pa_store_decode_host_workspace_size.restype = Z
    lib.pa_store_decode_host_layout.argtypes = [I, I, I, I, I, P]
    lib.pa_store_decode_host_layout.restype = Z
    lib.pa_prefill_varlen.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, I, I, I, I, I, I,
                                      F, I, I, P, P]
    lib.pa_prefill_varlen.restype = I
    lib.pa_decode_noalloc.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, P, P]
    lib.pa_decode_noalloc.restype = I
    lib.pa_decode_debug_tail_units.argtypes = [P, I, I, I, I, I, I]
    lib.pa_decode_debug_tail_units.restype = I
    L = ctypes.c_int64
    lib.pa_bm_create.argtypes = [I, I, I]
    lib.pa_bm_create.restype = P
    lib.pa_bm_destroy.argtypes = [P]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_allocate.argtypes = [P, L, P, I]
    lib.pa_bm_allocate.restype = I
    lib.pa_bm_can_allocate.argtypes = [P, P, I]
    lib.pa_bm_can_allocate.restype = I
    lib.pa_bm_append.argtypes = [P, L, ctypes.c_int32]
    lib.pa_bm_append.restype = L
    lib.pa_bm_release.argtypes = [P, L]
    lib.pa_bm_release.restype = I
    lib.pa_bm_block_table.argtypes = [P, L, P, I]
    lib.pa_bm_block_table.restype = I
    lib.pa_bm_num_tokens.argtypes = [P, L]
    lib.pa_bm_num_tokens.restype = I
    lib.pa_bm_num_free.argtypes = [P]
    lib.pa_bm_num_free.restype = I
    lib.pa_bm_refcount.argtypes = [P, I]
    lib.pa_bm_refcount.restype = I
    lib.pa_status_string.argtypes = [I]
    lib.pa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def pa_decode_debug_tail_units(workspace, B: int, Hq: int, Hkv: int, D: int,
                               max_blocks_per_seq: int, block_size: int) -> int:
    """Diagnostics: the dynamic-tail units the last completed pa_decode / pa_store_decode launch on
    this workspace ran (0: equal shares only); -1 on invalid sizes or a failed read."""
    return int(load().pa_decode_debug_tail_units(_ptr(workspace), int(B), int(Hq), int(Hkv), int(D),
                                                 int(max_blocks_per_seq), int(block_size)))


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _i32(t: torch.Tensor | None, name: str):
    if t is not None and t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _ptr(t)


def _stream(stream, ref: torch.Tensor) -> int | None:
    """The raw stream handle: the given stream, else the current stream of ref's device (read
    straight from torch's stream registry: building a torch Stream object costs ~3 us a call)."""
    if stream is None:
        return torch._C._cuda_getCurrentRawStream(ref.get_device())
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise PagedAttnError(fn, status)


def pa_store_kv(k, v, k_cache, v_cache, slot_mapping, err=None, stream=None) -> None:
    """Scatter k, v [T, Hkv, D] into k_cache, v_cache [NB, bs, Hkv, D] at slot_mapping [T]."""
    NB, bs, Hkv, D = k_cache.shape
    T = k.shape[0]
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [T]")
    dt = _dtype(k_cache)
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("k, v and the pools must share a dtype")
    _check("pa_store_kv", load().pa_store_kv(
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _i32(slot_mapping, "slot_mapping"), T, NB,
        bs, Hkv, D, dt, _i32(err, "err"), _stream(stream, k)))


def pa_decode_workspace_size(B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                             block_size: int) -> int:
    """Bytes of scratch pa_decode needs on the current device for these sizes."""
    return int(load().pa_decode_workspace_size(B, Hq, Hkv, D, max_blocks_per_seq, block_size))


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
              workspace=None, err=None, stream=None) -> None:
    """Paged GQA decode: out [B, Hq, D] from q [B, Hq, D] over the pools."""
    NB, bs, Hkv, D = k_cache.shape
    B, Hq, Dq = q.shape
    if Dq != D or tuple(out.shape) != (B, Hq, D) or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch")
    dt = _dtype(q)
    if out.dtype != q.dtype or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q, out and the pools must share a dtype")
    maxb = block_tables.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode", load().pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _i32(block_tables, "block_tables"), maxb,
        _i32(context_lens, "context_lens"), B, Hq, Hkv, D, bs, NB, float(scale), dt,
        _ptr(workspace), ws_bytes, _i32(err, "err"), _stream(stream, q)))


def pa_store_decode(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                    scale: float, workspace=None, err=None, stream=None) -> None:
    """Store the new tokens' rows k_new, v_new [B, Hkv, D] at position context_lens - 1 of each
    sequence and decode, in one launch (= pa_store_kv, then pa_decode)."""
    NB, bs, Hkv, D = k_cache.shape
    B, Hq, Dq = q.shape
    if (Dq != D or tuple(out.shape) != (B, Hq, D) or tuple(k_new.shape) != (B, Hkv, D) or
            tuple(v_new.shape) != (B, Hkv, D) or block_tables.shape[0] != B or
            context_lens.shape != (B,)):
        raise ValueError("shape mismatch")
    dt = _dtype(q)
    if any(t.dtype != q.dtype for t in (out, k_new, v_new, k_cache, v_cache)):
        raise TypeError("q, out, the new rows and the pools must share a dtype")
    maxb = block_tables.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_store_decode", load().pa_store_decode(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _i32(block_tables, "block_tables"), maxb, _i32(context_lens, "context_lens"), B, Hq, Hkv,
        D, bs, NB, float(scale), dt, _ptr(workspace), ws_bytes, _i32(err, "err"),
        _stream(stream, q)))


def _hptr(t: torch.Tensor | None):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("host tensors expected (page-locked ones let the copies run asynchronously)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def pa_store_decode_host_workspace_size(B, Hq, Hkv, D, max_blocks_per_seq, block_size) -> int:
    return int(load().pa_store_decode_host_workspace_size(B, Hq, Hkv, D, max_blocks_per_seq, block_size))


def pa_store_decode_host_layout(B, Hq, Hkv, D, max_blocks_per_seq):
    """(offsets of q, k_new, v_new, block_tables, context_lens; total bytes) of the packed host
    layout whose inputs pa_store_decode_host moves in one copy; (None, 0) for invalid sizes."""
    offs = (ctypes.c_size_t * 5)()
    n = int(load().pa_store_decode_host_layout(B, Hq, Hkv, D, max_blocks_per_seq, offs))
    return (tuple(int(x) for x in offs) if n else None), n


def pa_store_decode_host(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                         scale: float, workspace, err=None, stream=None) -> None:
    """pa_store_decode with q, k_new, v_new, block_tables, context_lens and out in host memory
    (the pools on the device): the library copies the inputs in, runs the step and copies the
    output back, all queued on the stream. Synchronise the stream before reading `out`."""
    NB, bs, Hkv, D = k_cache.shape
    B, Hq, Dq = q.shape
    if (Dq != D or tuple(out.shape) != (B, Hq, D) or tuple(k_new.shape) != (B, Hkv, D) or
            tuple(v_new.shape) != (B, Hkv, D) or block_tables.shape[0] != B or
            context_lens.shape != (B,)):
        raise ValueError("shape mismatch")
    dt = _dtype(q)
    if any(t.dtype != q.dtype for t in (out, k_new, v_new, k_cache, v_cache)):
        raise TypeError("q, out, the new rows and the pools must share a dtype")
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    maxb = block_tables.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pa_store_decode_host", load().pa_store_decode_host(
        _hptr(out), _hptr(q), _hptr(k_new), _hptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _hptr(block_tables), maxb, _hptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale), dt,
        _ptr(workspace), ws_bytes, _i32(err, "err"), _stream(stream, k_cache)))


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                      err=None, stream=None) -> None:
    """pa_decode without a workspace argument: for callers that cannot allocate device memory.
    Its scratch is the library's fixed device array (PA_DECODE_NOALLOC_SCRATCH_BYTES); sizes
    that need more raise PagedAttnError with status 5. Calls that overlap on the GPU race on
    that array."""
    NB, bs, Hkv, D = k_cache.shape
    B, Hq, Dq = q.shape
    if Dq != D or tuple(out.shape) != (B, Hq, D) or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch")
    dt = _dtype(q)
    if out.dtype != q.dtype or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q, out and the pools must share a dtype")
    _check("pa_decode_noalloc", load().pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _i32(block_tables, "block_tables"),
        block_tables.shape[1], _i32(context_lens, "context_lens"), B, Hq, Hkv, D, bs, NB,
        float(scale), dt, _i32(err, "err"), _stream(stream, q)))


def pa_prefill_varlen(out, q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                      max_seqlen_q: int, max_seqlen_k: int, block_tables=None, *, Hkv: int,
                      scale: float, causal: bool = True, err=None, stream=None) -> None:
    """Varlen (causal) prefill: out [Tq, Hq, D]. Keys come from the pools through block_tables,
    or from the packed k, v when block_tables is None."""
    Tq, Hq, D = q.shape
    if tuple(out.shape) != (Tq, Hq, D):
        raise ValueError("out must match q")
    S = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != S + 1:
        raise ValueError("cu_seqlens_k must have S+1 entries")
    dt = _dtype(q)
    if block_tables is not None:
        NB, bs, Hkv_c, Dc = k_cache.shape
        if Hkv_c != Hkv or Dc != D or block_tables.shape[0] != S:
            raise ValueError("pool / table shape mismatch")
        maxb = block_tables.shape[1]
    else:
        NB, bs, maxb = 0, 1, 0
        if k.shape[1:] != (Hkv, D) or v.shape != k.shape:
            raise ValueError("packed k, v must be [Tk, Hkv, D]")
    for t in (out, k, v, k_cache, v_cache):
        if t is not None and t.dtype != q.dtype:
            raise TypeError("all attention tensors must share a dtype")
    total_k = 0 if block_tables is not None else int(k.shape[0])
    _check("pa_prefill_varlen", load().pa_prefill_varlen(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
        _i32(cu_seqlens_q, "cu_seqlens_q"), _i32(cu_seqlens_k, "cu_seqlens_k"), S, Tq, total_k,
        int(max_seqlen_q), int(max_seqlen_k), _i32(block_tables, "block_tables"), maxb, Hq, Hkv, D,
        bs, NB, float(scale), int(bool(causal)), dt, _i32(err, "err"), _stream(stream, q)))


# ---------------------------------------------------------------------------------------------
# host block manager
# ---------------------------------------------------------------------------------------------

PA_BM_DEGENERATE_HASH = 1
BM_ERRORS = {-1: "bad argument", -2: "no free blocks", -3: "unknown sequence",
             -4: "sequence already allocated"}


class BlockManagerError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({BM_ERRORS.get(code, 'unknown')})")
        self.code = code


class BlockManager:
    """The library's host block manager (include/pa.h, pa_bm_*): block ids, reference counts and
    the exact full-block prefix cache, one block table per sequence. Marshalling only."""

    def __init__(self, num_blocks: int, block_size: int, flags: int = 0):
        self._lib = load()
        self._h = self._lib.pa_bm_create(int(num_blocks), int(block_size), int(flags))
        if not self._h:
            raise BlockManagerError("pa_bm_create", -1)
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pa_bm_destroy(h)

    @staticmethod
    def _tokens(tokens):
        import numpy as np
        a = np.ascontiguousarray(tokens, dtype=np.int32)
        return a, a.ctypes.data

    def _ok(self, fn: str, r: int) -> int:
        if r < 0:
            raise BlockManagerError(fn, int(r))
        return int(r)

    def allocate(self, seq: int, tokens) -> int:
        """Blocks for a new sequence; returns the number of its tokens already cached."""
        a, ptr = self._tokens(tokens)
        return self._ok("pa_bm_allocate", self._lib.pa_bm_allocate(self._h, int(seq), ptr, a.size))

    def can_allocate(self, tokens) -> bool:
        a, ptr = self._tokens(tokens)
        return bool(self._ok("pa_bm_can_allocate", self._lib.pa_bm_can_allocate(self._h, ptr, a.size)))

    def append(self, seq: int, token: int) -> int:
        """One more token; returns its slot."""
        return self._ok("pa_bm_append", self._lib.pa_bm_append(self._h, int(seq), int(token)))

    def release(self, seq: int) -> None:
        self._ok("pa_bm_release", self._lib.pa_bm_release(self._h, int(seq)))

    def block_table(self, seq: int) -> list:
        import numpy as np
        n = self._ok("pa_bm_block_table", self._lib.pa_bm_block_table(self._h, int(seq), None, 0))
        out = np.empty(max(n, 1), dtype=np.int32)
        self._ok("pa_bm_block_table", self._lib.pa_bm_block_table(self._h, int(seq), out.ctypes.data, n))
        return out[:n].tolist()

    def num_tokens(self, seq: int) -> int:
        return self._ok("pa_bm_num_tokens", self._lib.pa_bm_num_tokens(self._h, int(seq)))

    def num_free(self) -> int:
        return self._ok("pa_bm_num_free", self._lib.pa_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return self._ok("pa_bm_refcount", self._lib.pa_bm_refcount(self._h, int(block)))
