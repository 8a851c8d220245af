"""ctypes binding of ``libkvq.so`` (C ABI in ``include/kvq.h``).

Argument marshalling only: every step of the attention path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the library is not
built, importing the functions fails loudly; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

FMT_HQ2B = 0
FMT_BF16 = 1
FMT_HQ2B_HAD = 2   # the HQ2B layout over Walsh-Hadamard-rotated K and V rows
FMT_HQ2B_TOK = 3   # the HQ2B layout with K rows coded per token (V rule), no page close
FMT_FP8 = 4        # K and V rows as FP8 E4M3 with a per-tensor scale each

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE_TOO_SMALL = -3
ERR_CUDA = -4
ERR_ALIGNMENT = -5
ERR_SCRATCH_LIMIT = -6
NOALLOC_SCRATCH_BYTES = 32 << 20

STATUS_PAGE_OOB = 1
STATUS_LEN_GT_TABLE = 2
STATUS_BAD_INPUT = 4
STATUS_BAD_LEN = 8
STATUS_TIMEOUT = 16

EXPORTS = ("kvq_page_bytes", "kvq_token_bytes", "kvq_ring_bytes", "kvq_pool_pages",
           "kvq_decode_workspace_bytes", "kvq_prefill_workspace_bytes", "kvq_strerror",
           "kvq_build_arch", "kv_quant_append", "paged_decode_attn", "paged_prefill_attn",
           "paged_decode_attn_noalloc", "kvq_decode_step", "kvq_pages_gather", "kvq_pages_scatter",
           "kvq_selftest_wait_timeout")


class KvqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class Geom(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]

    def __repr__(self):
        return (f"Geom(format={self.format}, L={self.num_layers}, Hkv={self.num_kv_heads}, "
                f"Hq={self.num_q_heads}, D={self.head_dim}, P={self.page_tokens})")


def geom(fmt: int, num_layers: int, num_kv_heads: int, num_q_heads: int,
         head_dim: int = 256, page_tokens: int = 64, k_scale: float = 0.0, v_scale: float = 0.0) -> Geom:
    """k_scale / v_scale: the FP8 format's per-tensor scales (0 means 1)."""
    return Geom(fmt, num_layers, num_kv_heads, num_q_heads, head_dim, page_tokens, k_scale, v_scale)


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libkvq.so is not built ({LIB_PATH}); run "
                                   "compressed_paged_kv_quant_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, G = ctypes.c_void_p, ctypes.POINTER(Geom)
            i32, i64, sz, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
            L.kvq_page_bytes.argtypes = [G]
            L.kvq_page_bytes.restype = sz
            L.kvq_token_bytes.argtypes = [G]
            L.kvq_token_bytes.restype = sz
            L.kvq_ring_bytes.argtypes = [G, i32]
            L.kvq_ring_bytes.restype = sz
            L.kvq_pool_pages.argtypes = [G, sz]
            L.kvq_pool_pages.restype = i64
            L.kvq_decode_workspace_bytes.argtypes = [G, i32, i32]
            L.kvq_decode_workspace_bytes.restype = sz
            L.kvq_prefill_workspace_bytes.argtypes = [G, i32, i32]
            L.kvq_prefill_workspace_bytes.restype = sz
            L.kvq_strerror.argtypes = [i32]
            L.kvq_strerror.restype = ctypes.c_char_p
            L.kvq_build_arch.argtypes = []
            L.kvq_build_arch.restype = i32
            L.kv_quant_append.argtypes = [G, i32, P, sz, P, P, i32, i32, P, P, P, i32, i32, P, P, P, P]
            L.kv_quant_append.restype = i32
            L.paged_decode_attn.argtypes = [G, i32, P, sz, P, i32, P, i32, i32, P, i32, P, f32, P, sz, P,
                                            P, P]
            L.paged_decode_attn.restype = i32
            L.paged_prefill_attn.argtypes = [G, i32, P, sz, P, i32, P, i32, i32, P, P, P, i32, i32, P, i32,
                                             P, f32, P, sz, P, P, P]
            L.paged_prefill_attn.restype = i32
            L.paged_decode_attn_noalloc.argtypes = [G, i32, P, sz, P, i32, P, i32, i32, P, i32, P, f32, P, P, P]
            L.paged_decode_attn_noalloc.restype = i32
            L.kvq_decode_step.argtypes = [G, i32, P, sz, P, i32, P, i32, i32, P, P, P, i32, P, P, P, i32, P, f32, P,
                                          sz, P, P, P]
            L.kvq_decode_step.restype = i32
            L.kvq_pages_gather.argtypes = [G, P, sz, P, i32, P, P, P]
            L.kvq_pages_gather.restype = i32
            L.kvq_pages_scatter.argtypes = [G, P, sz, P, i32, P, P, P]
            L.kvq_pages_scatter.restype = i32
            L.kvq_selftest_wait_timeout.argtypes = [P, P]
            L.kvq_selftest_wait_timeout.restype = i32
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().kvq_strerror(int(code)).decode()


def page_bytes(g: Geom) -> int:
    return int(lib().kvq_page_bytes(ctypes.byref(g)))


def token_bytes(g: Geom) -> int:
    return int(lib().kvq_token_bytes(ctypes.byref(g)))


def ring_bytes(g: Geom, lanes: int) -> int:
    return int(lib().kvq_ring_bytes(ctypes.byref(g), lanes))


def pool_pages(g: Geom, pool_bytes: int) -> int:
    return int(lib().kvq_pool_pages(ctypes.byref(g), pool_bytes))


def decode_workspace_bytes(g: Geom, lanes: int, max_seq_len: int) -> int:
    return int(lib().kvq_decode_workspace_bytes(ctypes.byref(g), lanes, max_seq_len))


def prefill_workspace_bytes(g: Geom, n_q_rows: int, max_seq_len: int) -> int:
    return int(lib().kvq_prefill_workspace_bytes(ctypes.byref(g), n_q_rows, max_seq_len))


# ----------------------------------------------------------------------------- marshalling
def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    assert t.is_cuda and t.is_contiguous(), "device tensors must be contiguous CUDA tensors"
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(rc: int, what: str):
    if rc != OK:
        raise KvqError(rc, what)


def _arena_ptr(t) -> int:
    """A page arena: a contiguous CUDA tensor, or pinned host memory (under unified addressing the
    host pointer of pinned memory is valid on the device)."""
    assert t.is_contiguous() and (t.is_cuda or t.is_pinned()), "the arena must be a CUDA or pinned host tensor"
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def kv_quant_append(g: Geom, layer: int, pool, ring, page_table, start_pos, n_new, tok_offset,
                    max_new: int, k, v, status, stream=None, n_rows: Optional[int] = None):
    """Quantize and append new K/V rows of one layer (see ``kv_quant_append`` in kvq.h)."""
    lanes, max_pages = (page_table.shape[0], page_table.shape[1]) if page_table.dim() == 2 else (1, page_table.shape[0])
    rows = k.shape[0] if n_rows is None else n_rows
    rc = lib().kv_quant_append(ctypes.byref(g), layer, _ptr(pool), _nbytes(pool), _ptr(ring),
                               _ptr(page_table), max_pages, lanes, _ptr(start_pos), _ptr(n_new),
                               _ptr(tok_offset), max_new, rows, _ptr(k), _ptr(v), _ptr(status),
                               _stream(stream))
    _check(rc, "kv_quant_append")


def paged_decode_attn(g: Geom, layer: int, pool, ring, window: int, page_table, seq_len,
                      max_seq_len: int, q, sm_scale: float, workspace, out, status, stream=None,
                      lanes: Optional[int] = None):
    """One query token per lane attends its whole cache (see ``paged_decode_attn`` in kvq.h)."""
    n_lanes = page_table.shape[0] if lanes is None else lanes
    rc = lib().paged_decode_attn(ctypes.byref(g), layer, _ptr(pool), _nbytes(pool), _ptr(ring), window,
                                 _ptr(page_table), page_table.shape[1], n_lanes, _ptr(seq_len),
                                 max_seq_len, _ptr(q), float(sm_scale), _ptr(workspace),
                                 _nbytes(workspace), _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "paged_decode_attn")


def paged_decode_attn_noalloc(g: Geom, layer: int, pool, ring, window: int, page_table, seq_len,
                              max_seq_len: int, q, sm_scale: float, out, status, stream=None,
                              lanes: Optional[int] = None):
    """paged_decode_attn with the library's static scratch instead of a caller workspace, for
    callers that cannot allocate device memory (see ``paged_decode_attn_noalloc`` in kvq.h)."""
    n_lanes = page_table.shape[0] if lanes is None else lanes
    rc = lib().paged_decode_attn_noalloc(ctypes.byref(g), layer, _ptr(pool), _nbytes(pool), _ptr(ring), window,
                                         _ptr(page_table), page_table.shape[1], n_lanes, _ptr(seq_len), max_seq_len,
                                         _ptr(q), float(sm_scale), _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "paged_decode_attn_noalloc")


def kvq_decode_step(g: Geom, layer: int, pool, ring, window: int, page_table, start_pos, n_new, tok_offset, k, v,
                    seq_len, max_seq_len: int, q, sm_scale: float, workspace, out, status, stream=None,
                    n_rows: Optional[int] = None):
    """Append at most one token per lane, then decode attention over the cache that includes it
    (see ``kvq_decode_step`` in kvq.h)."""
    lanes, max_pages = page_table.shape[0], page_table.shape[1]
    rows = k.shape[0] if n_rows is None else n_rows
    rc = lib().kvq_decode_step(ctypes.byref(g), layer, _ptr(pool), _nbytes(pool), _ptr(ring), window,
                               _ptr(page_table), max_pages, lanes, _ptr(start_pos), _ptr(n_new), _ptr(tok_offset),
                               rows, _ptr(k), _ptr(v), _ptr(seq_len), max_seq_len, _ptr(q), float(sm_scale),
                               _ptr(workspace), _nbytes(workspace), _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "kvq_decode_step")


def pages_gather(g: Geom, pool, page_ids, arena, status, stream=None):
    """Copy pool pages page_ids[i] into arena slot i (see ``kvq_pages_gather`` in kvq.h)."""
    rc = lib().kvq_pages_gather(ctypes.byref(g), _ptr(pool), _nbytes(pool), _ptr(page_ids), page_ids.numel(),
                                _arena_ptr(arena), _ptr(status), _stream(stream))
    _check(rc, "kvq_pages_gather")


def pages_scatter(g: Geom, pool, page_ids, arena, status, stream=None):
    """Copy arena slot i into pool page page_ids[i] (see ``kvq_pages_scatter`` in kvq.h)."""
    rc = lib().kvq_pages_scatter(ctypes.byref(g), _ptr(pool), _nbytes(pool), _ptr(page_ids), page_ids.numel(),
                                 _arena_ptr(arena), _ptr(status), _stream(stream))
    _check(rc, "kvq_pages_scatter")


def selftest_wait_timeout(status, stream=None):
    """Run one bounded barrier wait that nothing ends (see ``kvq_selftest_wait_timeout``)."""
    _check(lib().kvq_selftest_wait_timeout(_ptr(status), _stream(stream)), "kvq_selftest_wait_timeout")


def paged_prefill_attn(g: Geom, layer: int, pool, ring, window: int, page_table, q_pos0, n_q,
                       q_offset, max_n_q: int, seq_len, max_seq_len: int, q, sm_scale: float,
                       workspace, out, status, stream=None, lanes: Optional[int] = None):
    """A chunk of queries attends causally over the cache (see ``paged_prefill_attn``)."""
    n_lanes = page_table.shape[0] if lanes is None else lanes
    rc = lib().paged_prefill_attn(ctypes.byref(g), layer, _ptr(pool), _nbytes(pool), _ptr(ring), window,
                                  _ptr(page_table), page_table.shape[1], n_lanes, _ptr(q_pos0), _ptr(n_q),
                                  _ptr(q_offset), max_n_q, q.shape[0], _ptr(seq_len), max_seq_len,
                                  _ptr(q), float(sm_scale), _ptr(workspace), _nbytes(workspace),
                                  _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "paged_prefill_attn")


# ----------------------------------------------------------------------------- convenience
class PagedCache:
    """Device buffers of one paged cache: the byte pool, the exact-key ring and a status word.

    Allocation goes through torch; the kernels only ever see the raw pointers.
    """

    def __init__(self, g: Geom, pool_pages: int, lanes: int, device="cuda", fill: Optional[int] = None):
        import torch
        self.g = g
        self.lanes = lanes
        pb = page_bytes(g)
        if pb == 0:
            raise KvqError(ERR_UNSUPPORTED, "PagedCache")
        self.pool = torch.empty(pool_pages * pb, dtype=torch.uint8, device=device)
        if fill is not None:
            self.pool.fill_(fill)
        rb = ring_bytes(g, lanes)
        self.ring = torch.zeros(max(rb // 2, 8), dtype=torch.bfloat16, device=device) if rb else None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def read_status(self) -> int:
        return int(self.status.item())

    def clear_status(self):
        self.status.zero_()
