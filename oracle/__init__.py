"""CPU oracle for the 2-bit paged KV cache: ctypes binding of ``kvq_oracle.c``.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg
may import this package; the library's compute path never does.  The oracle shares no code
with the CUDA path (see the header of ``kvq_oracle.c`` for what it computes and where the
pages define each step).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_HQ2B = 0
FMT_BF16 = 1
FMT_HQ2B_HAD = 2   # the 2-bit format over Walsh-Hadamard-rotated K and V rows
FMT_HQ2B_TOK = 3   # the 2-bit format with K quantized per token (V rule), no page close
FMT_FP8 = 4        # K and V rows as FP8 E4M3 (one byte a value) with a per-tensor scale each
PAGE_OOB, LEN_GT_TABLE, BAD_INPUT, BAD_LEN = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Geom(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


def geom(fmt: int, layers: int, kv_heads: int, q_heads: int, k_scale: float = 0.0, v_scale: float = 0.0) -> Geom:
    """k_scale / v_scale: the FP8 format's per-tensor scales (0 means 1); other formats ignore them."""
    return Geom(fmt, layers, kv_heads, q_heads, 256, 64, k_scale, v_scale)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            G = ctypes.POINTER(Geom)
            i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_round_bf16.argtypes = [ctypes.c_float]
            L.orc_round_bf16.restype = ctypes.c_float
            L.orc_kv_bytes_per_token.argtypes = [i32, i32, i32, dbl]
            L.orc_kv_bytes_per_token.restype = dbl
            L.orc_head_token_bytes.argtypes = [i32]
            L.orc_head_token_bytes.restype = i64
            L.orc_token_bytes.argtypes = [G]
            L.orc_token_bytes.restype = i64
            L.orc_page_bytes.argtypes = [G]
            L.orc_page_bytes.restype = i64
            L.orc_quant_v_row.argtypes = [P, P, P]
            L.orc_quant_k_page.argtypes = [P, P, P]
            L.orc_dequant_v_row.argtypes = [P, P, P]
            L.orc_dequant_k_row.argtypes = [P, P, P]
            L.orc_quant_v_row_f32.argtypes = [P, P, P]
            L.orc_quant_k_page_f32.argtypes = [P, P, P]
            L.orc_fwht_f32.argtypes = [P]
            L.orc_hadamard_f64.argtypes = [P, P]
            L.orc_append.argtypes = [G, i32, P, i64, P, P, i32, i32, P, P, P, P, P]
            L.orc_append.restype = i32
            L.orc_attend.argtypes = [G, i32, P, i64, P, i32, P, i32, i32, i32, i32, P, i64, dbl, P, P]
            L.orc_attend.restype = i32
            L.orc_decode.argtypes = [G, i32, P, i64, P, i32, P, i32, i32, P, P, dbl, P]
            L.orc_decode.restype = i32
            L.orc_prefill.argtypes = [G, i32, P, i64, P, i32, P, i32, i32, P, P, P, P, P, dbl, P]
            L.orc_prefill.restype = i32
            L.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
            L.orc_f32_to_e4m3.restype = ctypes.c_uint8
            L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_f64.restype = dbl
            L.orc_flat_sum.argtypes = [i32, i32, i32]
            L.orc_flat_sum.restype = dbl
            _lib = L
    return _lib


class _Keep:
    """Converts arguments to contiguous arrays and keeps them alive for the C call."""

    def __init__(self):
        self.refs = []

    def __call__(self, a, dt=None):
        if a is None:
            return None
        if dt is not None:
            a = np.ascontiguousarray(a, dtype=dt)
        assert a.flags.c_contiguous
        self.refs.append(a)
        return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------ scalar helpers
def f32_to_f16(x: float) -> int:
    return int(lib().orc_f32_to_f16(float(x)))


def f16_to_f32(h: int) -> float:
    return float(lib().orc_f16_to_f32(int(h)))


def f32_to_e4m3(x: float) -> int:
    """FP8 E4M3 byte of a float: round to nearest even, saturating at +-448."""
    return int(lib().orc_f32_to_e4m3(x))


def e4m3_to_f64(b: int) -> float:
    return float(lib().orc_e4m3_to_f64(b))


def round_bf16(x: float) -> float:
    return float(lib().orc_round_bf16(float(x)))


def kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_value) -> float:
    return lib().orc_kv_bytes_per_token(layers, kv_heads, head_dim, float(bytes_per_value))


def head_token_bytes(fmt: int) -> int:
    return int(lib().orc_head_token_bytes(fmt))


def token_bytes(g: Geom) -> int:
    return int(lib().orc_token_bytes(ctypes.byref(g)))


def page_bytes(g: Geom) -> int:
    return int(lib().orc_page_bytes(ctypes.byref(g)))


def flat_sum(n: int, kind: str, two_level: bool = False) -> float:
    return lib().orc_flat_sum(n, {"fp32": 0, "fp16": 1, "bf16": 2}[kind], int(two_level))


# ------------------------------------------------------------------ quantizer
def quant_v_row(x_bf16: np.ndarray):
    k = _Keep()
    codes = np.zeros(64, np.uint8)
    meta = np.zeros(4, np.uint16)
    lib().orc_quant_v_row(k(x_bf16, np.uint16), k(codes), k(meta))
    return codes, meta


def quant_k_page(x_bf16: np.ndarray):
    k = _Keep()
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    assert x.shape == (64, 256)
    codes = np.zeros((64, 64), np.uint8)
    scales = np.zeros(256, np.uint16)
    lib().orc_quant_k_page(k(x), k(codes), k(scales))
    return codes, scales


def dequant_v_row(codes, meta) -> np.ndarray:
    k = _Keep()
    out = np.zeros(256, np.float64)
    lib().orc_dequant_v_row(k(codes, np.uint8), k(meta, np.uint16), k(out))
    return out


def dequant_k_row(codes_row, scales) -> np.ndarray:
    k = _Keep()
    out = np.zeros(256, np.float64)
    lib().orc_dequant_k_row(k(codes_row, np.uint8), k(scales, np.uint16), k(out))
    return out


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """The rotated variant's quantizer input: fast Walsh-Hadamard transform of 256 floats in
    float (stages h = 1..128), then x 1/16."""
    k = _Keep()
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    assert y.shape == (256,)
    lib().orc_fwht_f32(k(y))
    return y


def hadamard_f64(x: np.ndarray) -> np.ndarray:
    """H x in double from the definition H[i][j] = (-1)^popcount(i & j) / 16."""
    k = _Keep()
    y = np.zeros(256, np.float64)
    lib().orc_hadamard_f64(k(x, np.float64), k(y))
    return y


# ------------------------------------------------------------------ cache
def append(g: Geom, layer: int, pool: np.ndarray, ring, page_table: np.ndarray, lanes: int,
           start_pos, n_new, tok_offset, k: np.ndarray, v: np.ndarray) -> int:
    """Sequential token-by-token append into ``pool`` (uint8) and ``ring`` (uint16, in place)."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    assert ring is None or (ring.dtype == np.uint16 and ring.flags.c_contiguous)
    K = _Keep()
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    return int(lib().orc_append(ctypes.byref(g), layer, K(pool), pool.nbytes, K(ring), K(pt),
                                pt.shape[1], lanes, K(start_pos, np.int32), K(n_new, np.int32),
                                K(tok_offset, np.int32), K(k, np.uint16), K(v, np.uint16)))


def attend(g: Geom, layer: int, pool, ring, window: int, page_row, lane: int, seq_len: int,
           q_head: int, q_row, n_keys: int, sm_scale: float):
    """One query row over keys 0..n_keys-1 -> (out[256] float64, top1 index, status)."""
    K = _Keep()
    out = np.zeros(256, np.float64)
    top1 = ctypes.c_int64(-1)
    pr = np.ascontiguousarray(page_row, dtype=np.int32)
    st = lib().orc_attend(ctypes.byref(g), layer, K(pool), pool.nbytes, K(ring), window, K(pr),
                          pr.shape[-1], lane, seq_len, q_head, K(q_row, np.uint16), n_keys,
                          sm_scale, K(out), ctypes.byref(top1))
    return out, int(top1.value), int(st)


def decode(g: Geom, layer: int, pool, ring, window: int, page_table, lanes: int, seq_len,
           q: np.ndarray, sm_scale: float):
    K = _Keep()
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    out = np.zeros((lanes, g.num_q_heads, 256), np.float64)
    st = lib().orc_decode(ctypes.byref(g), layer, K(pool), pool.nbytes, K(ring), window, K(pt),
                          pt.shape[1], lanes, K(seq_len, np.int32), K(q, np.uint16), sm_scale, K(out))
    return out, int(st)


def prefill(g: Geom, layer: int, pool, ring, window: int, page_table, lanes: int, q_pos0, n_q,
            q_offset, seq_len, q: np.ndarray, sm_scale: float):
    K = _Keep()
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    qa = np.ascontiguousarray(q, dtype=np.uint16)
    out = np.zeros((qa.shape[0], g.num_q_heads, 256), np.float64)
    st = lib().orc_prefill(ctypes.byref(g), layer, K(pool), pool.nbytes, K(ring), window, K(pt),
                           pt.shape[1], lanes, K(q_pos0, np.int32), K(n_q, np.int32),
                           K(q_offset, np.int32), K(seq_len, np.int32), K(qa), sm_scale, K(out))
    return out, int(st)


def pages_gather(g: Geom, pool: np.ndarray, page_ids) -> np.ndarray:
    """Page moves ("The KV cache and prompt reuse", "What a sequence is made of": whole pages are
    what a cache moves to a slower tier and back): arena slot i holds the bytes of pool page
    page_ids[i].  A page is opaque bytes; ids outside the pool are skipped (slot left zero) and
    reported as PAGE_OOB."""
    pb = page_bytes(g)
    n_pool = pool.size // pb
    arena = np.zeros(len(page_ids) * pb, np.uint8)
    st = 0
    for i, p in enumerate(page_ids):
        if 0 <= p < n_pool:
            arena[i * pb:(i + 1) * pb] = pool[p * pb:(p + 1) * pb]
        else:
            st |= PAGE_OOB
    return arena, st


def pages_scatter(g: Geom, pool: np.ndarray, page_ids, arena: np.ndarray) -> int:
    """Inverse move: pool page page_ids[i] takes the bytes of arena slot i (in place)."""
    pb = page_bytes(g)
    n_pool = pool.size // pb
    st = 0
    for i, p in enumerate(page_ids):
        if 0 <= p < n_pool:
            pool[p * pb:(p + 1) * pb] = arena[i * pb:(i + 1) * pb]
        else:
            st |= PAGE_OOB
    return st
