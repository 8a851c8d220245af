"""Host-side expectations for the GPU parity tests: inputs regenerated on the host by the
seeded generator and pushed through the CPU oracle only (nothing here reads a GPU result)."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle
from compressed_paged_kv_quant_gb300 import synth

ATOL, RTOL = 2e-3, 1e-3          # |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise
TWO_BIT = (oracle.FMT_HQ2B, oracle.FMT_HQ2B_HAD, oracle.FMT_HQ2B_TOK)   # formats with the exact-key ring
THREADS = max(1, min(32, os.cpu_count() or 1))


def assert_close(gpu, ref, atol=ATOL, rtol=RTOL, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"{err.max():.3e} (ref {ref.flat[np.argmax(err)]:.4f})")
    return float(err.max())


def host_kv(wl: synth.Workload, layer: int, lane: int, pos0: int, n: int, kv: int):
    """bf16 bits [n][H][256] regenerated on the host (parallel chunks)."""
    return synth.kv_np_parallel(wl, layer, lane, pos0, n, kv, threads=THREADS)


class LaneCache:
    """The oracle's cache for one lane of one layer (geometry with a single layer; the lane's
    pages renumbered 0..n-1 in table order)."""

    def __init__(self, wl: synth.Workload, fmt: int, layer: int, lane: int, upto: int = None,
                 fill: int = 0xA5):
        self.wl, self.fmt, self.layer, self.lane = wl, fmt, layer, lane
        n = wl.seq_len[lane] if upto is None else upto
        self.n = n
        self.g = oracle.geom(fmt, 1, wl.num_kv_heads, wl.num_q_heads)
        self.pb = oracle.page_bytes(self.g)
        npg = (n + 63) // 64
        self.pt = np.arange(npg, dtype=np.int32)[None, :]
        self.pool = np.full(max(npg, 1) * self.pb, fill, np.uint8)
        self.ring = np.zeros((1, 1, wl.num_kv_heads, 64, 256), np.uint16) if fmt in TWO_BIT else None
        self.k = host_kv(wl, layer, lane, 0, n, 0)
        self.v = host_kv(wl, layer, lane, 0, n, 1)
        st = oracle.append(self.g, 0, self.pool, self.ring, self.pt, 1, [0], [n], [0], self.k, self.v)
        assert st == 0

    def block(self, page_index: int, head: int, kv: int) -> np.ndarray:
        bb = self.pb // (self.wl.num_kv_heads * 2)
        off = page_index * self.pb + (head * 2 + kv) * bb
        return self.pool[off:off + bb]

    def attend(self, q_rows: np.ndarray, positions, window: int, sm_scale: float):
        """q_rows bf16 [R][Hq][256] at `positions` (causal) -> float64 [R][Hq][256]."""
        R, Hq = q_rows.shape[0], q_rows.shape[1]
        out = np.zeros((R, Hq, 256))
        units = [(r, j) for r in range(R) for j in range(Hq)]

        def one(u):
            r, j = u
            o, _, st = oracle.attend(self.g, 0, self.pool, self.ring, window, self.pt[0], 0, self.n, j,
                                     q_rows[r, j], positions[r] + 1, sm_scale)
            assert st == 0
            return u, o

        with cf.ThreadPoolExecutor(THREADS) as ex:
            for (r, j), o in ex.map(one, units):
                out[r, j] = o
        return out


def gpu_block(pool_u8: np.ndarray, page_bytes: int, num_kv_heads: int, fmt: int, phys: int, layer: int,
              head: int, kv: int) -> np.ndarray:
    """Bytes of one (layer, head, K/V) block of physical page `phys` of a copied-back pool."""
    bb = 64 * oracle.head_token_bytes(fmt)
    off = phys * page_bytes + ((layer * num_kv_heads + head) * 2 + kv) * bb
    return pool_u8[off:off + bb]
