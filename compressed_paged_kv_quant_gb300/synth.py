"""Seeded, counter-based synthetic inputs for the paged KV attention path.

The CPU oracle's tests and the GPU runs both draw their K, V and Q tensors and their page
tables from this module.  It therefore holds none of the method's arithmetic: only an
integer hash, a sum of uniforms, and the float32 -> bfloat16 rounding that turns a draw into
a bf16 input.

Every value is a pure function of ``(seed, tag, coordinates)``.  Any slice of a full-size
workload can be regenerated on the host for a sampled check of a GPU run, and the device
implementation (torch integer ops) yields the same bits as the host one (numpy).

Value recipe
------------
* hash: the SplitMix64 finaliser (Steele, Lea, Flood 2014) applied to ``base + 6*counter + k``.
* ``N(0,1)``: the Irwin-Hall sum of twelve 32-bit uniforms minus 6 (mean 0, variance 1,
  range +-6).  Every step is an exact integer or power-of-two operation, so the float64
  value is bit-identical on any IEEE machine; no transcendental function is involved.
* outliers, following the synthetic cache of "Half the Cache, Twice the Context",
  section "What the cache loses when you round it": keys get persistent channel outliers
  (every 16th channel x4) and values get outlier tokens (every 64th absolute position x6).
  The factor is applied in float64 (exact), then float64 -> float32 -> bfloat16,
  both round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

HEAD_DIM = 256
PAGE_TOKENS = 64

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK32 = 0xFFFFFFFF

TAG_KV = 1
TAG_Q = 2
TAG_PERM = 3
TAG_NEEDLE = 4

# counter field widths (bits): layer 6 | stream 6 | pos 21 | head 6 | kv 1 | dim 8
_POS_BITS = 21
_HEAD_BITS = 6
MAX_POS = 1 << _POS_BITS
MAX_HEADS = 1 << _HEAD_BITS
MAX_STREAMS = 64
MAX_LAYERS = 64


# --------------------------------------------------------------------------- hash (numpy)
def _mix_np(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = z + np.uint64(_GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        return z ^ (z >> np.uint64(31))


def _base(seed: int, tag: int) -> int:
    z = np.array([(seed * 256 + tag) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix_np(z)[0])


def rand_u64(seed: int, tag: int, idx: np.ndarray) -> np.ndarray:
    """Uniform 64-bit integers, one per counter in ``idx``."""
    with np.errstate(over="ignore"):
        return _mix_np(np.uint64(_base(seed, tag)) + np.asarray(idx, dtype=np.uint64))


def _normal_from_counter_np(seed: int, tag: int, counter: np.ndarray) -> np.ndarray:
    """Irwin-Hall(12) draws as float64 (exactly representable)."""
    base = np.uint64(_base(seed, tag))
    c6 = counter.astype(np.uint64) * np.uint64(6)
    acc = np.zeros(counter.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        for k in range(6):
            r = _mix_np(base + c6 + np.uint64(k))
            acc += (r & np.uint64(_MASK32)).astype(np.int64)
            acc += (r >> np.uint64(32)).astype(np.int64)
    acc -= 6 << 32
    return acc.astype(np.float64) * (2.0 ** -32)


def f32_to_bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit pattern, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32_np(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- counters
def _kv_counter(layer: int, stream: int, pos: np.ndarray, head: np.ndarray, kv: int,
                dim: np.ndarray) -> np.ndarray:
    assert 0 <= layer < MAX_LAYERS and 0 <= stream < MAX_STREAMS
    lead = ((layer * MAX_STREAMS + stream) << _POS_BITS)
    c = (np.uint64(lead) + pos.astype(np.uint64))
    c = (c << np.uint64(_HEAD_BITS)) + head.astype(np.uint64)
    c = (c << np.uint64(1)) + np.uint64(kv)
    c = (c << np.uint64(8)) + dim.astype(np.uint64)
    return c


def kv_block_np(seed: int, layer: int, stream: int, pos0: int, n: int, num_kv_heads: int,
                kv: int, k_outliers: bool = True, v_outliers: bool = True) -> np.ndarray:
    """bf16 bits ``[n][num_kv_heads][256]`` of K (kv=0) or V (kv=1) for absolute positions
    ``pos0 .. pos0+n-1`` of content stream ``stream``."""
    assert pos0 >= 0 and pos0 + n <= MAX_POS and num_kv_heads <= MAX_HEADS
    pos = (pos0 + np.arange(n, dtype=np.int64))[:, None, None]
    head = np.arange(num_kv_heads, dtype=np.int64)[None, :, None]
    dim = np.arange(HEAD_DIM, dtype=np.int64)[None, None, :]
    cnt = _kv_counter(layer, stream, pos, head, kv, dim)
    x = _normal_from_counter_np(seed, TAG_KV, cnt)
    x = x * _outlier_np(pos, dim, kv, k_outliers, v_outliers)
    return f32_to_bf16_bits_np(x.astype(np.float32))


def _outlier_np(pos, dim, kv, k_outliers, v_outliers):
    if kv == 0 and k_outliers:
        return np.where(dim % 16 == 0, 4.0, 1.0)
    if kv == 1 and v_outliers:
        return np.where(pos % 64 == 0, 6.0, 1.0)
    return np.float64(1.0)


def q_block_np(seed: int, layer: int, lane: int, pos0: int, n: int, num_q_heads: int) -> np.ndarray:
    """bf16 bits ``[n][num_q_heads][256]`` of queries for positions ``pos0..pos0+n-1``."""
    pos = (pos0 + np.arange(n, dtype=np.int64))[:, None, None]
    head = np.arange(num_q_heads, dtype=np.int64)[None, :, None]
    dim = np.arange(HEAD_DIM, dtype=np.int64)[None, None, :]
    cnt = _kv_counter(layer, lane, pos, head, 0, dim)
    x = _normal_from_counter_np(seed, TAG_Q, cnt)
    return f32_to_bf16_bits_np(x.astype(np.float32))


# --------------------------------------------------------------------------- torch (device) twin
def _s64(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _shr_t(z, k: int):
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix_t(z):
    z = z + _s64(_GOLDEN)
    z = (z ^ _shr_t(z, 30)) * _s64(_M1)
    z = (z ^ _shr_t(z, 27)) * _s64(_M2)
    return z ^ _shr_t(z, 31)


def _normal_from_counter_t(seed: int, tag: int, counter):
    import torch
    base = _s64(_base(seed, tag))
    c6 = counter * 6 + base
    acc = torch.zeros_like(counter)
    for k in range(6):
        r = _mix_t(c6 + k)
        acc += r & _MASK32
        acc += _shr_t(r, 32)
    acc -= 6 << 32
    return acc.to(torch.float64) * (2.0 ** -32)


def kv_block_torch(seed: int, layer: int, stream: int, pos0: int, n: int, num_kv_heads: int,
                   kv: int, device, k_outliers: bool = True, v_outliers: bool = True,
                   chunk: int = 8192):
    """Same values as :func:`kv_block_np`, generated with torch ops on ``device`` (bf16)."""
    import torch
    assert pos0 >= 0 and pos0 + n <= MAX_POS
    out = torch.empty((n, num_kv_heads, HEAD_DIM), dtype=torch.bfloat16, device=device)
    head = torch.arange(num_kv_heads, dtype=torch.int64, device=device)[None, :, None]
    dim = torch.arange(HEAD_DIM, dtype=torch.int64, device=device)[None, None, :]
    lead = (layer * MAX_STREAMS + stream) << _POS_BITS
    for c0 in range(0, n, chunk):
        m = min(chunk, n - c0)
        pos = (pos0 + c0 + torch.arange(m, dtype=torch.int64, device=device))[:, None, None]
        cnt = ((((lead + pos) << _HEAD_BITS) + head) << 1) + kv
        cnt = (cnt << 8) + dim
        x = _normal_from_counter_t(seed, TAG_KV, cnt)
        if kv == 0 and k_outliers:
            x = x * torch.where(dim % 16 == 0, 4.0, 1.0).to(torch.float64)
        elif kv == 1 and v_outliers:
            x = x * torch.where(pos % 64 == 0, 6.0, 1.0).to(torch.float64)
        out[c0:c0 + m] = x.to(torch.float32).to(torch.bfloat16)
    return out


def q_block_torch(seed: int, layer: int, lane: int, pos0: int, n: int, num_q_heads: int, device):
    import torch
    head = torch.arange(num_q_heads, dtype=torch.int64, device=device)[None, :, None]
    dim = torch.arange(HEAD_DIM, dtype=torch.int64, device=device)[None, None, :]
    pos = (pos0 + torch.arange(n, dtype=torch.int64, device=device))[:, None, None]
    lead = (layer * MAX_STREAMS + lane) << _POS_BITS
    cnt = (((((lead + pos) << _HEAD_BITS) + head) << 1) << 8) + dim
    x = _normal_from_counter_t(seed, TAG_Q, cnt)
    return x.to(torch.float32).to(torch.bfloat16)


# --------------------------------------------------------------------------- permutations
def permutation(seed: int, n: int, salt: int = 0) -> np.ndarray:
    """Seeded Fisher-Yates shuffle of ``range(n)`` driven by the SplitMix64 hash."""
    r = rand_u64(seed, TAG_PERM, np.arange(n, dtype=np.uint64) + np.uint64(salt << 40))
    a = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(r[i] % np.uint64(i + 1))
        a[i], a[j] = a[j], a[i]
    return a


def seeded_int(seed: int, salt: int, bound: int) -> int:
    """One seeded integer in ``[0, bound)``."""
    return int(rand_u64(seed, TAG_NEEDLE, np.array([salt], dtype=np.uint64))[0] % np.uint64(bound))


# --------------------------------------------------------------------------- workloads
@dataclasses.dataclass
class Workload:
    """One synthetic workload: geometry, lane lengths, page tables, content streams.

    ``seq_len[b]`` is lane b's length after the step's append.  ``stream_of(b, pos)`` names
    the content stream of token ``pos`` of lane ``b``; lanes that share a prefix read the
    same stream there, so their shared pages hold identical bytes.
    """
    name: str
    num_layers: int
    num_kv_heads: int
    num_q_heads: int
    seq_len: List[int]
    page_table: np.ndarray          # int32 [lanes][max_pages], -1 where unused
    pool_pages: int
    window: int = 0
    seed: int = 0
    k_outliers: bool = True
    v_outliers: bool = True
    shared_prefix: int = 0          # tokens shared by lanes listed in shared_lanes
    shared_lanes: Sequence[int] = ()
    needle: Optional[dict] = None   # {"pos": int, "onehot": [j per kv head]}
    prefill_chunk: int = 0          # > 0: last `prefill_chunk` tokens of lane 0 are a prefill chunk

    @property
    def lanes(self) -> int:
        return len(self.seq_len)

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def stream_of(self, lane: int, pos: int) -> int:
        if lane in self.shared_lanes and pos < self.shared_prefix:
            return MAX_STREAMS - 1
        return lane

    def segments(self, lane: int, pos0: int, n: int):
        """Split ``[pos0, pos0+n)`` into runs of one content stream: (pos, count, stream)."""
        out = []
        p = pos0
        end = pos0 + n
        while p < end:
            s = self.stream_of(lane, p)
            q = p + 1
            if lane in self.shared_lanes and p < self.shared_prefix:
                q = min(end, self.shared_prefix)
            else:
                q = end
            out.append((p, q - p, s))
            p = q
        return out

    def kv_np(self, layer: int, lane: int, pos0: int, n: int, kv: int) -> np.ndarray:
        parts = [kv_block_np(self.seed, layer, s, p, m, self.num_kv_heads, kv,
                             self.k_outliers, self.v_outliers)
                 for (p, m, s) in self.segments(lane, pos0, n)]
        x = np.concatenate(parts, axis=0) if parts else np.zeros((0, self.num_kv_heads, HEAD_DIM), np.uint16)
        return self._apply_needle_np(x, layer, lane, pos0, n, kv)

    def kv_torch(self, layer: int, lane: int, pos0: int, n: int, kv: int, device):
        import torch
        parts = [kv_block_torch(self.seed, layer, s, p, m, self.num_kv_heads, kv, device,
                                self.k_outliers, self.v_outliers)
                 for (p, m, s) in self.segments(lane, pos0, n)]
        x = torch.cat(parts, 0) if parts else torch.zeros((0, self.num_kv_heads, HEAD_DIM),
                                                          dtype=torch.bfloat16, device=device)
        if self.needle is not None and lane == 0:
            npos = self.needle["pos"]
            if pos0 <= npos < pos0 + n:
                row = self.needle_rows_np(layer)[kv]
                x[npos - pos0] = torch.from_numpy(row.astype(np.int16)).view(torch.bfloat16).to(device)
        return x

    def q_np(self, layer: int, lane: int, pos0: int, n: int) -> np.ndarray:
        return q_block_np(self.seed, layer, lane, pos0, n, self.num_q_heads)

    def q_torch(self, layer: int, lane: int, pos0: int, n: int, device):
        return q_block_torch(self.seed, layer, lane, pos0, n, self.num_q_heads, device)

    # --- needle: key = 3*sqrt(D)*q_hat of the group's first query head, value one-hot.
    def needle_rows_np(self, layer: int) -> np.ndarray:
        """bf16 bits ``[2][Hkv][256]``: the needle's K and V rows (lane 0)."""
        assert self.needle is not None
        qpos = self.seq_len[0] - 1
        q = bf16_bits_to_f32_np(self.q_np(layer, 0, qpos, 1)[0]).astype(np.float64)
        k = np.zeros((self.num_kv_heads, HEAD_DIM), np.float64)
        v = np.zeros((self.num_kv_heads, HEAD_DIM), np.float64)
        for g in range(self.num_kv_heads):
            qg = q[g * self.group]
            k[g] = 3.0 * np.sqrt(HEAD_DIM) * qg / np.sqrt(np.dot(qg, qg))
            v[g, self.needle["onehot"][g]] = 1.0
        return np.stack([f32_to_bf16_bits_np(k.astype(np.float32)),
                         f32_to_bf16_bits_np(v.astype(np.float32))])

    def _apply_needle_np(self, x, layer, lane, pos0, n, kv):
        if self.needle is None or lane != 0:
            return x
        npos = self.needle["pos"]
        if pos0 <= npos < pos0 + n:
            x = x.copy()
            x[npos - pos0] = self.needle_rows_np(layer)[kv]
        return x


def kv_np_parallel(wl: "Workload", layer: int, lane: int, pos0: int, n: int, kv: int, chunk: int = 4096,
                   threads: Optional[int] = None) -> np.ndarray:
    """``wl.kv_np`` computed in parallel chunks of tokens (numpy releases the GIL)."""
    import concurrent.futures as cf
    import os
    if n <= chunk:
        return wl.kv_np(layer, lane, pos0, n, kv)
    threads = threads or max(1, min(32, os.cpu_count() or 1))
    starts = list(range(pos0, pos0 + n, chunk))
    with cf.ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda p: wl.kv_np(layer, lane, p, min(chunk, pos0 + n - p), kv), starts))
    return np.concatenate(parts, 0)


def _table(lanes_pages: List[np.ndarray], max_pages: int) -> np.ndarray:
    t = np.full((len(lanes_pages), max_pages), -1, dtype=np.int32)
    for b, p in enumerate(lanes_pages):
        t[b, :len(p)] = p
    return t


def tiny_decode(seed: int = 0) -> Workload:
    """1 layer, 1 KV head, GQA 4, one 256-token lane on 4 pages scattered in a 16-page pool."""
    perm = permutation(seed, 16)
    return Workload("tiny_decode_256", 1, 1, 4, [256], _table([perm[:4]], 4), 16, seed=seed)


def batched_decode_27b(seed: int = 0, lanes: int = 8, ctx: int = 40960, layers: int = 16) -> Workload:
    """16 layers x 4 KV heads x 256, 24 query heads, 8 lanes at 40,960 tokens, permuted pool."""
    per = ctx // PAGE_TOKENS
    perm = permutation(seed, lanes * per)
    return Workload(f"decode_27b_{lanes}x{ctx}", layers, 4, 24, [ctx] * lanes,
                    _table([perm[b * per:(b + 1) * per] for b in range(lanes)], per), lanes * per,
                    seed=seed)


def mixed_shared_27b(seed: int = 0, long_ctx: int = 131072, short_ctx: int = 4096, shared: int = 2048,
                     n_short: int = 8, layers: int = 16) -> Workload:
    """1 long lane + 8 short lanes whose first `shared` tokens live on the same physical pages."""
    lp, sp, shp = long_ctx // 64, short_ctx // 64, shared // 64
    total = lp + shp + n_short * (sp - shp)
    perm = permutation(seed, total)
    long_pages = perm[:lp]
    shared_pages = perm[lp:lp + shp]
    rows = [long_pages]
    off = lp + shp
    for _ in range(n_short):
        rows.append(np.concatenate([shared_pages, perm[off:off + sp - shp]]))
        off += sp - shp
    return Workload(f"mixed_shared_27b_{long_ctx}+{n_short}x{short_ctx}", layers, 4, 24,
                    [long_ctx] + [short_ctx] * n_short, _table(rows, lp), total, window=64,
                    seed=seed, v_outliers=False, shared_prefix=shared,
                    shared_lanes=tuple(range(1, n_short + 1)))


def chunked_prefill_27b(seed: int = 0, prefix: int = 65536, chunk: int = 1024, layers: int = 16) -> Workload:
    """One lane: `prefix` tokens already paged, then a `chunk`-token prefill chunk."""
    n = prefix + chunk
    pages = (n + 63) // 64
    perm = permutation(seed, pages)
    return Workload(f"prefill_27b_{prefix}+{chunk}", layers, 4, 24, [n], _table([perm], pages), pages,
                    seed=seed, prefill_chunk=chunk)


def needle_131k(seed: int = 0, ctx: int = 131072) -> Workload:
    """1 layer, 4 KV heads, 24 query heads, 131,072 tokens, one needle at a seeded position."""
    pages = ctx // 64
    perm = permutation(seed, pages)
    pos = seeded_int(seed, 1, ctx - 64)          # a closed page, not the last one
    onehot = [seeded_int(seed, 2 + g, HEAD_DIM) for g in range(4)]
    return Workload(f"needle_{ctx}", 1, 4, 24, [ctx], _table([perm], pages), pages, seed=seed,
                    needle={"pos": pos, "onehot": onehot})
