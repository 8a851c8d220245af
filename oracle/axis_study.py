"""Axis study: which axis to scale K by, on the page's 3-level grid and on this format's 4-level
grids.  TEST INFRASTRUCTURE (a study run on the CPU, numpy only); nothing on the GPU path uses it.

"Half the Cache, Twice the Context", section "What the cache loses when you round it", Block 2,
measures two things on synthetic caches shaped like real ones (K: every 16th channel x4;
V: every 64th token x6; N = 4,096 tokens x D = 128 dims, numpy Generator seed 7):
  * the relative L2 reconstruction error of the cache when each token row (per-token) or each
    channel column (per-channel) gets its own scale, at 8, 4 and 2 bits, with a symmetric
    round-to-nearest grid of 2^(bits-1) - 1 positive levels (2 bits: the three levels -1, 0, 1);
  * needle recovery: 200 trials of one key set 0.5 logits above every other score (its
    direction is the query's), K per-channel and V per-token at 8/8, 4/4, 3/3 and 2/2 bits:
    how often the top-1 key changes, the mean of the largest attention-weight error, and the
    mean relative L2 error of the attention output.
`page_tables()` recomputes both with the same seed and draw order, so it must print the page's
numbers (a pin of this code).  `four_level_tables()` asks the same questions of the grids this
format actually stores (2 bits, four levels):
  * K rule: per channel over a 64-token page, s = fp16(max|x| / 3), k^ = s (2c - 3);
  * V rule: per token over 128 dims (one half row), z = fp16(min), s = fp16((max - min) / 3),
    v^ = z + c s; used for V and, in the per-token-K format, for K.
Both are the rules of the CPU oracle's format definition, written here in float64 with the
fp16 rounding of the stored scales (numpy's binary16 conversion, round-to-nearest-even).

Usage: python -m oracle.axis_study
"""
from __future__ import annotations

import numpy as np

N, D, TRIALS, MARGIN, SEED = 4096, 128, 200, 0.5, 7


# ----------------------------------------------------------------------------- the page's grid
def sym_quant(x: np.ndarray, bits: int, axis: int) -> np.ndarray:
    """Symmetric grid with 2^(bits-1) - 1 positive levels; one scale per slice along `axis`
    (axis 1: one scale per token row; axis 0: one per channel column)."""
    top = 2 ** (bits - 1) - 1
    amax = np.max(np.abs(x), axis=axis, keepdims=True)
    step = np.where(amax == 0, 1.0, amax / top)
    return np.clip(np.round(x / step), -top, top) * step


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _outlier_k(rng, n=N):
    k = rng.normal(0.0, 1.0, (n, D))
    k[:, ::16] *= 4.0
    return k


def _needle_trials(rng, kq, vq, trials=TRIALS):
    """The needle experiment with quantizers kq(K) and vq(V); returns (flips, mean max weight
    error, mean output relative L2)."""
    flips, werr, oerr = 0, 0.0, 0.0
    for _ in range(trials):
        q = rng.normal(0.0, 1.0, D)
        k = _outlier_k(rng)
        v = rng.normal(0.0, 1.0, (N, D))
        at = N // 2
        k[at] = q * ((k @ q).max() + MARGIN) / (q @ q)
        w = _softmax(k @ q)
        sq = kq(k) @ q
        wq = _softmax(sq)
        flips += int(np.argmax(sq) != at)
        werr += np.max(np.abs(wq - w))
        ref = w @ v
        oerr += np.linalg.norm(wq @ vq(v) - ref) / np.linalg.norm(ref)
    return flips, werr / trials, oerr / trials


def _softmax(s):
    e = np.exp(s - s.max())
    return e / e.sum()


def page_tables():
    """Block 2 as printed: ([(cache, bits, per_token, per_channel)], [(kb, vb, flips, werr, oerr)])."""
    rng = np.random.default_rng(SEED)
    k = _outlier_k(rng)
    v = rng.normal(0.0, 1.0, (N, D))
    v[::64, :] *= 6.0
    recon = [(name, bits, _rel(sym_quant(x, bits, 1), x), _rel(sym_quant(x, bits, 0), x))
             for name, x in (("K", k), ("V", v)) for bits in (8, 4, 2)]
    needle = []
    for kb, vb in ((8, 8), (4, 4), (3, 3), (2, 2)):
        f, we, oe = _needle_trials(rng, lambda x, b=kb: sym_quant(x, b, 0), lambda x, b=vb: sym_quant(x, b, 1))
        needle.append((kb, vb, f, we, oe))
    return recon, needle


# ----------------------------------------------------------------------------- this format's grids
def _f16(x):
    return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)


def k_rule_per_channel(x: np.ndarray) -> np.ndarray:
    """The K rule: per channel over each 64-token page, symmetric 4 levels s (2c - 3)."""
    out = np.empty_like(x)
    for p0 in range(0, x.shape[0], 64):
        blk = x[p0:p0 + 64]
        s = _f16(np.max(np.abs(blk), axis=0) / 3.0)
        safe = np.where(s == 0, 1.0, s)
        c = np.where(s == 0, 2, np.clip(np.rint((blk / safe + 3.0) * 0.5), 0, 3))
        out[p0:p0 + 64] = s * (2 * c - 3)
    return out


def v_rule(x: np.ndarray, axis: int = 1) -> np.ndarray:
    """The V rule along `axis` (1: per token over the row's 128 dims; 0: per channel over each
    64-token page): z = fp16(min), s = fp16((max - min) / 3), four levels z + c s."""
    if axis == 0:
        return np.concatenate([v_rule(x[p0:p0 + 64].T, 1).T for p0 in range(0, x.shape[0], 64)])
    z = _f16(np.min(x, axis=1, keepdims=True))
    s = _f16((np.max(x, axis=1, keepdims=True) - np.min(x, axis=1, keepdims=True)) / 3.0)
    safe = np.where(s == 0, 1.0, s)
    c = np.where(s == 0, 0, np.clip(np.rint((x - z) / safe), 0, 3))
    return z + c * s


def rotated(rule):
    """`rule` applied to rows turned by the orthonormal Sylvester Hadamard matrix of the row
    length (H = H^T = H^-1), the result turned back: the rotated variant's order of steps."""
    from scipy.linalg import hadamard

    def q(x):
        h = hadamard(x.shape[1]).astype(np.float64) / np.sqrt(x.shape[1])
        return rule(x @ h) @ h
    return q


def four_level_tables(trials: int = TRIALS):
    """(reconstruction rows, needle rows) on this format's 2-bit grids, same synthetic caches."""
    rng = np.random.default_rng(SEED)
    k = _outlier_k(rng)
    v = rng.normal(0.0, 1.0, (N, D))
    v[::64, :] *= 6.0
    recon = [
        ("K", "per-channel (K rule, 64-token page)", _rel(k_rule_per_channel(k), k)),
        ("K", "per-token (V rule, 128 dims)", _rel(v_rule(k, 1), k)),
        ("V", "per-token (V rule, 128 dims)", _rel(v_rule(v, 1), v)),
        ("V", "per-channel (V rule, 64-token page)", _rel(v_rule(v, 0), v)),
        ("K", "per-channel after a Hadamard rotation", _rel(rotated(k_rule_per_channel)(k), k)),
        ("K", "per-token after a Hadamard rotation", _rel(rotated(v_rule)(k), k)),
    ]
    needle = []
    for name, kq in (("K per-channel (K rule)", k_rule_per_channel), ("K per-token (V rule)", v_rule),
                     ("K per-channel, rotated", rotated(k_rule_per_channel)), ("K per-token, rotated", rotated(v_rule))):
        f, we, oe = _needle_trials(np.random.default_rng(SEED + 1), kq, v_rule, trials)
        needle.append((name, f, trials, we, oe))
    return recon, needle


def main():
    recon, needle = page_tables()
    print("page grid (symmetric, 2^(bits-1)-1 levels each side), relative L2 of the cache:")
    print("| cache | bits | per-token | per-channel |\n|---|---|---|---|")
    for name, bits, pt, pc in recon:
        print(f"| {name} | {bits} | {pt:.3e} | {pc:.3e} |")
    print("\nneedle, margin 0.5, K per-channel / V per-token:")
    print("| K / V bits | top-1 flips | max w err | out rel-L2 |\n|---|---|---|---|")
    for kb, vb, f, we, oe in needle:
        print(f"| {kb}/{vb} | {f}/{TRIALS} | {we:.2e} | {oe:.2e} |")
    recon4, needle4 = four_level_tables()
    print("\nthis format's 2-bit grids (four levels), relative L2 of the cache:")
    print("| cache | axis (rule) | rel. L2 |\n|---|---|---|")
    for name, axis, e in recon4:
        print(f"| {name} | {axis} | {e:.3e} |")
    print("\nneedle, margin 0.5, V per-token (V rule), 2-bit grids:")
    print("| K axis | top-1 flips | max w err | out rel-L2 |\n|---|---|---|---|")
    for name, f, n, we, oe in needle4:
        print(f"| {name} | {f}/{n} | {we:.2e} | {oe:.2e} |")


if __name__ == "__main__":
    main()
