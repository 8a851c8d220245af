"""Codec study: the 2-bit format against its Walsh-Hadamard-rotated variant on the outlier data.

Runs the CPU oracle only (no GPU) and prints one markdown table.  For each format, one KV head
of N tokens of the seeded synthetic data (K ~ N(0,1) with every 16th channel x4, V ~ N(0,1)
with every 64th token x6) is appended through ``oracle.append``; then, against the
unquantized bf16 rows in double:
  * relative L2 error of the reconstructed keys and values (rows dequantized from the pages,
    turned back with H for the rotated format),
  * RMS error of the attention logits (sm_scale q.k) and relative L2 error of the attention
    output of Q queries x G heads (oracle.decode, window 0, keys of the open page exact),
  * the fraction of queries whose highest-scoring key is the exact one's.
Usage: python -m oracle.codec_study [N] [Q]
"""
from __future__ import annotations

import sys

import numpy as np

import oracle
from compressed_paged_kv_quant_gb300 import synth


def _f(u):
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def study(n_tokens: int = 8192, n_queries: int = 16, seed: int = 0):
    G = 6
    pages = (n_tokens + 63) // 64
    table = np.arange(pages, dtype=np.int32)[None, :]
    wl = synth.Workload("codec_study", 1, 1, G, [n_tokens], table, pages, seed=seed)
    k = wl.kv_np(0, 0, 0, n_tokens, 0)            # [n][1][256] bf16 bits
    v = wl.kv_np(0, 0, 0, n_tokens, 1)
    kx, vx = _f(k[:, 0]), _f(v[:, 0])
    H = None
    rows = []
    for fmt, name in ((oracle.FMT_HQ2B, "2-bit (K per channel, V per token)"),
                      (oracle.FMT_HQ2B_HAD, "2-bit over Walsh-Hadamard-rotated K, V")):
        g = oracle.geom(fmt, 1, 1, G)
        pb = oracle.page_bytes(g)
        pool = np.zeros(pages * pb, np.uint8)
        ring = np.zeros((1, 1, 1, 64, 256), np.uint16)
        assert oracle.append(g, 0, pool, ring, table, 1, [0], [n_tokens], [0], k, v) == 0
        closed = (n_tokens // 64) * 64
        kh, vh = np.zeros((closed, 256)), np.zeros((closed, 256))
        for t in range(closed):
            base = (t // 64) * pb
            kb, vb = pool[base:base + 4608], pool[base + 4608:base + 9216]
            s = t % 64
            kh[t] = oracle.dequant_k_row(kb[s * 64:(s + 1) * 64], kb[4096:].view(np.uint16))
            vh[t] = oracle.dequant_v_row(vb[s * 64:(s + 1) * 64], vb[4096 + 8 * s:4096 + 8 * s + 8].view(np.uint16))
            if fmt == oracle.FMT_HQ2B_HAD:
                kh[t], vh[t] = oracle.hadamard_f64(kh[t]), oracle.hadamard_f64(vh[t])
        ek = np.linalg.norm(kh - kx[:closed]) / np.linalg.norm(kx[:closed])
        ev = np.linalg.norm(vh - vx[:closed]) / np.linalg.norm(vx[:closed])
        lerr, oerr, top = [], [], 0
        for qi in range(n_queries):
            q = synth.q_block_np(seed + 1, 0, qi, n_tokens - 1, 1, G)       # [1][G][256]
            out, st = oracle.decode(g, 0, pool, ring, 0, table, 1, [n_tokens], q, 0.0625)
            assert st == 0
            for j in range(G):
                qq = _f(q[0, j])
                exact = 0.0625 * (kx @ qq)
                approx = 0.0625 * (np.vstack([kh, kx[closed:]]) @ qq)
                lerr.append(np.sqrt(np.mean((approx - exact) ** 2)))
                w = np.exp(exact - exact.max())
                ref = (w @ vx) / w.sum()
                oerr.append(np.linalg.norm(out[0, j] - ref) / np.linalg.norm(ref))
                top += int(np.argmax(approx) == np.argmax(exact))
        rows.append((name, ek, ev, float(np.mean(lerr)), float(np.mean(oerr)), top / (n_queries * G)))
    lines = [f"| format ({n_tokens} tokens, {n_queries} x {G} queries, seed {seed}) | K rel. L2 | V rel. L2 | "
             "logit RMS error | output rel. L2 | top-1 kept |", "|---|---|---|---|---|---|"]
    for r in rows:
        lines.append(f"| {r[0]} | {r[1]:.3f} | {r[2]:.3f} | {r[3]:.3f} | {r[4]:.3f} | {100 * r[5]:.0f} % |")
    return "\n".join(lines)


if __name__ == "__main__":
    n = int(sys.argv[1]) if len(sys.argv) > 1 else 8192
    qn = int(sys.argv[2]) if len(sys.argv) > 2 else 16
    print(study(n, qn))
