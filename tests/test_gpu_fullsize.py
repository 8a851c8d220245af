"""GPU vs oracle at the full sizes of the five workloads, in the launch configuration the
benchmark uses: whole outputs where the oracle can afford them, sampled (lane, layer) pairs
and query rows otherwise.  Inputs for the oracle are regenerated on the host."""
import numpy as np
import pytest

import oracle
from compressed_paged_kv_quant_gb300 import synth
from oracle_side import TWO_BIT, LaneCache, assert_close, gpu_block

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HQ, BF = oracle.FMT_HQ2B, oracle.FMT_BF16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_paged_kv_quant_gb300 import build
    build.build()


def _dw(wl, fmt, fill=0xA5):
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    return DeviceWorkload(wl, fmt, "cuda", fill)


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _decode_step(dw, layers, fused=True):
    """One decode step over `layers`.  fused=True is the benchmark's launch configuration: every
    layer's kvq_decode_step (append + decode kernels overlapped by programmatic dependent
    launch) back to back, captured once in a CUDA graph and replayed, with one workspace shared
    by the layers and one output buffer per layer.  fused=False: kv_quant_append then
    paged_decode_attn, eagerly, with a garbage-filled workspace before each layer."""
    layers = list(layers)
    ws, out = dw.decode_buffers()
    ws.view(torch.int32).fill_(-1)
    outs = torch.empty((len(layers),) + tuple(out.shape), dtype=out.dtype, device=out.device)
    qkv = []
    for l in layers:
        k, v = dw.step_kv(l)
        qkv.append((dw.step_q(l), k, v))
    if fused:
        dw.decode(layers[0], qkv[0][0], ws, outs[0])   # read-only warm-up: first-call set-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i, l in enumerate(layers):
                q, k, v = qkv[i]
                dw.decode_step(l, q, k, v, ws, outs[i])
        g.replay()
    else:
        for i, l in enumerate(layers):
            q, k, v = qkv[i]
            dw.append_step(l, k, v)
            ws.view(torch.int32).fill_(-1)
            dw.decode(l, q, ws, outs[i])
    torch.cuda.synchronize()
    host = outs.cpu().numpy()
    return {l: host[i] for i, l in enumerate(layers)}


def _check_lane(dw, wl, fmt, layer, lane, got, pages=(0, 1)):
    oc = LaneCache(wl, fmt, layer, lane)
    n = wl.seq_len[lane]
    q = wl.q_np(layer, lane, n - 1, 1)
    ref = oc.attend(q, [n - 1], wl.window, dw.sm_scale)[0]
    err = assert_close(got, ref, what=f"{wl.name} layer {layer} lane {lane}")
    # page bytes of this lane/layer: GPU pool block == oracle block
    pool = dw.cache.pool
    pb = oracle.page_bytes(oracle.geom(fmt, wl.num_layers, wl.num_kv_heads, wl.num_q_heads))
    npg = (n + 63) // 64
    for p in list(pages) + [npg - 1]:
        phys = int(wl.page_table[lane, p])
        blk = pool[phys * pb:(phys + 1) * pb].cpu().numpy()
        for h in range(wl.num_kv_heads):
            for kv in (0, 1):
                g_blk = gpu_block(blk, pb, wl.num_kv_heads, fmt, 0, layer, h, kv)
                np.testing.assert_array_equal(g_blk, oc.block(p, h, kv), err_msg=f"page {p} head {h} kv {kv}")
    if fmt in TWO_BIT:
        ring = _u16(dw.cache.ring).reshape(wl.lanes, wl.num_layers, wl.num_kv_heads, 64, 256)
        np.testing.assert_array_equal(ring[lane, layer], oc.ring[0, 0])
    return err, oc


def test_batched_decode_27b_sampled():
    """8 lanes x 40,960 tokens, 16 layers x 4 KV heads, 24 q heads, through the step the
    benchmark times (every layer's kvq_decode_step in one CUDA graph, the step token closing page
    639 of every lane); four (layer, lane) pairs compared in full against the oracle, with the
    bytes of pages 0, 1 and the page the step closed, and the ring."""
    wl = synth.batched_decode_27b()
    dw = _dw(wl, HQ, fill=None)
    dw.fill_history([n - 1 for n in wl.seq_len])
    outs = _decode_step(dw, range(wl.num_layers))
    assert dw.cache.read_status() == 0
    for layer, lane in ((0, 3), (5, 0), (10, 5), (15, 7)):
        _check_lane(dw, wl, HQ, layer, lane, outs[layer][lane])
    for l in range(wl.num_layers):
        assert np.all(np.isfinite(outs[l]))


def test_batched_decode_27b_separate_calls_sampled():
    """The same workload on two layers through kv_quant_append then paged_decode_attn (separate
    calls, no kernel overlap); two (layer, lane) pairs against the oracle."""
    wl = synth.batched_decode_27b(layers=2)
    dw = _dw(wl, HQ, fill=None)
    dw.fill_history([n - 1 for n in wl.seq_len])
    outs = _decode_step(dw, range(wl.num_layers), fused=False)
    assert dw.cache.read_status() == 0
    for layer, lane in ((0, 6), (1, 2)):
        _check_lane(dw, wl, HQ, layer, lane, outs[layer][lane])


@pytest.mark.parametrize("fmt", [oracle.FMT_HQ2B_HAD, oracle.FMT_HQ2B_TOK, oracle.FMT_FP8])
def test_batched_decode_27b_format_variants_sampled(fmt):
    """The 27B decode workload's per-layer sizes (8 lanes x 40,960 tokens, 4 KV heads, 24 q
    heads; two layers) in the rotated, per-token-K and FP8 formats, through the step the
    benchmark times for them (kvq_decode_step in a CUDA graph); two (layer, lane) pairs compared
    in full."""
    wl = synth.batched_decode_27b(layers=2)
    dw = _dw(wl, fmt, fill=None)
    dw.fill_history([n - 1 for n in wl.seq_len])
    outs = _decode_step(dw, range(wl.num_layers))
    assert dw.cache.read_status() == 0
    for layer, lane in ((0, 3), (1, 7)):
        _check_lane(dw, wl, fmt, layer, lane, outs[layer][lane])


def test_mixed_shared_prefix_window64_sampled():
    """1 x 131,072 + 8 x 4,096 tokens whose first 2,048 live on 32 shared pages; W = 64; every
    layer's kvq_decode_step in one CUDA graph; four (layer, lane) pairs against the oracle."""
    wl = synth.mixed_shared_27b()
    dw = _dw(wl, HQ, fill=None)
    dw.fill_history([n - 1 for n in wl.seq_len])
    outs = _decode_step(dw, range(wl.num_layers))
    assert dw.cache.read_status() == 0
    _check_lane(dw, wl, HQ, 0, 0, outs[0][0])
    _check_lane(dw, wl, HQ, 9, 4, outs[9][4])
    _check_lane(dw, wl, HQ, 15, 1, outs[15][1])
    # the short lanes read the shared pages in place: lanes 2..8 never appended them
    _check_lane(dw, wl, HQ, 0, 8, outs[0][8], pages=(0, 31, 32))


def _prefill_rows(chunk, group, extra=16, seed=0):
    """Query rows of a chunk that meet every tile boundary of the tensor-core prefill (a CTA
    takes 128 // group consecutive queries of one GQA group), the first and last rows, and a
    seeded sample of the rest."""
    qt = 128 // group
    rows = {0, 1, chunk - 2, chunk - 1}
    for t in range(qt, chunk, qt):
        rows |= {t - 1, t}
    rng = np.random.default_rng(seed)
    rows |= set(int(x) for x in rng.choice(chunk, size=extra, replace=False))
    return sorted(r for r in rows if 0 <= r < chunk)


def test_chunked_prefill_65536_plus_1024_sampled():
    """A 1,024-token chunk over a 65,536-token compressed prefix; garbage-filled workspace; on
    layers 0, 7 and 15, every query row at a CTA tile boundary plus the first, last and a seeded
    sample (> 100 rows of 24 heads) against the oracle."""
    wl = synth.chunked_prefill_27b()
    dw = _dw(wl, HQ, fill=None)
    prefix, chunk = 65536, 1024
    layers = (0, 7, 15)
    rows = _prefill_rows(chunk, wl.group)
    assert len(rows) >= 64
    dw.fill_history([prefix], layers=layers)
    ws, out = dw.prefill_buffers(chunk)
    for l in layers:
        k = wl.kv_torch(l, 0, prefix, chunk, 0, "cuda")
        v = wl.kv_torch(l, 0, prefix, chunk, 1, "cuda")
        dw.append(l, [0], [prefix], [chunk], k, v)
        ws.view(torch.int32).fill_(-1)
        q = wl.q_torch(l, 0, prefix, chunk, "cuda")
        dw.prefill(l, q, [prefix], [chunk], [0], ws, out)
        got = out.cpu().numpy()
        assert dw.cache.read_status() == 0
        oc = LaneCache(wl, HQ, l, 0)
        qh = wl.q_np(l, 0, prefix, chunk)[rows]
        ref = oc.attend(qh, [prefix + i for i in rows], 0, dw.sm_scale)
        assert_close(got[rows], ref, what=f"prefill layer {l}")
        assert np.all(np.isfinite(got))


@pytest.mark.parametrize("fmt", [oracle.FMT_HQ2B_TOK, oracle.FMT_HQ2B_HAD, oracle.FMT_FP8])
def test_chunked_prefill_65536_plus_1024_format_variants_sampled(fmt):
    """The 1,024-token chunk over the 65,536-token prefix (one layer) in the per-token-K, rotated
    and FP8 formats on the tensor-core prefill: the first and last rows, the rows at both sides
    of every fourth CTA tile boundary, and a seeded sample, against the oracle."""
    wl = synth.chunked_prefill_27b(layers=1)
    dw = _dw(wl, fmt, fill=None)
    prefix, chunk = 65536, 1024
    rows = _prefill_rows(chunk, wl.group, extra=8)[::2]
    if fmt == oracle.FMT_HQ2B_HAD:
        # the oracle's rotated format applies a dense 256 x 256 Hadamard matrix to every key of
        # every query: three rows (first, middle, last) keep it to about a minute
        rows = [0, 777, chunk - 1]
    dw.fill_history([prefix])
    ws, out = dw.prefill_buffers(chunk)
    k = wl.kv_torch(0, 0, prefix, chunk, 0, "cuda")
    v = wl.kv_torch(0, 0, prefix, chunk, 1, "cuda")
    dw.append(0, [0], [prefix], [chunk], k, v)
    ws.view(torch.int32).fill_(-1)
    dw.prefill(0, wl.q_torch(0, 0, prefix, chunk, "cuda"), [prefix], [chunk], [0], ws, out)
    got = out.cpu().numpy()
    assert dw.cache.read_status() == 0
    oc = LaneCache(wl, fmt, 0, 0)
    ref = oc.attend(wl.q_np(0, 0, prefix, chunk)[rows], [prefix + i for i in rows], 0, dw.sm_scale)
    assert_close(got[rows], ref, what=f"prefill fmt={fmt}")
    assert np.all(np.isfinite(got))


def test_prefill_prefix_over_three_splits_in_full():
    """A 200-token chunk over a 20,000-token prefix: the keys span three 8,192-key splits, so
    every query's result is a merge of three or more split partials; every row and head against
    the oracle (one layer, 2 KV heads, GQA 6)."""
    prefix, chunk = 20000, 200
    n = prefix + chunk
    wl = synth.Workload("prefill_3splits", 1, 2, 12, [n], np.arange((n + 63) // 64, dtype=np.int32)[None, :][:, ::-1]
                        .copy(), (n + 63) // 64, window=0, seed=11)
    dw = _dw(wl, HQ)
    dw.fill_history([n])
    ws, out = dw.prefill_buffers(chunk)
    ws.view(torch.int32).fill_(-1)
    q = wl.q_torch(0, 0, prefix, chunk, "cuda")
    dw.prefill(0, q, [prefix], [chunk], [0], ws, out)
    got = out.cpu().numpy()
    assert dw.cache.read_status() == 0
    oc = LaneCache(wl, HQ, 0, 0)
    ref = oc.attend(wl.q_np(0, 0, prefix, chunk), [prefix + i for i in range(chunk)], 0, dw.sm_scale)
    assert_close(got, ref, what="prefill over three splits")


def test_needle_131072_hq_and_bf16():
    """One needle key (3 sqrt(D) q^) with a one-hot value among 131,072 tokens: the oracle
    finds it top-1 for the defining heads, and both GPU formats keep it (out ~ e_j)."""
    wl = synth.needle_131k()
    n = wl.seq_len[0]
    got = {}
    for fmt in (HQ, BF):
        dw = _dw(wl, fmt, fill=None)
        dw.fill_history([n - 1])
        outs = _decode_step(dw, [0])
        assert dw.cache.read_status() == 0
        got[fmt] = outs[0][0]
        err, oc = _check_lane(dw, wl, fmt, 0, 0, got[fmt], pages=(wl.needle["pos"] // 64,))
        q = wl.q_np(0, 0, n - 1, 1)[0]
        for g in range(wl.num_kv_heads):
            j = g * wl.group
            _, top1, st = oracle.attend(oc.g, 0, oc.pool, oc.ring, 0, oc.pt[0], 0, n, j, q[j], n, dw.sm_scale)
            assert st == 0 and top1 == wl.needle["pos"]
            one = wl.needle["onehot"][g]
            assert got[fmt][j][one] > 0.99
            assert np.max(np.abs(np.delete(got[fmt][j], one))) < 1e-2
        del dw
        torch.cuda.empty_cache()
    # on the defining heads the two formats agree within the attention tolerance
    for g in range(4):
        j = g * wl.group
        assert_close(got[HQ][j], got[BF][j], atol=2e-3, rtol=1e-3, what="hq vs bf16 needle head")
