"""GPU path vs the CPU oracle on small, seeded workloads that span several pages, splits and
ragged tails: bit-exact pool and ring bytes after append, attention within tolerance."""
import numpy as np
import pytest

import oracle
from compressed_paged_kv_quant_gb300 import synth
from oracle_side import assert_close, host_kv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HQ, BF, HAD, TOK, FP8 = oracle.FMT_HQ2B, oracle.FMT_BF16, oracle.FMT_HQ2B_HAD, oracle.FMT_HQ2B_TOK, oracle.FMT_FP8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_paged_kv_quant_gb300 import build
    build.build()


def _dw(wl, fmt, fill=0xA5, scales=(0.0, 0.0)):
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    return DeviceWorkload(wl, fmt, "cuda", fill, k_scale=scales[0], v_scale=scales[1])


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _custom(lens, L=1, H=1, Hq=4, seed=0, window=0, extra_pages=3, k_out=True, v_out=True):
    pages = [(n + 63) // 64 for n in lens]
    total = sum(pages) + extra_pages
    perm = synth.permutation(seed, total, salt=7)
    rows, off = [], 0
    for p in pages:
        rows.append(perm[off:off + p])
        off += p
    mp = max(max(pages), 1)
    t = np.full((len(lens), mp), -1, np.int32)
    for b, r in enumerate(rows):
        t[b, :len(r)] = r
    return synth.Workload(f"custom_{lens}", L, H, Hq, list(lens), t, total, window=window, seed=seed,
                          k_outliers=k_out, v_outliers=v_out)


def _oracle_full(wl, fmt, layers=None, fill=0xA5, scales=(0.0, 0.0)):
    """Oracle pool/ring with the workload's own geometry and page table, every lane filled."""
    g = oracle.geom(fmt, wl.num_layers, wl.num_kv_heads, wl.num_q_heads, *scales)
    pool = np.full(wl.pool_pages * oracle.page_bytes(g), fill, np.uint8)
    ring = np.zeros((wl.lanes, wl.num_layers, wl.num_kv_heads, 64, 256), np.uint16)
    for layer in (range(wl.num_layers) if layers is None else layers):
        for b, n in enumerate(wl.seq_len):
            k = host_kv(wl, layer, b, 0, n, 0)
            v = host_kv(wl, layer, b, 0, n, 1)
            pt = np.ascontiguousarray(wl.page_table[b:b + 1])
            ring_b = np.ascontiguousarray(ring[b:b + 1])
            gl = g
            st = oracle.append(gl, layer, pool, ring_b, pt, 1, [0], [n], [0], k, v)
            assert st == 0
            ring[b] = ring_b[0]
    return g, pool, ring


def _gpu_fill(dw, chunking="one"):
    wl = dw.wl
    rng = np.random.default_rng(1)
    for layer in range(wl.num_layers):
        if chunking == "one":
            dw.fill_history(wl.seq_len, layers=[layer], chunk=1 << 20)
            continue
        # batched ragged calls: every call appends a random count to every lane
        pos = [0] * wl.lanes
        while any(p < n for p, n in zip(pos, wl.seq_len)):
            lanes, starts, counts, ks, vs = [], [], [], [], []
            for b, n in enumerate(wl.seq_len):
                if pos[b] >= n:
                    continue
                c = 1 if chunking == "tokens" else int(rng.integers(1, 150))
                c = min(c, n - pos[b])
                lanes.append(b)
                starts.append(pos[b])
                counts.append(c)
                ks.append(wl.kv_torch(layer, b, pos[b], c, 0, "cuda"))
                vs.append(wl.kv_torch(layer, b, pos[b], c, 1, "cuda"))
                pos[b] += c
            dw.append(layer, lanes, starts, counts, torch.cat(ks), torch.cat(vs))
    torch.cuda.synchronize()


def test_device_generator_matches_host():
    wl = synth.tiny_decode()
    for kv in (0, 1):
        a = _u16(wl.kv_torch(0, 0, 0, 256, kv, "cuda"))
        np.testing.assert_array_equal(a, wl.kv_np(0, 0, 0, 256, kv))
    np.testing.assert_array_equal(_u16(wl.q_torch(0, 0, 255, 1, "cuda")), wl.q_np(0, 0, 255, 1))


@pytest.mark.parametrize("window", [0, 64])
def test_tiny_decode_bytes_and_output(window):
    """The tiny decode step: 1 layer, 1 KV head, GQA 4, 256 tokens on 4 scattered pages."""
    wl = synth.tiny_decode()
    dw = _dw(wl, HQ)
    _gpu_fill(dw)
    g, pool, ring = _oracle_full(wl, HQ)
    np.testing.assert_array_equal(dw.cache.pool.cpu().numpy(), pool)
    np.testing.assert_array_equal(_u16(dw.cache.ring), ring.ravel())
    q = dw.step_q(0)
    ws, out = dw.decode_buffers()
    ws.view(torch.int32).fill_(-1)                       # garbage: NaN bit patterns everywhere
    dw.decode(0, q, ws, out, window=window)
    assert dw.cache.read_status() == 0
    ref, st = oracle.decode(g, 0, pool, ring, window, wl.page_table, 1, wl.seq_len, wl.q_np(0, 0, 255, 1),
                            dw.sm_scale)
    assert st == 0
    assert_close(out.cpu().numpy(), ref, what="tiny decode")


@pytest.mark.parametrize("chunking", ["one", "tokens", "random"])
def test_append_bytes_independent_of_chunking(chunking):
    wl = _custom([300, 129, 64, 5], L=2, H=2, Hq=4)
    dw = _dw(wl, HQ)
    _gpu_fill(dw, chunking)
    assert dw.cache.read_status() == 0
    g, pool, ring = _oracle_full(wl, HQ)
    np.testing.assert_array_equal(dw.cache.pool.cpu().numpy(), pool)
    np.testing.assert_array_equal(_u16(dw.cache.ring), ring.ravel())


@pytest.mark.parametrize("chunking", ["one", "tokens", "random"])
def test_rotated_append_bytes(chunking):
    """The Walsh-Hadamard-rotated format: pool and ring bytes equal the oracle's, whatever the
    call sizes (the rotated page close and V rows, the unrotated ring)."""
    wl = _custom([300, 129, 64, 5], L=2, H=2, Hq=4)
    dw = _dw(wl, HAD)
    _gpu_fill(dw, chunking)
    assert dw.cache.read_status() == 0
    g, pool, ring = _oracle_full(wl, HAD)
    np.testing.assert_array_equal(dw.cache.pool.cpu().numpy(), pool)
    np.testing.assert_array_equal(_u16(dw.cache.ring), ring.ravel())


@pytest.mark.parametrize("chunking", ["one", "tokens", "random"])
def test_per_token_k_append_bytes(chunking):
    """The per-token-K format: every K row coded at append by the V rule, no page close; pool
    and ring bytes equal the oracle's whatever the call sizes."""
    wl = _custom([300, 129, 64, 5], L=2, H=2, Hq=4)
    dw = _dw(wl, TOK)
    _gpu_fill(dw, chunking)
    assert dw.cache.read_status() == 0
    g, pool, ring = _oracle_full(wl, TOK)
    np.testing.assert_array_equal(dw.cache.pool.cpu().numpy(), pool)
    np.testing.assert_array_equal(_u16(dw.cache.ring), ring.ravel())


@pytest.mark.parametrize("chunking,scales", [("one", (0.0, 0.0)), ("random", (0.0, 0.0)), ("random", (0.25, 3.0))])
def test_fp8_append_bytes(chunking, scales):
    """The FP8 E4M3 format: every page byte equals the oracle's E4M3 of x / scale."""
    wl = _custom([300, 129, 64, 5], L=2, H=2, Hq=4)
    dw = _dw(wl, FP8, scales=scales)
    _gpu_fill(dw, chunking)
    assert dw.cache.read_status() == 0
    g, pool, _ = _oracle_full(wl, FP8, scales=scales)
    np.testing.assert_array_equal(dw.cache.pool.cpu().numpy(), pool)


@pytest.mark.parametrize("scales", [(0.0, 0.0), (0.25, 3.0)])
def test_fp8_decode_with_scales(scales):
    wl = _custom(LENS, L=1, H=2, Hq=12)
    dw = _dw(wl, FP8, scales=scales)
    _gpu_fill(dw)
    g, pool, _ = _oracle_full(wl, FP8, scales=scales)
    ws, out = dw.decode_buffers()
    ws.view(torch.int32).fill_(0x7FC00001)
    dw.decode(0, dw.step_q(0), ws, out)
    qh = np.concatenate([wl.q_np(0, b, n - 1, 1) for b, n in enumerate(LENS)])
    ref, st = oracle.decode(g, 0, pool, None, 0, wl.page_table, wl.lanes, LENS, qh, dw.sm_scale)
    assert st == 0
    assert_close(out.cpu().numpy(), ref, what=f"fp8 decode scales={scales}")
    assert dw.cache.read_status() == 0


def test_bf16_append_bytes():
    wl = _custom([200, 64, 1], L=2, H=2, Hq=4)
    dw = _dw(wl, BF)
    _gpu_fill(dw, "random")
    g, pool, _ = _oracle_full(wl, BF)
    np.testing.assert_array_equal(dw.cache.pool.cpu().numpy(), pool)


LENS = [1, 63, 64, 65, 700, 1500, 2049, 3000]


@pytest.mark.parametrize("fmt,window", [(HQ, 0), (HQ, 64), (HQ, 17), (BF, 0), (HAD, 0), (HAD, 64), (HAD, 17),
                                        (TOK, 0), (TOK, 64), (TOK, 17), (FP8, 0)])
def test_decode_ragged_lanes(fmt, window):
    wl = _custom(LENS, L=2, H=2, Hq=12, window=window)
    dw = _dw(wl, fmt)
    _gpu_fill(dw)
    g, pool, ring = _oracle_full(wl, fmt)
    ws, out = dw.decode_buffers()
    for layer in range(2):
        ws.view(torch.int32).fill_(0x7FC00001)
        q = dw.step_q(layer)
        dw.decode(layer, q, ws, out)
        qh = np.concatenate([wl.q_np(layer, b, n - 1, 1) for b, n in enumerate(LENS)])
        ref, st = oracle.decode(g, layer, pool, ring if fmt not in (BF, FP8) else None, window, wl.page_table, wl.lanes,
                                LENS, qh, dw.sm_scale)
        assert st == 0
        assert_close(out.cpu().numpy(), ref, what=f"decode fmt={fmt} W={window} layer={layer}")
    assert dw.cache.read_status() == 0


@pytest.mark.parametrize("fmt", [HQ, BF, FP8])
@pytest.mark.parametrize("G", [1, 2, 3, 5, 7, 8])
def test_decode_group_sizes(G, fmt):
    """Every GQA group size the kernels take (heads padded to 8 in the tensor-core tiles)."""
    lens = [333, 1100]
    wl = _custom(lens, L=1, H=2, Hq=2 * G)
    dw = _dw(wl, fmt)
    _gpu_fill(dw)
    g, pool, ring = _oracle_full(wl, fmt)
    ws, out = dw.decode_buffers()
    ws.view(torch.int32).fill_(-1)
    dw.decode(0, dw.step_q(0), ws, out)
    qh = np.concatenate([wl.q_np(0, b, n - 1, 1) for b, n in enumerate(lens)])
    ref, _ = oracle.decode(g, 0, pool, ring if fmt == HQ else None, 0, wl.page_table, 2, lens, qh, dw.sm_scale)
    assert_close(out.cpu().numpy(), ref, what=f"fmt={fmt} G={G}")
    assert dw.cache.read_status() == 0


def test_decode_zero_length_lane_gives_zeros():
    wl = _custom([130, 0, 64], L=1, H=1, Hq=4)
    dw = _dw(wl, HQ)
    dw.fill_history([130, 0, 64])
    ws, out = dw.decode_buffers()
    out.fill_(7.0)
    q = torch.cat([wl.q_torch(0, b, max(n - 1, 0), 1, "cuda") for b, n in enumerate(wl.seq_len)])
    dw.decode(0, q, ws, out)
    assert dw.cache.read_status() == 0
    assert torch.all(out[1] == 0)
    assert torch.all(torch.isfinite(out))


@pytest.mark.parametrize("fmt,window,scales", [(HQ, 0, None), (HQ, 64, None), (BF, 0, None), (TOK, 0, None),
                                               (TOK, 64, None), (HAD, 0, None), (HAD, 64, None),
                                               (FP8, 0, None), (FP8, 0, (0.25, 3.0))])
def test_prefill_chunks(fmt, window, scales):
    """Causal chunks over a compressed prefix: (prefix, chunk) = (300, 100), (0, 70), (1000, 1100);
    every compressed format on the tensor-core prefill, BF16 on the CUDA-core split kernel."""
    scales = scales or (0.0, 0.0)
    prefix, chunk = [300, 0, 1000], [100, 70, 1100]
    layers = range(2)
    if fmt == HAD:
        # the oracle turns every key and value of every query back with a dense 256 x 256
        # Hadamard matrix: smaller chunks on one layer keep it to seconds
        prefix, chunk = [128, 0, 260], [40, 24, 72]
        layers = [1]
    lens = [p + c for p, c in zip(prefix, chunk)]
    wl = _custom(lens, L=2, H=2, Hq=12, window=window)
    dw = _dw(wl, fmt, scales=scales)
    _gpu_fill(dw)            # prefix and chunk K/V appended (the chunk's own K/V first, as required)
    g, pool, ring = _oracle_full(wl, fmt, scales=scales)
    rows = sum(chunk)
    ws, out = dw.prefill_buffers(rows)
    offs = np.cumsum([0] + chunk[:-1]).tolist()
    for layer in layers:
        ws.view(torch.int32).fill_(-1)
        q = torch.cat([wl.q_torch(layer, b, prefix[b], chunk[b], "cuda") for b in range(3)])
        dw.prefill(layer, q, prefix, chunk, offs, ws, out)
        qh = np.concatenate([wl.q_np(layer, b, prefix[b], chunk[b]) for b in range(3)])
        ref, st = oracle.prefill(g, layer, pool, ring if fmt not in (BF, FP8) else None, window, wl.page_table, 3, prefix,
                                 chunk, offs, lens, qh, dw.sm_scale)
        assert st == 0
        assert_close(out.cpu().numpy(), ref, what=f"prefill fmt={fmt} W={window} layer={layer}")
    assert dw.cache.read_status() == 0


def test_device_status_flags():
    from compressed_paged_kv_quant_gb300 import kvq
    wl = _custom([200], L=1, H=1, Hq=4)
    dw = _dw(wl, HQ)
    dw.fill_history([200])
    torch.cuda.synchronize()
    assert dw.cache.read_status() == 0
    # a page id outside the pool inside the length
    saved = dw.page_table.clone()
    dw.page_table[0, 1] = wl.pool_pages + 5
    ws, out = dw.decode_buffers()
    dw.decode(0, dw.step_q(0), ws, out)
    assert dw.cache.read_status() & kvq.STATUS_PAGE_OOB
    dw.page_table.copy_(saved)
    dw.cache.clear_status()
    # a NaN input is flagged and not quantized
    k = wl.kv_torch(0, 0, 200, 1, 0, "cuda")
    k[0, 0, 3] = float("nan")
    v = wl.kv_torch(0, 0, 200, 1, 1, "cuda")
    dw.append(0, [0], [199], [1], k, v)
    assert dw.cache.read_status() & kvq.STATUS_BAD_INPUT
    dw.cache.clear_status()
    # a count beyond max_new
    kvq.kv_quant_append(dw.g, 0, dw.cache.pool, dw.cache.ring, dw.page_table,
                        torch.tensor([0], dtype=torch.int32, device="cuda"),
                        torch.tensor([5], dtype=torch.int32, device="cuda"),
                        torch.tensor([0], dtype=torch.int32, device="cuda"), 2, k.repeat(5, 1, 1),
                        v.repeat(5, 1, 1), dw.cache.status)
    assert dw.cache.read_status() & kvq.STATUS_BAD_LEN


def test_flat_attention_over_131072_keys_keeps_full_mass():
    """q = 0 gives a flat softmax over 131,072 keys: the output must be the mean of the
    values.  With an accumulator rounded to bf16 after every add the weights would sum to
    0.001953 ("Half the Cache", accumulator table); the FP32 two-level path keeps 1.0."""
    n = 131072
    wl = _custom([n], L=1, H=1, Hq=4, extra_pages=0)
    dw = _dw(wl, HQ)
    _gpu_fill(dw)
    g, pool, ring = _oracle_full(wl, HQ)
    q = torch.zeros((1, 4, 256), dtype=torch.bfloat16, device="cuda")
    ws, out = dw.decode_buffers()
    dw.decode(0, q, ws, out)
    o = out.cpu().numpy()
    ref, _ = oracle.decode(g, 0, pool, ring, 0, wl.page_table, 1, [n], np.zeros((1, 4, 256), np.uint16), 1.0)
    # 2e-4 on unit-scale values: the FP32 partials lose nothing measurable (a bf16 running sum
    # would be off by ~1.0); what remains is the tensor core's own FP32 accumulation within a
    # warp's run of pages, well inside the 2e-3 + 1e-3 |ref| contract
    assert_close(o, ref, atol=2e-4, rtol=2e-4, what="flat 131072")


@pytest.mark.parametrize("fmt,window", [(HQ, 64), (HQ, 32), (HQ, 0), (TOK, 0), (HAD, 32), (FP8, 0)])
def test_decode_step_equals_append_then_decode(fmt, window):
    """kvq_decode_step (for the 2-bit format: the append, then the decode kernels overlapped with
    it by programmatic dependent launch; for the other formats: the two calls in stream order)
    leaves the same pool and ring bytes as kv_quant_append followed by paged_decode_attn and the
    same outputs, bit for bit, over 70 steps with page closes on every lane and one lane that
    appends nothing on odd steps; windows 64, 32 and 0 put the closing page's keys in the ring,
    split, and in the codes."""
    from compressed_paged_kv_quant_gb300 import kvq
    steps = 70
    final = [700, 1500, 130, 3001]
    wl = _custom(final, L=2, H=2, Hq=12, seed=5, window=window)
    dev = "cuda"
    A, B = _dw(wl, fmt), _dw(wl, fmt)
    # lane 3 skips odd steps, so its history stops steps // 2 tokens short of its final length
    base = [n - steps for n in final[:3]] + [final[3] - steps // 2]
    for dw in (A, B):
        dw.fill_history(base)
    torch.cuda.synchronize()
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=dev)
    ws_a, out_a = A.decode_buffers()
    ws_b, out_b = B.decode_buffers()
    ws_b.view(torch.int32).fill_(-1)
    pos = list(base)
    for s in range(steps):
        layer = s % 2
        n_new = [1, 1, 1, int(s % 2 == 0)]
        start = list(pos)
        seq = [p + n for p, n in zip(pos, n_new)]
        rows = [b for b in range(4) if n_new[b]]
        off = [0] * 4
        for i, b in enumerate(rows):
            off[b] = i
        k = torch.cat([wl.kv_torch(layer, b, pos[b], 1, 0, dev) for b in rows])
        v = torch.cat([wl.kv_torch(layer, b, pos[b], 1, 1, dev) for b in rows])
        q = torch.cat([wl.q_torch(layer, b, max(seq[b] - 1, 0), 1, dev) for b in range(4)])
        sp, nn, to, sl = i32(start), i32(n_new), i32(off), i32(seq)
        kvq.kv_quant_append(A.g, layer, A.cache.pool, A.cache.ring, A.page_table, sp, nn, to, 1, k, v, A.cache.status)
        kvq.paged_decode_attn(A.g, layer, A.cache.pool, A.cache.ring, window, A.page_table, sl, max(final), q,
                              A.sm_scale, ws_a, out_a, A.cache.status)
        kvq.kvq_decode_step(B.g, layer, B.cache.pool, B.cache.ring, window, B.page_table, sp, nn, to, k, v, sl,
                            max(final), q, B.sm_scale, ws_b, out_b, B.cache.status)
        torch.cuda.synchronize()
        assert A.cache.read_status() == 0 and B.cache.read_status() == 0, f"step {s}"
        a, b = out_a.cpu().numpy(), out_b.cpu().numpy()
        assert np.array_equal(a, b), f"step {s}: max diff {np.abs(a - b).max()}"
        pos = seq
    assert pos == final
    assert torch.equal(A.cache.pool, B.cache.pool)
    assert (A.cache.ring is None) == (B.cache.ring is None)              # the FP8 format has no ring
    assert A.cache.ring is None or torch.equal(A.cache.ring, B.cache.ring)


@pytest.mark.parametrize("call,fmt", [("decode", HQ), ("decode", TOK), ("decode", HAD), ("decode", FP8),
                                      ("decode", BF), ("step", HQ), ("prefill", HQ), ("prefill", BF)])
def test_lane_longer_than_max_seq_len_is_skipped(call, fmt):
    """A lane whose seq_len exceeds the host bound max_seq_len (but not the page table) is
    flagged BAD_LEN and skipped by every kernel of the call: no byte past the workspace the
    bound sizes is touched, and the other lanes' results stay those of the oracle."""
    from compressed_paged_kv_quant_gb300 import kvq
    lens, bound = [200, 300], 256           # lane 1: 300 tokens, inside its 5-page table row
    wl = _custom(lens, L=1, H=2, Hq=12)
    dw = _dw(wl, fmt)
    _gpu_fill(dw)
    g, pool, ring = _oracle_full(wl, fmt)
    ring_o = ring if fmt not in (BF, FP8) else None
    guard = 1 << 16
    if call == "prefill":
        need = kvq.prefill_workspace_bytes(dw.g, 2, bound)
    else:
        need = kvq.decode_workspace_bytes(dw.g, 2, bound)
    buf = torch.full((need + guard,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = buf[:need]
    out = torch.full((2, 12, 256), 7.0, dtype=torch.float32, device="cuda")
    if call == "prefill":
        q = torch.cat([wl.q_torch(0, b, n - 1, 1, "cuda") for b, n in enumerate(lens)])
        kvq.paged_prefill_attn(dw.g, 0, dw.cache.pool, dw.cache.ring, 0, dw.page_table,
                               dw._i32([n - 1 for n in lens]), dw._i32([1, 1]), dw._i32([0, 1]), 1, dw.seq_len,
                               bound, q, dw.sm_scale, ws, out, dw.cache.status)
    elif call == "step":
        # the step's token is the lane's last one, already in the cache: append it again
        k, v = dw.step_kv(0)
        kvq.kvq_decode_step(dw.g, 0, dw.cache.pool, dw.cache.ring, 0, dw.page_table, dw.step_start, dw.step_n,
                            dw.step_off, k, v, dw.seq_len, bound, dw.step_q(0), dw.sm_scale, ws, out,
                            dw.cache.status)
    else:
        kvq.paged_decode_attn(dw.g, 0, dw.cache.pool, dw.cache.ring, 0, dw.page_table, dw.seq_len, bound,
                              dw.step_q(0), dw.sm_scale, ws, out, dw.cache.status)
    torch.cuda.synchronize()
    assert dw.cache.read_status() & kvq.STATUS_BAD_LEN
    assert torch.all(buf[need:] == 0x5A), "bytes past the workspace were written"
    qh = wl.q_np(0, 0, lens[0] - 1, 1)
    ref, st = oracle.decode(g, 0, pool, ring_o, 0, wl.page_table[:1], 1, lens[:1], qh, dw.sm_scale)
    assert st == 0
    assert_close(out[:1].cpu().numpy(), ref, what=f"{call} fmt={fmt}: the valid lane")
