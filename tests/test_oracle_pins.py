"""Pins for the CPU oracle: each check ties the oracle to something other than itself --
numbers the pages print, closed forms, library routines (numpy / torch conversions), grid
round trips, invariants and brute force on tiny inputs."""
import numpy as np
import pytest
import torch

import oracle
from compressed_paged_kv_quant_gb300 import synth
from conftest import golden

F16_ONE_THIRD = 0x3555  # binary16 nearest to 1/3 = 0.333251953125


# ----------------------------------------------------------------------------- byte budget
def test_block1_sizing_table():
    """Half the Cache, Twice the Context -- Size the cache (Block 1 output)."""
    for name, L, H, D, kib, gib, gib8, reqs in golden("block1_kv_sizing.txt"):
        L, H, D = int(L), int(H), int(D)
        b = oracle.kv_bytes_per_token(L, H, D, 2)
        b8 = oracle.kv_bytes_per_token(L, H, D, 1)
        assert f"{b / 1024:.0f}" == kib, name
        assert f"{b * 131072 / 1024**3:.1f}" == gib, name
        assert f"{b8 * 131072 / 1024**3:.1f}" == gib8, name
        assert str(int(24.0 * 1024**3 / (b * 8192))) == reqs, name


def test_kv_format_numbers():
    """KV at 9 KB a token -- How it works (format table) and The numbers."""
    v = {k: float(x) for k, x in golden("kv_format_numbers.txt")}
    L, H = int(v["layers"]), int(v["kv_heads"])
    assert oracle.head_token_bytes(oracle.FMT_BF16) == v["bf16_bytes_per_head_token"]
    assert oracle.head_token_bytes(oracle.FMT_HQ2B) == v["hq2b_bytes_per_head_token"]
    assert v["hq2b_code_bytes_per_head_token"] * 8 == 2 * v["head_dim"]  # 2 bits x 256 dims
    assert v["hq2b_code_bytes_per_head_token"] + v["hq2b_meta_bytes_per_head_token"] == 72
    assert L * H * 2 == v["head_token_multiplier"]
    gh = oracle.geom(oracle.FMT_HQ2B, L, H, 24)
    gb = oracle.geom(oracle.FMT_BF16, L, H, 24)
    assert oracle.token_bytes(gh) == v["hq2b_bytes_per_token"]
    assert oracle.token_bytes(gb) == v["bf16_bytes_per_token"]
    # the general formula with 72/256 bytes per value gives the same 9,216
    assert oracle.kv_bytes_per_token(L, H, 256, 72 / 256) == v["hq2b_bytes_per_token"]
    assert round(oracle.token_bytes(gb) / oracle.token_bytes(gh), 2) == v["capacity_ratio"]
    assert 100.0 * v["hq2b_meta_bytes_per_head_token"] / v["hq2b_code_bytes_per_head_token"] == \
        v["metadata_overhead_percent"]
    assert oracle.page_bytes(gh) == v["page_tokens"] * v["hq2b_bytes_per_token"]
    n = v["lanes"] * v["context_tokens"]
    assert round(n * oracle.token_bytes(gh) / 1e9, 2) == v["hq2b_pool_GB"]
    assert round(n * oracle.token_bytes(gb) / 2**30, 1) == v["bf16_pool_GiB"]


# ----------------------------------------------------------------------------- accumulator model
def test_block3_flat_sum_table():
    """Half the Cache -- The cliff is in the accumulator (Block 3 printed table)."""
    for n, f32, f16, b16, two in golden("block3_flat_sum.txt"):
        n = int(n)
        assert f"{oracle.flat_sum(n, 'fp32'):.6f}" == f32
        assert f"{oracle.flat_sum(n, 'fp16'):.6f}" == f16
        assert f"{oracle.flat_sum(n, 'bf16'):.6f}" == b16
        assert f"{oracle.flat_sum(n, 'bf16', two_level=True):.6f}" == two


def test_flat_sum_floor_is_a_power_of_two():
    # a stuck accumulator stops where the term is half an ulp: 2^-(mantissa bits) * n
    assert oracle.flat_sum(1 << 12, "fp16") == 2.0 ** -1
    assert oracle.flat_sum(1 << 10, "bf16") == 2.0 ** -2


# ----------------------------------------------------------------------------- conversions
def _f16_numpy(x32):
    with np.errstate(over="ignore"):
        return np.asarray(x32, np.float32).astype(np.float16).view(np.uint16)


def test_f32_to_f16_matches_numpy():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    # concentrate on the binary16 range, subnormals, the overflow edge and exact ties
    near = (rng.integers(0x33000000, 0x47800000, 20000, dtype=np.uint64)).astype(np.uint32)
    ties = ((rng.integers(0x38800000 >> 13, 0x477FE000 >> 13, 4000, dtype=np.uint64) << 13)
            | 0x1000).astype(np.uint32)
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x477FE000, 0x477FF000, 0x477FEFFF,
                        0x33000000, 0x33000001, 0x387FC000, 0x38800000, 0x3EAAAAAB], np.uint32)
    allb = np.concatenate([bits, near, ties, special])
    x = allb.view(np.float32)
    x = x[np.isfinite(x)]
    got = np.array([oracle.f32_to_f16(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, _f16_numpy(x))


def test_f16_to_f32_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(v)) for v in h], np.float32)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.all(np.isnan(got[np.isnan(ref)]))


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(5000) * np.exp2(rng.integers(-20, 20, 5000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x], np.float32)
    np.testing.assert_array_equal(got, ref)


def test_one_third_in_binary16():
    assert oracle.f32_to_f16(np.float32(1.0) / np.float32(3.0)) == F16_ONE_THIRD
    assert oracle.f16_to_f32(F16_ONE_THIRD) == 0.333251953125


# ----------------------------------------------------------------------------- V quantizer
def _bf16(x):
    return synth.f32_to_bf16_bits_np(np.asarray(x, np.float32))


def _codes_of_row(codes):
    c = np.asarray(codes, np.uint8)
    return np.stack([(c >> (2 * j)) & 3 for j in range(4)], axis=-1).reshape(*c.shape[:-1], -1)


def test_v_grid_round_trip():
    rng = np.random.default_rng(3)
    for _ in range(200):
        x = np.empty(256)
        want = []
        for half in range(2):
            e = int(rng.integers(-8, 4))
            s = float(rng.choice([1, 3, 5, 7])) * 2.0 ** e
            z = float(rng.integers(-63, 64)) * 2.0 ** e
            c = rng.integers(0, 4, 128)
            c[rng.integers(0, 128)] = 0
            c[rng.integers(0, 128)] = 3
            c[c.argmin()] = 0
            x[half * 128:(half + 1) * 128] = z + c * s
            want.append((c, s, z))
        xb = _bf16(x)
        assert np.all(synth.bf16_bits_to_f32_np(xb) == x)  # the grid values are exact in bf16
        codes, meta = oracle.quant_v_row(xb)
        got = _codes_of_row(codes)
        for half, (c, s, z) in enumerate(want):
            np.testing.assert_array_equal(got[half * 128:(half + 1) * 128], c)
            assert oracle.f16_to_f32(meta[2 * half]) == s
            assert oracle.f16_to_f32(meta[2 * half + 1]) == z
        np.testing.assert_array_equal(oracle.dequant_v_row(codes, meta), x)


def test_v_worked_cases():
    # the needle's one-hot value row: a half {0,...,0,1} -> z = 0, s = fp16(1/3), c(1) = 3
    x = np.zeros(256)
    x[77] = 1.0
    codes, meta = oracle.quant_v_row(_bf16(x))
    assert meta[0] == F16_ONE_THIRD and meta[1] == 0
    assert meta[2] == 0 and meta[3] == 0            # an all-zero half: s = 0, z = 0
    c = _codes_of_row(codes)
    assert c[77] == 3 and c.sum() == 3
    v = oracle.dequant_v_row(codes, meta)
    assert v[77] == 3 * 0.333251953125 == 0.999755859375
    assert np.count_nonzero(v) == 1
    # a constant half: s = 0 -> every code 0 and v^ = fp16(constant)
    x = np.full(256, 0.1)
    codes, meta = oracle.quant_v_row(_bf16(x))
    assert meta[0] == 0 and np.all(codes == 0)
    assert oracle.dequant_v_row(codes, meta)[0] == np.float16(np.float32(_bf16_val(0.1)))


def _bf16_val(x):
    return float(synth.bf16_bits_to_f32_np(_bf16([x]))[0])


def test_v_code_bit_layout():
    # dim 4b+j of a row is code bits 2j..2j+1 of byte b
    for d in (0, 1, 2, 3, 4, 77, 127, 128, 129, 200, 255):
        x = np.zeros(256)
        x[d] = 1.0
        x[(d + 128) % 256] = -0.5 if d < 128 else 0.0
        codes, _ = oracle.quant_v_row(_bf16(x))
        assert codes[d // 4] >> (2 * (d % 4)) & 3 == 3
        others = np.delete(_codes_of_row(codes)[(d // 128) * 128:(d // 128 + 1) * 128], d % 128)
        assert np.all(others == 0)


def test_v_error_bound_random():
    rng = np.random.default_rng(4)
    for _ in range(100):
        xb = _bf16(rng.standard_normal(256) * rng.choice([0.01, 1, 30]))
        x = synth.bf16_bits_to_f32_np(xb).astype(np.float64)
        codes, meta = oracle.quant_v_row(xb)
        v = oracle.dequant_v_row(codes, meta)
        for half in range(2):
            sl = slice(half * 128, half * 128 + 128)
            s = oracle.f16_to_f32(meta[2 * half])
            mn, mx = x[sl].min(), x[sl].max()
            assert s == pytest.approx((mx - mn) / 3, rel=2**-10)
            slack = 2**-10 * (abs(mn) + abs(mx))
            assert np.max(np.abs(v[sl] - x[sl])) <= 0.5 * s * (1 + 2**-9) + slack
            c = _codes_of_row(codes)[sl]
            assert c[np.argmax(x[sl])] == 3 and c[np.argmin(x[sl])] == 0


# ----------------------------------------------------------------------------- K quantizer
def test_k_grid_round_trip():
    rng = np.random.default_rng(5)
    for _ in range(20):
        s = (rng.choice([1, 3, 5, 7], 256) * np.exp2(rng.integers(-8, 3, 256))).astype(np.float64)
        c = rng.integers(0, 4, (64, 256))
        c[rng.integers(0, 64, 256), np.arange(256)] = rng.choice([0, 3], 256)   # +-3s attained
        x = s[None, :] * (2 * c - 3)
        xb = _bf16(x)
        assert np.all(synth.bf16_bits_to_f32_np(xb) == x)
        codes, scales = oracle.quant_k_page(xb)
        np.testing.assert_array_equal(_codes_of_row(codes), c)
        np.testing.assert_array_equal([oracle.f16_to_f32(v) for v in scales], s)
        for t in range(0, 64, 7):
            np.testing.assert_array_equal(oracle.dequant_k_row(codes[t], scales), x[t])


def test_k_code_layout_is_token_by_channel():
    x = np.full((64, 256), 1.0)
    x[:, ::2] = -1.0
    t, d = 13, 201
    x[t, d] = 3.0 if d % 2 else -3.0   # channel d: max|x| = 3, so s = 1 and codes are {1,2} or 0/3
    codes, scales = oracle.quant_k_page(_bf16(x))
    c = _codes_of_row(codes)
    assert c.shape == (64, 256)
    assert c[t, d] == (3 if d % 2 else 0)
    assert oracle.f16_to_f32(scales[d]) == 1.0
    assert oracle.f16_to_f32(scales[d - 1]) == pytest.approx(1 / 3, rel=2**-10)
    # channels other than d: |x| = 1 everywhere -> s = fp16(1/3), codes 0 (x=-1) or 3 (x=+1)
    other = [dd for dd in range(256) if dd != d]
    for dd in other[:20]:
        assert np.all(c[:, dd] == (0 if dd % 2 == 0 else 3))


def test_k_zero_channel_and_sign_mirror():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 256)) * 2
    x[:, 5] = 0.0
    xb = _bf16(x)
    codes, scales = oracle.quant_k_page(xb)
    c = _codes_of_row(codes)
    assert scales[5] == 0 and np.all(c[:, 5] == 2)
    assert np.all(oracle.dequant_k_row(codes[0], scales)[5] == 0.0)
    # negating a page mirrors every code except at the exact ties x/s in {0, +-2}, where
    # half-even rounding is not sign-symmetric
    codes_n, scales_n = oracle.quant_k_page(xb ^ np.uint16(0x8000))
    cn = _codes_of_row(codes_n)
    xf = synth.bf16_bits_to_f32_np(xb).astype(np.float64)
    sf = np.array([oracle.f16_to_f32(v) for v in scales])[None, :]
    ok = (xf != 0) & (np.abs(xf) != 2 * sf)
    assert ok.sum() > 16000
    np.testing.assert_array_equal(cn[ok], 3 - c[ok])
    tie = (np.abs(xf) == 2 * sf) & (sf > 0)
    np.testing.assert_array_equal(c[tie], np.where(xf[tie] > 0, 2, 0))   # 2.5 -> 2, 0.5 -> 0
    np.testing.assert_array_equal(scales_n, scales)


def test_k_error_bound_random():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 256))
    x[:, ::16] *= 4
    xb = _bf16(x)
    xf = synth.bf16_bits_to_f32_np(xb).astype(np.float64)
    codes, scales = oracle.quant_k_page(xb)
    s = np.array([oracle.f16_to_f32(v) for v in scales])
    np.testing.assert_allclose(s, np.abs(xf).max(0) / 3, rtol=2**-10)
    k = np.stack([oracle.dequant_k_row(codes[t], scales) for t in range(64)])
    assert np.all(np.abs(k - xf) <= s[None, :] * (1 + 2**-8))


# ----------------------------------------------------------------------------- paged cache
def _fill(pool_pages, page_bytes, byte=0xA5):
    return np.full(pool_pages * page_bytes, byte, np.uint8)


def test_append_layout_spec():
    """Blocks [layer][kv_head][K,V] of 4,608 B; K: codes[64][64] + 256 fp16 scales,
    V: codes[64][64] + meta[64][4] fp16 ([s0, z0, s1, z1])."""
    L, H = 2, 3
    g = oracle.geom(oracle.FMT_HQ2B, L, H, 6)
    pb = oracle.page_bytes(g)
    assert pb == L * H * 2 * 4608
    pool = _fill(8, pb)
    ring = np.zeros((1, L, H, 64, 256), np.uint16)
    rng = np.random.default_rng(8)
    k = _bf16(rng.standard_normal((64, H, 256)))
    v = _bf16(rng.standard_normal((64, H, 256)))
    pt = np.array([[5]], np.int32)
    layer = 1
    # first 63 tokens: V rows are written, the K block is not (page still open)
    st = oracle.append(g, layer, pool, ring, pt, 1, [0], [63], [0], k, v)
    assert st == 0
    page = pool[5 * pb:6 * pb]
    for h in range(H):
        kb = page[((layer * H + h) * 2 + 0) * 4608:][:4608]
        vb = page[((layer * H + h) * 2 + 1) * 4608:][:4608]
        assert np.all(kb == 0xA5)
        for slot in (0, 31, 62):
            c, m = oracle.quant_v_row(v[slot, h])
            np.testing.assert_array_equal(vb[slot * 64:(slot + 1) * 64], c)
            np.testing.assert_array_equal(vb[4096 + slot * 8:4096 + slot * 8 + 8].view(np.uint16), m)
        np.testing.assert_array_equal(ring[0, layer, h, :63], k[:63, h])
    # token 63 closes the page: the K block is the page quantization of the 64 keys
    st = oracle.append(g, layer, pool, ring, pt, 1, [63], [1], [63], k, v)
    assert st == 0
    for h in range(H):
        kb = page[((layer * H + h) * 2 + 0) * 4608:][:4608]
        c, s = oracle.quant_k_page(k[:, h])
        np.testing.assert_array_equal(kb[:4096].reshape(64, 64), c)
        np.testing.assert_array_equal(kb[4096:].view(np.uint16), s)
    # layer 0 blocks and every other page are untouched
    assert np.all(page[:H * 2 * 4608] == 0xA5)
    mask = np.ones(pool.size, bool)
    mask[5 * pb:6 * pb] = False
    assert np.all(pool[mask] == 0xA5)


def _append_all(g, pool, ring, pt, lanes, lens, kvs, chunks):
    for b in range(lanes):
        k, v = kvs[b]
        pos = 0
        for n in chunks[b]:
            st = oracle.append(g, 0, pool, ring, pt[b:b + 1].copy(), 1, [pos], [n], [pos], k, v)
            assert st == 0
            pos += n
        assert pos == lens[b]


def test_append_chunk_invariance():
    g = oracle.geom(oracle.FMT_HQ2B, 1, 2, 4)
    pb = oracle.page_bytes(g)
    rng = np.random.default_rng(9)
    n = 300
    k = _bf16(rng.standard_normal((n, 2, 256)))
    v = _bf16(rng.standard_normal((n, 2, 256)))
    pt = np.array([[3, 0, 6, 1, 4]], np.int32)
    results = []
    for chunks in ([n], [1] * n, [5, 64, 1, 100, 63, 67], [129, 171]):
        pool = _fill(7, pb)
        ring = np.zeros((1, 1, 2, 64, 256), np.uint16)
        pos = 0
        for c in chunks:
            assert oracle.append(g, 0, pool, ring, pt, 1, [pos], [c], [pos], k, v) == 0
            pos += c
        results.append((pool.copy(), ring.copy()))
    for p, r in results[1:]:
        np.testing.assert_array_equal(p, results[0][0])
        np.testing.assert_array_equal(r, results[0][1])


def test_append_status_flags():
    g = oracle.geom(oracle.FMT_HQ2B, 1, 1, 1)
    pb = oracle.page_bytes(g)
    pool = _fill(2, pb)
    ring = np.zeros((1, 1, 1, 64, 256), np.uint16)
    k = np.zeros((130, 1, 256), np.uint16)
    v = np.zeros((130, 1, 256), np.uint16)
    assert oracle.append(g, 0, pool, ring, np.array([[0, 2]], np.int32), 1, [0], [70], [0], k, v) \
        == oracle.PAGE_OOB
    assert oracle.append(g, 0, pool, ring, np.array([[0, 1]], np.int32), 1, [0], [130], [0], k, v) \
        == oracle.LEN_GT_TABLE
    for bad in (0x7FC0, 0x7F80, 0x4780):   # NaN, +Inf, 65536
        k2 = k.copy()
        k2[3, 0, 9] = bad
        assert oracle.append(g, 0, pool, ring, np.array([[0, 1]], np.int32), 1, [0], [5], [0], k2, v) \
            == oracle.BAD_INPUT


# ----------------------------------------------------------------------------- attention
def _tiny_cache(fmt, n_tokens, H=1, Hq=4, seed=0, pages=None, pool_pages=None, window=0):
    rng = np.random.default_rng(seed)
    g = oracle.geom(fmt, 1, H, Hq)
    pb = oracle.page_bytes(g)
    npg = (n_tokens + 63) // 64
    if pages is None:
        pages = rng.permutation(pool_pages or npg + 3)[:npg]
    pt = np.array([pages], np.int32)
    pool = _fill(int(pool_pages or npg + 3), pb)
    ring = np.zeros((1, 1, H, 64, 256), np.uint16)
    x = rng.standard_normal((n_tokens, H, 256))
    x[:, :, ::16] *= 4
    k = _bf16(x)
    y = rng.standard_normal((n_tokens, H, 256))
    y[::64] *= 6
    v = _bf16(y)
    assert oracle.append(g, 0, pool, ring, pt, 1, [0], [n_tokens], [0], k, v) == 0
    return g, pool, ring, pt, k, v


def _dequant_all(g, pool, ring, pt, n, head, window=0):
    """Keys/values as the attention must see them, gathered through the page table."""
    pb = oracle.page_bytes(g)
    H = g.num_kv_heads
    K = np.zeros((n, 256))
    V = np.zeros((n, 256))
    open_start = (n // 64) * 64
    exact_from = min(n - window, open_start)
    for t in range(n):
        page = pool[pt[0, t // 64] * pb:][:pb]
        kb = page[(head * 2 + 0) * 4608:][:4608]
        vb = page[(head * 2 + 1) * 4608:][:4608]
        slot = t % 64
        if t >= exact_from:
            K[t] = synth.bf16_bits_to_f32_np(ring[0, 0, head, slot])
        else:
            K[t] = oracle.dequant_k_row(kb[slot * 64:(slot + 1) * 64], kb[4096:].view(np.uint16))
        V[t] = oracle.dequant_v_row(vb[slot * 64:(slot + 1) * 64], vb[4096 + slot * 8:][:8].view(np.uint16))
    return K, V


def _softmax_attn(q, K, V, scale):
    s = scale * (K @ q)
    w = np.exp(s - s.max())
    return (w / w.sum()) @ V


@pytest.mark.parametrize("n", [256, 200, 64, 1, 130])
def test_decode_brute_force_tiny(n):
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, n)
    q = _bf16(np.random.default_rng(11).standard_normal((1, 4, 256)))
    out, st = oracle.decode(g, 0, pool, ring, 0, pt, 1, [n], q, 0.0625)
    assert st == 0
    K, V = _dequant_all(g, pool, ring, pt, n, 0)
    for j in range(4):
        ref = _softmax_attn(synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64), K, V, 0.0625)
        np.testing.assert_allclose(out[0, j], ref, rtol=1e-12, atol=1e-12)


def test_decode_window_reads_exact_keys():
    n = 256
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, n)
    q = _bf16(np.random.default_rng(12).standard_normal((1, 4, 256)))
    out0, _ = oracle.decode(g, 0, pool, ring, 0, pt, 1, [n], q, 0.0625)
    out64, _ = oracle.decode(g, 0, pool, ring, 64, pt, 1, [n], q, 0.0625)
    K, V = _dequant_all(g, pool, ring, pt, n, 0, window=64)
    np.testing.assert_array_equal(K[-64:], synth.bf16_bits_to_f32_np(k[-64:, 0]))
    for j in range(4):
        qj = synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64)
        np.testing.assert_allclose(out64[0, j], _softmax_attn(qj, K, V, 0.0625), rtol=1e-12, atol=1e-12)
    assert np.max(np.abs(out64 - out0)) > 1e-6


def test_decode_bf16_format_is_exact_attention():
    n = 150
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_BF16, n, H=2, Hq=6)
    q = _bf16(np.random.default_rng(13).standard_normal((1, 6, 256)))
    out, st = oracle.decode(g, 0, pool, None, 0, pt, 1, [n], q, 0.0625)
    assert st == 0
    K = synth.bf16_bits_to_f32_np(k).astype(np.float64)
    V = synth.bf16_bits_to_f32_np(v).astype(np.float64)
    for j in range(6):
        qj = synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64)
        np.testing.assert_allclose(out[0, j], _softmax_attn(qj, K[:, j // 3], V[:, j // 3], 0.0625),
                                   rtol=1e-12, atol=1e-12)


def test_decode_zero_query_is_mean_of_values():
    n = 256
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, n)
    q = np.zeros((1, 4, 256), np.uint16)
    out, _ = oracle.decode(g, 0, pool, ring, 0, pt, 1, [n], q, 0.0625)
    _, V = _dequant_all(g, pool, ring, pt, n, 0)
    for j in range(4):
        np.testing.assert_allclose(out[0, j], V.mean(0), rtol=1e-13, atol=1e-14)


def test_decode_single_key_and_empty():
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, 64)
    q = _bf16(np.random.default_rng(14).standard_normal((1, 4, 256)))
    out, _ = oracle.decode(g, 0, pool, ring, 0, pt, 1, [1], q, 0.0625)
    _, V = _dequant_all(g, pool, ring, pt, 1, 0)
    np.testing.assert_array_equal(out[0, 0], V[0])
    out, _ = oracle.decode(g, 0, pool, ring, 0, pt, 1, [0], q, 0.0625)
    assert np.all(out == 0)


def test_decode_gqa_groups_and_page_relabelling():
    n = 192
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, n, H=2, Hq=6, pool_pages=5)
    qrow = _bf16(np.random.default_rng(15).standard_normal(256))
    q = np.tile(qrow, (1, 6, 1))
    out, _ = oracle.decode(g, 0, pool, ring, 0, pt, 1, [n], q, 0.0625)
    np.testing.assert_array_equal(out[0, 0], out[0, 2])      # same group, same query
    np.testing.assert_array_equal(out[0, 3], out[0, 5])
    assert np.max(np.abs(out[0, 0] - out[0, 3])) > 1e-3      # different KV heads
    # move every physical page to another slot of the pool: outputs are unchanged
    pb = oracle.page_bytes(g)
    relabel = np.array([4, 2, 0, 1, 3])
    pool2 = np.empty_like(pool)
    for old, new in enumerate(relabel):
        pool2[new * pb:(new + 1) * pb] = pool[old * pb:(old + 1) * pb]
    out2, _ = oracle.decode(g, 0, pool2, ring, 0, relabel[pt], 1, [n], q, 0.0625)
    np.testing.assert_array_equal(out, out2)


def test_decode_needle_is_top1():
    n = 640
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, n, seed=3)
    # rebuild with a needle key aligned to q at position 333 and a one-hot value
    rng = np.random.default_rng(16)
    qf = rng.standard_normal(256)
    q = _bf16(np.tile(qf, (1, 4, 1)))
    qd = synth.bf16_bits_to_f32_np(q[0, 0]).astype(np.float64)
    kx = synth.bf16_bits_to_f32_np(k).astype(np.float64)
    vx = synth.bf16_bits_to_f32_np(v).astype(np.float64)
    kx[333, 0] = 3 * 16 * qd / np.linalg.norm(qd)
    vx[333, 0] = 0
    vx[333, 0, 42] = 1
    pb = oracle.page_bytes(g)
    pool = _fill(pool.size // pb, pb)
    ring[:] = 0
    assert oracle.append(g, 0, pool, ring, pt, 1, [0], [n], [0], _bf16(kx), _bf16(vx)) == 0
    out, top1, st = oracle.attend(g, 0, pool, ring, 0, pt[0], 0, n, 0, q[0, 0], n, 0.0625)
    assert st == 0 and top1 == 333
    assert abs(out[42] - 0.999755859375) < 1e-6
    assert np.max(np.abs(np.delete(out, 42))) < 1e-6


def test_prefill_rows_are_causal_decodes():
    n = 200
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, n, H=1, Hq=2)
    q = _bf16(np.random.default_rng(17).standard_normal((40, 2, 256)))
    out, st = oracle.prefill(g, 0, pool, ring, 0, pt, 1, [160], [40], [0], [n], q, 0.0625)
    assert st == 0
    K, V = _dequant_all(g, pool, ring, pt, n, 0)
    for i in (0, 7, 39):
        p = 160 + i
        for j in range(2):
            qj = synth.bf16_bits_to_f32_np(q[i, j]).astype(np.float64)
            np.testing.assert_allclose(out[i, j], _softmax_attn(qj, K[:p + 1], V[:p + 1], 0.0625),
                                       rtol=1e-12, atol=1e-12)
    # a query past the cache is flagged
    _, st = oracle.prefill(g, 0, pool, ring, 0, pt, 1, [190], [11], [0], [n], q, 0.0625)
    assert st & oracle.BAD_LEN


def test_attend_flags_missing_page():
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B, 128)
    bad = pt.copy()
    bad[0, 1] = -1
    _, _, st = oracle.attend(g, 0, pool, ring, 0, bad[0], 0, 128, 0, np.zeros(256, np.uint16), 100, 0.0625)
    assert st & oracle.PAGE_OOB


def test_page_moves_round_trip_and_identity():
    """Gather then scatter back to the same ids is the identity; scatter to other ids moves each
    page's bytes unchanged (the pool is opaque bytes per page); a bad id is flagged."""
    g = oracle.geom(oracle.FMT_HQ2B, 2, 1, 4)
    pb = oracle.page_bytes(g)
    assert pb == 2 * 9216
    rng = np.random.default_rng(3)
    pool = rng.integers(0, 256, 7 * pb, dtype=np.uint8)
    ids = [5, 0, 3]
    arena, st = oracle.pages_gather(g, pool, ids)
    assert st == 0
    for i, p in enumerate(ids):
        assert np.array_equal(arena[i * pb:(i + 1) * pb], pool[p * pb:(p + 1) * pb])
    back = pool.copy()
    back[:] = 0
    assert oracle.pages_scatter(g, back, ids, arena) == 0
    for p in range(7):
        want = pool[p * pb:(p + 1) * pb] if p in ids else np.zeros(pb, np.uint8)
        assert np.array_equal(back[p * pb:(p + 1) * pb], want)
    _, st = oracle.pages_gather(g, pool, [1, 7])
    assert st == oracle.PAGE_OOB


def test_hadamard_rotation_matches_scipy_and_is_orthonormal():
    """The rotated variant's transform: the fast float transform and the double definition both
    equal scipy's Sylvester Hadamard matrix / 16 applied to x; H H = I; dot products survive."""
    from scipy.linalg import hadamard
    H = hadamard(256).astype(np.float64) / 16.0
    rng = np.random.default_rng(11)
    x = rng.standard_normal(256).astype(np.float32)
    ref = H @ x.astype(np.float64)
    assert np.allclose(oracle.hadamard_f64(x.astype(np.float64)), ref, atol=1e-12)
    assert np.allclose(oracle.fwht_f32(x), ref, rtol=0, atol=2e-6 * np.abs(x).max() * 16)
    y = oracle.hadamard_f64(oracle.hadamard_f64(x.astype(np.float64)))
    assert np.allclose(y, x, atol=1e-12)
    e = np.zeros(256)
    e[5] = 1.0
    assert np.array_equal(np.abs(oracle.hadamard_f64(e)), np.full(256, 1.0 / 16))
    q = rng.standard_normal(256)
    assert abs(q @ x - oracle.hadamard_f64(q) @ oracle.hadamard_f64(x.astype(np.float64))) < 1e-9


def test_rotated_format_attention_matches_unrotated_brute_force():
    """A tiny rotated-format cache: the oracle's attention equals brute force over keys and
    values dequantized from the codes and turned back with scipy's Hadamard matrix (one full
    page plus an open page read from the ring)."""
    from scipy.linalg import hadamard
    H = hadamard(256).astype(np.float64) / 16.0
    g = oracle.geom(oracle.FMT_HQ2B_HAD, 1, 1, 2)
    pb = oracle.page_bytes(g)
    n = 100
    rng = np.random.default_rng(5)
    kf = (rng.standard_normal((n, 256)) * np.where(np.arange(256) % 16 == 0, 4, 1)).astype(np.float32)
    vf = rng.standard_normal((n, 256)).astype(np.float32)
    bf = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)       # truncation is fine for inputs
    k, v = bf(kf), bf(vf)
    pool = np.zeros(3 * pb, np.uint8)
    ring = np.zeros((1, 1, 1, 64, 256), np.uint16)
    pt = np.array([[2, 0]], np.int32)
    assert oracle.append(g, 0, pool, ring, pt, 1, [0], [n], [0], k, v) == 0
    q = bf(rng.standard_normal((1, 2, 256)).astype(np.float32))
    out, st = oracle.decode(g, 0, pool, ring, 0, pt, 1, np.array([n], np.int32), q, 0.0625)
    assert st == 0
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    keys, vals = np.zeros((n, 256)), np.zeros((n, 256))
    kb = pool[2 * pb:2 * pb + 4608]
    vb = pool[2 * pb + 4608:2 * pb + 9216]
    scales = kb[4096:].view(np.uint16)
    for t in range(n):
        if t < 64:
            keys[t] = H @ oracle.dequant_k_row(kb[t * 64:(t + 1) * 64], scales)
        else:
            keys[t] = f(k[t])                                            # the open page: ring, exact
        blk = vb if t < 64 else pool[0 * pb + 4608:0 * pb + 9216]
        s = t % 64
        vals[t] = H @ oracle.dequant_v_row(blk[s * 64:(s + 1) * 64], blk[4096 + s * 8:4096 + s * 8 + 8].view(np.uint16))
    for j in range(2):
        sc = 0.0625 * (keys @ f(q[0, j]))
        w = np.exp(sc - sc.max())
        ref = (w @ vals) / w.sum()
        assert np.allclose(out[0, j], ref, atol=1e-10)


# ----------------------------------------------------------------------------- per-token-K format
def _grid_rows(rng, n, H):
    """bf16 rows whose every 128-dim half sits on a 4-level grid z + {0,1,2,3}*s with fp16-exact
    z and s, both ends present: the 2-bit V rule reproduces them exactly."""
    zs = np.array([-1.5, -0.75, 0.25, -3.0, 2.0])
    ss = np.array([1.0, 0.5, 0.25, 2.0, 0.125])
    x = np.zeros((n, H, 256))
    for t in range(n):
        for h in range(H):
            for half in range(2):
                z, s = zs[rng.integers(5)], ss[rng.integers(5)]
                c = rng.integers(0, 4, 128)
                c[0], c[1] = 0, 3
                rng.shuffle(c)
                x[t, h, 128 * half:128 * (half + 1)] = z + c * s
    assert np.array_equal(synth.bf16_bits_to_f32_np(_bf16(x)), x.astype(np.float32))
    return _bf16(x), x


@pytest.mark.parametrize("n,window", [(150, 0), (64, 0), (130, 17), (200, 64)])
def test_tok_format_on_grid_rows_is_exact_attention(n, window):
    """Per-token-K format, K and V rows already on the 2-bit grid: the quantization is lossless,
    so the oracle's attention equals exact softmax attention over the inputs (numpy, double)
    for every window, open page included."""
    rng = np.random.default_rng(21 + n)
    g = oracle.geom(oracle.FMT_HQ2B_TOK, 1, 2, 6)
    pb = oracle.page_bytes(g)
    npg = (n + 63) // 64
    pool = _fill(npg + 2, pb)
    ring = np.zeros((1, 1, 2, 64, 256), np.uint16)
    pt = np.array([rng.permutation(npg + 2)[:npg]], np.int32)
    k, kx = _grid_rows(rng, n, 2)
    v, vx = _grid_rows(rng, n, 2)
    assert oracle.append(g, 0, pool, ring, pt, 1, [0], [n], [0], k, v) == 0
    q = _bf16(rng.standard_normal((1, 6, 256)))
    out, st = oracle.decode(g, 0, pool, ring, window, pt, 1, [n], q, 0.0625)
    assert st == 0
    for j in range(6):
        qj = synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64)
        np.testing.assert_allclose(out[0, j], _softmax_attn(qj, kx[:, j // 3], vx[:, j // 3], 0.0625),
                                   rtol=1e-12, atol=1e-12)


def test_tok_format_bytes_follow_the_v_rule():
    """Per-token-K append: each K row's 64 code bytes and 8 meta bytes are the V rule applied to
    that key (the V quantizer is pinned above); the V block equals the plain format's; no
    page-close scales are written; the ring holds the last 64 keys."""
    n = 130
    g, pool, ring, pt, k, v = _tiny_cache(oracle.FMT_HQ2B_TOK, n, seed=3, pages=[2, 0, 4], pool_pages=5)
    gp, poolp, ringp, _, _, _ = _tiny_cache(oracle.FMT_HQ2B, n, seed=3, pages=[2, 0, 4], pool_pages=5)
    pb = oracle.page_bytes(g)
    for t in range(n):
        page = pool[pt[0, t // 64] * pb:][:pb]
        pagep = poolp[pt[0, t // 64] * pb:][:pb]
        s = t % 64
        codes, meta = oracle.quant_v_row(k[t, 0])
        assert np.array_equal(page[s * 64:(s + 1) * 64], codes)
        assert np.array_equal(page[4096 + s * 8:4096 + s * 8 + 8].view(np.uint16), meta)
        assert np.array_equal(page[4608:9216], pagep[4608:9216])
    assert np.array_equal(ring, ringp)
    # page 0 closed in the plain format (per-channel scales); the per-token format wrote meta rows
    assert not np.array_equal(pool[2 * pb + 4096:2 * pb + 4608], poolp[2 * pb + 4096:2 * pb + 4608])


def test_tok_format_reads_codes_of_the_open_page():
    """Window 0: the per-token-K format reads every key from its codes (the open page too),
    the plain format reads the open page from the ring; window 64 makes the last 64 keys exact
    in both, so the two formats then differ only in how the closed pages' keys were coded."""
    n = 100
    gt, poolt, ringt, pt, k, v = _tiny_cache(oracle.FMT_HQ2B_TOK, n, seed=4)
    q = _bf16(np.random.default_rng(15).standard_normal((1, 4, 256)))
    out, st = oracle.decode(gt, 0, poolt, ringt, 0, pt, 1, [n], q, 0.0625)
    assert st == 0
    pb = oracle.page_bytes(gt)
    K = np.zeros((n, 256))
    V = np.zeros((n, 256))
    for t in range(n):
        page = poolt[pt[0, t // 64] * pb:][:pb]
        s = t % 64
        K[t] = oracle.dequant_v_row(page[s * 64:(s + 1) * 64], page[4096 + s * 8:][:8].view(np.uint16))
        V[t] = oracle.dequant_v_row(page[4608 + s * 64:4608 + (s + 1) * 64], page[4608 + 4096 + s * 8:][:8].view(np.uint16))
    kx = synth.bf16_bits_to_f32_np(k[:, 0]).astype(np.float64)
    assert np.max(np.abs(K[64:] - kx[64:])) > 0.05                     # the open page is coded
    for j in range(4):
        qj = synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64)
        np.testing.assert_allclose(out[0, j], _softmax_attn(qj, K, V, 0.0625), rtol=1e-12, atol=1e-12)
    out64, _ = oracle.decode(gt, 0, poolt, ringt, 64, pt, 1, [n], q, 0.0625)
    K[n - 64:] = kx[n - 64:]
    for j in range(4):
        qj = synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64)
        np.testing.assert_allclose(out64[0, j], _softmax_attn(qj, K, V, 0.0625), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- axis study
def test_axis_study_reproduces_block2_tables():
    """Half the Cache -- What the cache loses when you round it (Block 2 printed tables): the
    study's page-grid part, same seed and draw order, prints the page's numbers."""
    from oracle import axis_study
    recon, needle = axis_study.page_tables()
    want = golden("block2_axis_needle.txt")
    want_r = [r[1:] for r in want if r[0] == "recon"]
    want_n = [r[1:] for r in want if r[0] == "needle"]
    assert [[c, str(b), f"{pt:.3e}", f"{pc:.3e}"] for c, b, pt, pc in recon] == want_r
    assert [[str(kb), str(vb), f"{f}/200", f"{we:.2e}", f"{oe:.2e}"] for kb, vb, f, we, oe in needle] == want_n


def test_axis_study_grids_are_the_oracle_quantizers():
    """The study's 4-level rules are the format's: on bf16 inputs the V rule equals the oracle's
    V row quantizer (both halves), and the K rule equals the oracle's page quantizer."""
    from oracle import axis_study
    rng = np.random.default_rng(31)
    x = rng.standard_normal((64, 256))
    x[:, ::16] *= 4
    x[::7] *= 6
    xb = _bf16(x)
    xf = synth.bf16_bits_to_f32_np(xb).astype(np.float64)
    for t in range(64):
        want = oracle.dequant_v_row(*oracle.quant_v_row(xb[t]))
        got = np.concatenate([axis_study.v_rule(xf[t:t + 1, :128], 1), axis_study.v_rule(xf[t:t + 1, 128:], 1)], 1)
        np.testing.assert_array_equal(got[0], want)
    codes, scales = oracle.quant_k_page(xb)
    want = np.stack([oracle.dequant_k_row(codes[t], scales) for t in range(64)])
    np.testing.assert_array_equal(axis_study.k_rule_per_channel(xf), want)


# ----------------------------------------------------------------------------- FP8 format
def test_e4m3_encoder_matches_torch_on_every_bf16():
    """The oracle's E4M3 encoder (written from the format definition) against torch's
    float8_e4m3fn conversion on every finite bf16 value below the rounding limit 464; past it
    the encoder saturates to +-448 (torch gives NaN there: the format has no infinity)."""
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = synth.bf16_bits_to_f32_np(u)
    fin = np.isfinite(x)
    mine = np.array([oracle.f32_to_e4m3(float(v)) for v in x[fin]], np.uint8)
    ref = torch.from_numpy(x[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    small = np.abs(x[fin]) < 464
    np.testing.assert_array_equal(mine[small], ref[small])
    big = ~small
    np.testing.assert_array_equal(mine[big], np.where(x[fin][big] < 0, 0xFE, 0x7E).astype(np.uint8))


def test_e4m3_decoder_matches_torch_on_every_byte():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_f64(int(v)) for v in b])
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    assert oracle.e4m3_to_f64(0x7E) == 448.0 and oracle.e4m3_to_f64(0x01) == 2.0 ** -9


@pytest.mark.parametrize("k_scale,v_scale", [(0.0, 0.0), (0.25, 3.0)])
def test_fp8_format_bytes_and_attention_follow_torch(k_scale, v_scale):
    """FP8 pages: every stored byte is torch's E4M3 of x / scale (fp32 division; in range here),
    and the oracle's attention equals brute force over torch's decoded values times the scale."""
    n, H, Hq = 150, 2, 6
    g = oracle.geom(oracle.FMT_FP8, 1, H, Hq, k_scale, v_scale)
    assert oracle.head_token_bytes(oracle.FMT_FP8) == 256
    pb = oracle.page_bytes(g)
    rng = np.random.default_rng(41)
    npg = (n + 63) // 64
    pt = np.array([rng.permutation(npg + 2)[:npg]], np.int32)
    pool = _fill(npg + 2, pb)
    xk = rng.standard_normal((n, H, 256))
    xk[:, :, ::16] *= 4
    xv = rng.standard_normal((n, H, 256))
    xv[::64] *= 6
    k, v = _bf16(xk), _bf16(xv)
    assert oracle.append(g, 0, pool, None, pt, 1, [0], [n], [0], k, v) == 0
    ks, vs = (k_scale or 1.0), (v_scale or 1.0)
    kq = torch.from_numpy(synth.bf16_bits_to_f32_np(k) / np.float32(ks)).to(torch.float8_e4m3fn)
    vq = torch.from_numpy(synth.bf16_bits_to_f32_np(v) / np.float32(vs)).to(torch.float8_e4m3fn)
    for t in range(n):
        page = pool[pt[0, t // 64] * pb:][:pb]
        s = t % 64
        for h in range(H):
            kb = page[(h * 2) * 16384 + s * 256:][:256]
            vb = page[(h * 2 + 1) * 16384 + s * 256:][:256]
            np.testing.assert_array_equal(kb, kq[t, h].view(torch.uint8).numpy())
            np.testing.assert_array_equal(vb, vq[t, h].view(torch.uint8).numpy())
    K = kq.to(torch.float64).numpy() * ks
    V = vq.to(torch.float64).numpy() * vs
    q = _bf16(rng.standard_normal((1, Hq, 256)))
    out, st = oracle.decode(g, 0, pool, None, 0, pt, 1, [n], q, 0.0625)
    assert st == 0
    for j in range(Hq):
        qj = synth.bf16_bits_to_f32_np(q[0, j]).astype(np.float64)
        np.testing.assert_allclose(out[0, j], _softmax_attn(qj, K[:, j // 3], V[:, j // 3], 0.0625),
                                   rtol=1e-12, atol=1e-12)


def test_fp8_format_saturates_and_flags_bad_input():
    g = oracle.geom(oracle.FMT_FP8, 1, 1, 4)
    pb = oracle.page_bytes(g)
    pool = np.zeros(pb, np.uint8)
    pt = np.array([[0]], np.int32)
    x = np.zeros((2, 1, 256), np.float32)
    x[0, 0, 0], x[0, 0, 1], x[0, 0, 2] = 1000.0, -600.0, 450.0
    k = _bf16(x)
    assert oracle.append(g, 0, pool, None, pt, 1, [0], [1], [0], k, k) == 0
    assert list(pool[:3]) == [0x7E, 0xFE, 0x7E]
    k2 = k.copy()
    k2[1, 0, 5] = 0x7F80                                 # +inf in bf16
    assert oracle.append(g, 0, pool, None, pt, 1, [1], [1], [1], k2, k2) == oracle.BAD_INPUT
