"""The C ABI library loads, exports every symbol include/kvq.h declares, sizes buffers as the
format says, and rejects bad calls on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from compressed_paged_kv_quant_gb300 import build, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return kvq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b([a-z_0-9]+)\s*\([^;{]*\)\s*;", src))


def test_every_declared_symbol_is_exported(L):
    declared = _declared()
    assert {"kv_quant_append", "paged_decode_attn", "paged_prefill_attn"} <= declared
    assert declared == set(kvq.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_build_targets_sm103(L):
    assert L.kvq_build_arch() == 103


def test_sizes_27b_geometry(L):
    gh = kvq.geom(kvq.FMT_HQ2B, 16, 4, 24)
    gb = kvq.geom(kvq.FMT_BF16, 16, 4, 24)
    assert kvq.token_bytes(gh) == 9216 and kvq.token_bytes(gb) == 65536
    assert kvq.page_bytes(gh) == 64 * 9216
    assert kvq.pool_pages(gh, 8 * 40960 * 9216) == 5120
    assert kvq.ring_bytes(gh, 8) == 8 * 16 * 4 * 64 * 256 * 2
    assert kvq.ring_bytes(gb, 8) == 0
    # decode: 8 lanes x 24 heads x 40 splits x (256 + 2) floats
    assert kvq.decode_workspace_bytes(gh, 8, 40960) >= 8 * 24 * 40 * 258 * 4


def test_two_bit_variants_share_the_layout(L):
    """The rotated and per-token-K formats keep the 72 B rows of the 2-bit format and its ring;
    the rotated one needs room for the rotated query in the decode workspace."""
    gh = kvq.geom(kvq.FMT_HQ2B, 16, 4, 24)
    for f in (kvq.FMT_HQ2B_HAD, kvq.FMT_HQ2B_TOK):
        g = kvq.geom(f, 16, 4, 24)
        assert kvq.page_bytes(g) == kvq.page_bytes(gh) == 64 * 9216
        assert kvq.ring_bytes(g, 8) == kvq.ring_bytes(gh, 8)
    base = kvq.decode_workspace_bytes(gh, 8, 40960)
    assert kvq.decode_workspace_bytes(kvq.geom(kvq.FMT_HQ2B_TOK, 16, 4, 24), 8, 40960) == base
    assert kvq.decode_workspace_bytes(kvq.geom(kvq.FMT_HQ2B_HAD, 16, 4, 24), 8, 40960) == base + 8 * 24 * 512


def test_fp8_sizes_and_scales(L):
    """FP8 E4M3 pages: 256 B per head per token for K and for V, no ring; a negative or
    non-finite scale is refused."""
    g = kvq.geom(kvq.FMT_FP8, 16, 4, 24)
    assert kvq.token_bytes(g) == 16 * 4 * 2 * 256
    assert kvq.page_bytes(g) == 64 * 16 * 4 * 2 * 256
    assert kvq.ring_bytes(g, 8) == 0
    assert kvq.page_bytes(kvq.geom(kvq.FMT_FP8, 16, 4, 24, k_scale=0.5, v_scale=2.0)) == kvq.page_bytes(g)
    for bad in (-1.0, float("inf"), float("nan")):
        assert kvq.page_bytes(kvq.geom(kvq.FMT_FP8, 16, 4, 24, k_scale=bad)) == 0
        assert kvq.page_bytes(kvq.geom(kvq.FMT_FP8, 16, 4, 24, v_scale=bad)) == 0


@pytest.mark.parametrize("bad", [dict(head_dim=128), dict(page_tokens=32), dict(format=7),
                                 dict(num_q_heads=36), dict(num_q_heads=10)])
def test_unsupported_geometry_is_refused(L, bad):
    args = dict(format=0, num_layers=16, num_kv_heads=4, num_q_heads=24, head_dim=256, page_tokens=64)
    args.update(bad)
    g = kvq.Geom(**args)
    assert kvq.page_bytes(g) == 0
    assert kvq.pool_pages(g, 1 << 30) == -1
    rc = L.paged_decode_attn(ctypes.byref(g), 0, 16, 1 << 20, 16, 0, 16, 1, 1, 16, 64, 16, 0.0625, 16,
                             1 << 20, 16, 16, None)
    assert rc in (kvq.ERR_UNSUPPORTED, kvq.ERR_INVALID_ARG)


def _decode(L, g, **kw):
    a = dict(layer=0, pool=256, pool_bytes=1 << 24, ring=512, window=0, pt=768, max_pages=4, lanes=1,
             seq_len=1024, max_seq_len=256, q=1280, scale=0.0625, ws=1536, ws_bytes=1 << 24, out=1792,
             status=2048)
    a.update(kw)
    return L.paged_decode_attn(ctypes.byref(g), a["layer"], a["pool"], a["pool_bytes"], a["ring"], a["window"],
                               a["pt"], a["max_pages"], a["lanes"], a["seq_len"], a["max_seq_len"], a["q"],
                               a["scale"], a["ws"], a["ws_bytes"], a["out"], a["status"], None)


def test_decode_host_validation(L):
    g = kvq.geom(kvq.FMT_HQ2B, 2, 1, 4)
    assert _decode(L, g, layer=2) == kvq.ERR_INVALID_ARG
    assert _decode(L, g, layer=-1) == kvq.ERR_INVALID_ARG
    assert _decode(L, g, window=65) == kvq.ERR_INVALID_ARG
    assert _decode(L, g, max_seq_len=257) == kvq.ERR_INVALID_ARG     # past max_pages * 64
    assert _decode(L, g, ring=None) == kvq.ERR_INVALID_ARG           # 2-bit needs the ring
    assert _decode(L, g, q=None) == kvq.ERR_INVALID_ARG
    assert _decode(L, g, pool_bytes=100) == kvq.ERR_INVALID_ARG      # smaller than one page
    assert _decode(L, g, q=1288) == kvq.ERR_ALIGNMENT
    assert _decode(L, g, ws_bytes=64) == kvq.ERR_WORKSPACE_TOO_SMALL
    assert _decode(L, g, lanes=0) == kvq.OK                           # nothing to do, nothing launched


def test_append_host_validation(L):
    g = kvq.geom(kvq.FMT_HQ2B, 1, 1, 4)

    def app(**kw):
        a = dict(layer=0, pool=256, pool_bytes=1 << 20, ring=512, pt=768, max_pages=4, lanes=1, start=1024,
                 n=1040, off=1056, max_new=64, n_rows=64, k=1280, v=1536, status=2048)
        a.update(kw)
        return L.kv_quant_append(ctypes.byref(g), a["layer"], a["pool"], a["pool_bytes"], a["ring"], a["pt"],
                                 a["max_pages"], a["lanes"], a["start"], a["n"], a["off"], a["max_new"],
                                 a["n_rows"], a["k"], a["v"], a["status"], None)

    assert app(layer=1) == kvq.ERR_INVALID_ARG
    assert app(max_new=-1) == kvq.ERR_INVALID_ARG
    assert app(ring=None) == kvq.ERR_INVALID_ARG
    assert app(k=None) == kvq.ERR_INVALID_ARG
    assert app(v=1544) == kvq.ERR_ALIGNMENT
    assert app(max_new=0) == kvq.OK
    gb = kvq.geom(kvq.FMT_BF16, 1, 1, 4)
    assert L.kv_quant_append(ctypes.byref(gb), 0, 256, 1 << 20, None, 768, 4, 1, 1024, 1040, 1056, 0, 0,
                             1280, 1536, 2048, None) == kvq.OK


def test_prefill_host_validation(L):
    g = kvq.geom(kvq.FMT_BF16, 1, 1, 4)

    def pre(**kw):
        a = dict(pool=256, pool_bytes=1 << 22, pt=768, max_pages=4, lanes=1, qp=1024, nq=1040, qo=1056,
                 max_n_q=16, rows=16, seq=1072, max_seq=256, q=1280, ws=1536, ws_bytes=1 << 24, out=1792,
                 status=2048)
        a.update(kw)
        return L.paged_prefill_attn(ctypes.byref(g), 0, a["pool"], a["pool_bytes"], None, 0, a["pt"],
                                    a["max_pages"], a["lanes"], a["qp"], a["nq"], a["qo"], a["max_n_q"],
                                    a["rows"], a["seq"], a["max_seq"], a["q"], 0.0625, a["ws"], a["ws_bytes"],
                                    a["out"], a["status"], None)

    assert pre(qp=None) == kvq.ERR_INVALID_ARG
    assert pre(max_n_q=-1) == kvq.ERR_INVALID_ARG
    assert pre(ws_bytes=1024) == kvq.ERR_WORKSPACE_TOO_SMALL
    assert pre(max_n_q=0) == kvq.OK


def test_strerror(L):
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(kvq.strerror(code), str) and kvq.strerror(code)


def test_format_variants_host_validation(L):
    """Host-side answers for the format variants, all returned before any launch: the 2-bit
    variants need the ring, FP8 does not; a bad FP8 scale is refused by every call; the rotated
    format's prefill needs no more workspace than the plain format's."""
    tok = kvq.geom(kvq.FMT_HQ2B_TOK, 2, 1, 4)
    had = kvq.geom(kvq.FMT_HQ2B_HAD, 2, 1, 4)
    assert _decode(L, tok, ring=None) == kvq.ERR_INVALID_ARG
    assert _decode(L, had, ring=None) == kvq.ERR_INVALID_ARG
    assert _decode(L, tok, ws_bytes=64) == kvq.ERR_WORKSPACE_TOO_SMALL
    fp8 = kvq.geom(kvq.FMT_FP8, 2, 1, 4)
    assert _decode(L, fp8, ring=None, ws_bytes=64) == kvq.ERR_WORKSPACE_TOO_SMALL   # no ring needed
    assert _decode(L, fp8, ring=None, lanes=0) == kvq.OK
    bad = kvq.geom(kvq.FMT_FP8, 2, 1, 4, k_scale=-2.0)
    assert _decode(L, bad, ring=None) == kvq.ERR_INVALID_ARG
    assert L.kv_quant_append(ctypes.byref(bad), 0, 256, 1 << 24, None, 768, 4, 1, 1024, 1040, 1056, 1, 1,
                             1280, 1536, 2048, None) == kvq.ERR_INVALID_ARG
    plain = kvq.prefill_workspace_bytes(kvq.geom(kvq.FMT_HQ2B, 2, 1, 4), 16, 256)
    assert kvq.prefill_workspace_bytes(had, 16, 256) == plain
    rc = L.paged_prefill_attn(ctypes.byref(had), 0, 256, 1 << 22, 512, 0, 768, 4, 1, 1024, 1040, 1056, 16, 16,
                              1072, 256, 1280, 0.0625, 1536, plain - 256, 1792, 2048, None)
    assert rc == kvq.ERR_WORKSPACE_TOO_SMALL


def _noalloc(L, g, **kw):
    a = dict(layer=0, pool=256, pool_bytes=1 << 24, ring=512, window=0, pt=768, max_pages=4, lanes=1,
             seq_len=1024, max_seq_len=256, q=1280, scale=0.0625, out=1792, status=2048)
    a.update(kw)
    gp = ctypes.byref(g) if g is not None else None
    return L.paged_decode_attn_noalloc(gp, a["layer"], a["pool"], a["pool_bytes"], a["ring"], a["window"], a["pt"],
                                       a["max_pages"], a["lanes"], a["seq_len"], a["max_seq_len"], a["q"],
                                       a["scale"], a["out"], a["status"], None)


def test_noalloc_host_validation_matches_decode(L):
    """The no-allocation decode checks its arguments exactly as paged_decode_attn does, before
    its own scratch limit, and refuses a request over the limit before anything is launched."""
    g = kvq.geom(kvq.FMT_HQ2B, 2, 1, 4)
    assert L.paged_decode_attn_noalloc(None, 0, 256, 1 << 24, 512, 0, 768, 4, 1, 1024, 256, 1280, 0.0625, 1792,
                                       2048, None) == kvq.ERR_INVALID_ARG
    bad_group = kvq.geom(kvq.FMT_HQ2B, 2, 4, 10)          # 10 query heads over 4 KV heads
    assert _noalloc(L, bad_group) == _decode(L, bad_group) == kvq.ERR_INVALID_ARG
    wide_group = kvq.geom(kvq.FMT_HQ2B, 2, 1, 12)          # group 12 > 8
    assert _noalloc(L, wide_group) == _decode(L, wide_group) == kvq.ERR_UNSUPPORTED
    for kw in (dict(layer=2), dict(window=65), dict(max_seq_len=257), dict(ring=None), dict(q=None),
               dict(pool_bytes=100), dict(q=1288), dict(out=None), dict(status=None)):
        assert _noalloc(L, g, **kw) == _decode(L, g, **kw), kw
    assert _noalloc(L, g, lanes=0) == kvq.OK
    # 4,096 lanes of 2^22 tokens need far more than the static scratch: refused on the host
    huge = 1 << 22
    assert kvq.decode_workspace_bytes(g, 4096, huge) > kvq.NOALLOC_SCRATCH_BYTES
    assert _noalloc(L, g, lanes=4096, max_seq_len=huge, max_pages=huge // 64) == kvq.ERR_SCRATCH_LIMIT


def test_selftest_wait_timeout_host_validation(L):
    """The bounded-wait self-test refuses a null status word on the host, before any launch."""
    assert L.kvq_selftest_wait_timeout(None, None) == kvq.ERR_INVALID_ARG


def _step(L, g, **kw):
    a = dict(layer=0, pool=256, pool_bytes=1 << 24, ring=512, window=0, pt=768, max_pages=4, lanes=1,
             start=2304, n_new=2560, tok_off=2816, n_rows=1, k=3072, v=3328, seq_len=1024, max_seq_len=256,
             q=1280, scale=0.0625, ws=1536, ws_bytes=1 << 24, out=1792, status=2048)
    a.update(kw)
    return L.kvq_decode_step(ctypes.byref(g), a["layer"], a["pool"], a["pool_bytes"], a["ring"], a["window"],
                             a["pt"], a["max_pages"], a["lanes"], a["start"], a["n_new"], a["tok_off"], a["n_rows"],
                             a["k"], a["v"], a["seq_len"], a["max_seq_len"], a["q"], a["scale"], a["ws"],
                             a["ws_bytes"], a["out"], a["status"], None)


@pytest.mark.parametrize("window", [0, 64])
def test_decode_step_host_validation(L, window):
    """kvq_decode_step checks the append's arguments and the attention's before it launches
    anything, in both launch orders (window 64: the append runs last)."""
    g = kvq.geom(kvq.FMT_HQ2B, 2, 1, 4)
    assert _step(L, g, window=window, start=None) == kvq.ERR_INVALID_ARG
    assert _step(L, g, window=window, n_rows=-1) == kvq.ERR_INVALID_ARG
    assert _step(L, g, window=window, k=3080) == kvq.ERR_ALIGNMENT
    assert _step(L, g, window=window, v=None) == kvq.ERR_INVALID_ARG
    assert _step(L, g, window=window, ws_bytes=64) == kvq.ERR_WORKSPACE_TOO_SMALL
    assert _step(L, g, window=window, layer=2) == kvq.ERR_INVALID_ARG
    assert _step(L, g, window=window, lanes=0) == kvq.OK
