"""Page moves on the GPU: pool pages gathered into a pinned host arena (and a device arena) are
byte-identical to the oracle's gather of the same pool, and scattering them to other page ids
with the page table pointed there leaves decode attention bit for bit the same."""
import numpy as np
import pytest

import oracle
from compressed_paged_kv_quant_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_paged_kv_quant_gb300 import build
    build.build()


def _workload(lens, seed=2):
    pages = [(n + 63) // 64 for n in lens]
    total = sum(pages) + 5
    perm = synth.permutation(seed, total, salt=9)
    t = np.full((len(lens), max(pages)), -1, np.int32)
    off = 0
    for b, p in enumerate(pages):
        t[b, :p] = perm[off:off + p]
        off += p
    return synth.Workload(f"pages_{lens}", 2, 2, 8, list(lens), t, total, window=64, seed=seed)


@pytest.mark.parametrize("where,fmt", [("host", oracle.FMT_HQ2B), ("device", oracle.FMT_HQ2B), ("device", oracle.FMT_FP8)])
def test_gather_scatter_moves_pages_bit_exact(where, fmt):
    """Pages of the 2-bit format and of the FP8 format move bit for bit."""
    from compressed_paged_kv_quant_gb300 import kvq
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    wl = _workload([700, 130, 2000])
    dw = DeviceWorkload(wl, fmt, "cuda", fill=0x5A)
    dw.fill_history(wl.seq_len)
    torch.cuda.synchronize()
    g = oracle.geom(fmt, wl.num_layers, wl.num_kv_heads, wl.num_q_heads)
    pb = oracle.page_bytes(g)
    used = sorted({int(p) for p in wl.page_table.ravel() if p >= 0})
    ids = [used[i] for i in np.random.default_rng(4).permutation(len(used))]
    ids_t = torch.tensor(ids, dtype=torch.int32, device="cuda")
    if where == "host":
        arena = torch.empty(len(ids) * pb, dtype=torch.uint8).pin_memory()
    else:
        arena = torch.empty(len(ids) * pb, dtype=torch.uint8, device="cuda")
    kvq.pages_gather(dw.g, dw.cache.pool, ids_t, arena, dw.cache.status)
    torch.cuda.synchronize()
    assert dw.cache.read_status() == 0
    pool_np = dw.cache.pool.cpu().numpy()
    ref, st = oracle.pages_gather(g, pool_np, ids)
    assert st == 0
    assert np.array_equal(arena.cpu().numpy(), ref)

    # scatter into a second pool at other ids, repoint the page table, decode: same bits
    new_ids = [(p + 3) % wl.pool_pages for p in ids]
    remap = dict(zip(ids, new_ids))
    dw2 = DeviceWorkload(wl, fmt, "cuda", fill=0x33)
    if dw.cache.ring is not None:                      # the ring is per lane, not paged (FP8: none)
        dw2.cache.ring.copy_(dw.cache.ring)
    kvq.pages_scatter(dw2.g, dw2.cache.pool, torch.tensor(new_ids, dtype=torch.int32, device="cuda"), arena,
                      dw2.cache.status)
    pt2 = np.vectorize(lambda p: remap.get(int(p), -1) if p >= 0 else -1)(wl.page_table).astype(np.int32)
    dw2.page_table = torch.from_numpy(pt2).cuda()
    torch.cuda.synchronize()
    assert dw2.cache.read_status() == 0
    pool2 = dw2.cache.pool.cpu().numpy()
    for p, q in remap.items():
        assert np.array_equal(pool2[q * pb:(q + 1) * pb], pool_np[p * pb:(p + 1) * pb])
    for layer in range(wl.num_layers):
        q = dw.step_q(layer)
        ws1, out1 = dw.decode_buffers()
        ws2, out2 = dw2.decode_buffers()
        dw.decode(layer, q, ws1, out1)
        dw2.decode(layer, q, ws2, out2)
        torch.cuda.synchronize()
        assert torch.equal(out1, out2)
    assert dw.cache.read_status() == 0 and dw2.cache.read_status() == 0


def test_page_move_flags_bad_id():
    from compressed_paged_kv_quant_gb300 import kvq
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    wl = _workload([64])
    dw = DeviceWorkload(wl, kvq.FMT_HQ2B, "cuda", fill=0x11)
    pb = kvq.page_bytes(dw.g)
    arena = torch.full((2 * pb,), 0x77, dtype=torch.uint8, device="cuda")
    ids = torch.tensor([0, wl.pool_pages], dtype=torch.int32, device="cuda")
    kvq.pages_gather(dw.g, dw.cache.pool, ids, arena, dw.cache.status)
    torch.cuda.synchronize()
    assert dw.cache.read_status() == oracle.PAGE_OOB
    a = arena.cpu().numpy()
    assert np.all(a[:pb] == 0x11) and np.all(a[pb:] == 0x77)     # the bad slot is left alone


def test_bounded_wait_runs_out_and_context_stays_usable():
    """A barrier wait that nothing ends gives up within its bound: the TIMEOUT status bit is set,
    the call returns, and the context then runs further kernels (the library's own page move)."""
    import time
    from compressed_paged_kv_quant_gb300 import kvq
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvq.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == kvq.STATUS_TIMEOUT
    assert elapsed < 5.0
    g = kvq.Geom(oracle.FMT_HQ2B, 2, 2, 8, 256, 64, 1.0, 1.0)
    pb = kvq.page_bytes(g)
    pool = torch.arange(4 * pb, device="cuda").to(torch.uint8)
    arena = torch.zeros(2 * pb, dtype=torch.uint8, device="cuda")
    ids = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.pages_gather(g, pool, ids, arena, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(arena[:pb], pool[3 * pb:4 * pb]) and torch.equal(arena[pb:], pool[pb:2 * pb])
