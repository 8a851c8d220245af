"""paged_decode_attn_noalloc against paged_decode_attn.

Some callers cannot allocate device memory -- plugins of a serving engine whose allocator
owns the whole GPU and hands out no scratch, hosts that forbid allocation after start-up.
The no-allocation entry point serves them from a static scratch array inside the library
instead of a caller workspace.  This test first leaves partials of a larger call in that
array (a wider split stride), then calls the entry point through the C ABI twice in a row
(with different queries, so a stale result cannot pass for a fresh one) and checks each
output against the regular entry point with a caller-allocated workspace, within the
attention tolerance.  It sits in a file of its own that pytest collects last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

ATOL, RTOL = 2e-3, 1e-3


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_paged_kv_quant_gb300 import build, kvq, synth
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    build.build()

    lens = [700, 1500, 64, 3001]
    pages = [(n + 63) // 64 for n in lens]
    perm = synth.permutation(3, sum(pages), salt=11)
    table = np.full((len(lens), max(pages)), -1, np.int32)
    off = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[off:off + p]
        off += p
    wl = synth.Workload("noalloc", 2, 2, 12, lens, table, sum(pages), window=64, seed=3)
    dw = DeviceWorkload(wl, kvq.FMT_HQ2B, "cuda", fill=0xA5)
    dw.fill_history(lens)
    ws, ref = dw.decode_buffers()
    out = torch.empty_like(ref)
    # a larger call first: a page table four times as wide and a bound to match give every
    # (lane, head) more split records, so the array is left holding non-zero partials laid
    # out under another stride than the calls checked below
    wide = torch.full((len(lens), 4 * max(pages)), -1, dtype=torch.int32, device="cuda")
    wide[:, :max(pages)] = dw.page_table
    wide_bound = 64 * wide.shape[1]
    assert kvq.decode_workspace_bytes(dw.g, len(lens), wide_bound) > kvq.decode_workspace_bytes(
        dw.g, len(lens), dw.max_seq_len)
    kvq.paged_decode_attn_noalloc(dw.g, 1, dw.cache.pool, dw.cache.ring, wl.window, wide, dw.seq_len, wide_bound,
                                  dw.step_q(1) * 3.0, dw.sm_scale, out, dw.cache.status)
    torch.cuda.synchronize()
    assert dw.cache.read_status() == 0
    for call, layer in enumerate((1, 0)):
        q = dw.step_q(layer) * (1.0 + call)          # a different query on each call
        dw.decode(layer, q, ws, ref)
        out.fill_(float("nan"))
        kvq.paged_decode_attn_noalloc(dw.g, layer, dw.cache.pool, dw.cache.ring, wl.window, dw.page_table,
                                      dw.seq_len, dw.max_seq_len, q, dw.sm_scale, out, dw.cache.status)
        torch.cuda.synchronize()
        assert dw.cache.read_status() == 0
        a, r = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(a - r) <= ATOL + RTOL * np.abs(r)), f"call {call}: max {np.abs(a - r).max()}"

    # a request larger than the static scratch is refused on the host, nothing launched
    huge = 1 << 22
    need = kvq.decode_workspace_bytes(dw.g, 4096, huge)
    assert need > kvq.NOALLOC_SCRATCH_BYTES
    big_table = torch.zeros((1, huge // 64), dtype=torch.int32, device="cuda")
    tiny = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.paged_decode_attn_noalloc(dw.g, 0, dw.cache.pool, dw.cache.ring, 0, big_table, tiny, huge,
                                      torch.zeros(256, dtype=torch.bfloat16, device="cuda"), dw.sm_scale,
                                      torch.zeros(256, dtype=torch.float32, device="cuda"), dw.cache.status,
                                      lanes=4096)
    assert e.value.code == kvq.ERR_SCRATCH_LIMIT
