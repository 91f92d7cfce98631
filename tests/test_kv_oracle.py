"""Pins for the oracle's attention K/V pool layout and copy_prefix: the block
stride worked example of vLLM-Ascend "非连续 KV Cache" §3.4 through a K/V pool,
the lane stride of the merged two-lane view, a numpy strided-view brute force
of copy_prefix with every other byte unchanged, a whole prefix copied block by
block read back as token rows, and the rejections.  CPU only.
"""
import numpy as np

import oracle

from _util import golden_kv


def test_block_stride_worked_example_kv_pool():
    """§3.4: a 48-element fp16 block (96 B) in a 128 B page advances by 64
    elements; the merged view's lane stride is num_blocks pages."""
    g = golden_kv("block_stride_example.txt")
    # 3 tokens x 1 kv head x 16 dims = 48 elements
    p = oracle.KvPool(2, 5, 3, 1, 16, oracle.F16, g["page_bytes"])
    rc, L = oracle.kv_layout(p)
    assert rc == oracle.OK
    assert L["payload"] == g["logical_payload_bytes"]
    assert L["block_stride_elems"] == g["block_stride_elements"]
    assert L["block_stride_elems"] - L["payload"] // g["element_bytes"] == g["gap_elements"]
    assert L["lane_stride_elems"] == 5 * g["page_bytes"] // g["element_bytes"]
    assert L["region_bytes"] == 2 * 5 * g["page_bytes"]


def test_kv_layout_rejects_bad_pages():
    assert oracle.kv_layout(oracle.KvPool(1, 4, 3, 1, 16, oracle.F16, 94))[0] == oracle.REJECT_LAYOUT  # < payload
    assert oracle.kv_layout(oracle.KvPool(1, 4, 3, 1, 16, oracle.F32, 194))[0] == oracle.REJECT_LAYOUT  # % 4
    assert oracle.kv_layout(oracle.KvPool(1, 0, 3, 1, 16, oracle.F16, 128))[0] == oracle.REJECT_ARG


def make(layers=2, blocks=9, bt=4, heads=2, hd=8, dtype=oracle.BF16, pad=48, seed=0):
    es = oracle.esize(dtype)
    page = bt * heads * hd * es + pad
    p = oracle.KvPool(layers, blocks, bt, heads, hd, dtype, page)
    rng = np.random.default_rng(seed)
    regions = [rng.integers(0, 256, 2 * blocks * page, dtype=np.uint8) for _ in range(layers)]
    return p, regions, page, bt * heads * hd * es // bt


def test_copy_prefix_brute_force():
    p, regions, page, row = make()
    pre = [r.copy() for r in regions]
    src = np.array([1, 1, 7, 3], np.int32)
    dst = np.array([0, 5, 2, 8], np.int32)
    nt = np.array([4, 2, 1, 0], np.int32)        # full, partial, one row, nothing
    assert oracle.copy_prefix(p, regions, src, dst, nt) == oracle.OK
    for l in range(2):
        want = pre[l].reshape(2, 9, page).copy()  # (lane, block, page bytes)
        for s_, d_, n_ in zip(src, dst, nt):
            want[:, d_, :n_ * row] = want[:, s_, :n_ * row]
        np.testing.assert_array_equal(regions[l], want.reshape(-1))


def test_whole_prefix_block_by_block_reads_back_as_token_rows():
    """A prefix of 10 tokens in blocks [3, 0, 6] (4 tokens each) copied into
    blocks [1, 2, 4]: the destination's logical token rows 0..9 equal the
    source's, row 10 onwards of the last block keeps its old content."""
    p, regions, page, row = make(blocks=8, seed=3)
    pre = [r.copy() for r in regions]
    T, bt = 10, 4
    src_blocks, dst_blocks = [3, 0, 6], [1, 2, 4]
    nt = [min(bt, T - bt * i) for i in range(3)]
    assert oracle.copy_prefix(p, regions, src_blocks, dst_blocks, nt) == oracle.OK

    def rows(reg, lane, blocks, n):
        v = reg.reshape(2, 8, page)[lane]
        return np.concatenate([v[b, :bt * row].reshape(bt, row) for b in blocks])[:n]

    for l in range(2):
        for lane in range(2):
            np.testing.assert_array_equal(rows(regions[l], lane, dst_blocks, T), rows(pre[l], lane, src_blocks, T))
            np.testing.assert_array_equal(rows(regions[l], lane, dst_blocks, 12)[T:],
                                          rows(pre[l], lane, dst_blocks, 12)[T:])


def test_copy_prefix_rejections_leave_regions_unchanged():
    p, regions, page, row = make()
    pre = [r.copy() for r in regions]
    cases = [
        (([1, 2], [0, 0], [4, 4]), oracle.REJECT_DUP_DST),
        (([1, 0], [0, 3], [4, 1]), oracle.REJECT_SRC_IS_DST),
        (([1], [9], [1]), oracle.REJECT_RANGE),
        (([-1], [2], [1]), oracle.REJECT_RANGE),
        (([1], [2], [5]), oracle.REJECT_ARG),      # more tokens than a block holds
    ]
    for (s_, d_, n_), want in cases:
        assert oracle.copy_prefix(p, regions, s_, d_, n_) == want, (s_, d_, n_)
    for r, q in zip(regions, pre):
        np.testing.assert_array_equal(r, q)
    # ops copying nothing are not checked
    assert oracle.copy_prefix(p, regions, [99, 1], [0, 0], [0, 0]) == oracle.OK
    for r, q in zip(regions, pre):
        np.testing.assert_array_equal(r, q)
