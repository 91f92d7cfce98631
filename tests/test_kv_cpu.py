"""The K/V pool through the C ABI on the host (no GPU calls): layout and views
against the oracle's layout, descriptor errors, and copy_prefix's validation,
which rejects before anything is enqueued.  Host-only pools borrow a fake
base address that is never dereferenced.

Sources: vLLM-Ascend "非连续 KV Cache" §3, §3.4; Kapitsa figure 2.
"""

import oracle
from linear_attention_state_lsc_gb300 import lsc as L

from _util import golden_kv, gpu_present

FAKE_BASE = 1 << 40


def desc(layers=3, blocks=16, bt=4, heads=2, hd=8, dtype=L.LSC_BF16, page=None):
    es = 4 if dtype == L.LSC_F32 else 2
    page = page if page is not None else (bt * heads * hd * es + 15) // 16 * 16 + 32
    return L.lsc_kv_pool_desc(layers, blocks, bt, heads, hd, dtype, page)


def host_pool(d):
    rc, pool = L.lsc_kv_pool_create(d, FAKE_BASE, 1 << 44)
    assert rc == L.LSC_OK, L.lsc_error_string(rc)
    return pool


def test_views_match_oracle_layout(lsc):
    for dt, odt in ((L.LSC_BF16, oracle.BF16), (L.LSC_F32, oracle.F32)):
        d = desc(dtype=dt)
        pool = host_pool(d)
        rc, Lo = oracle.kv_layout(oracle.KvPool(d.num_layers, d.num_blocks, d.block_tokens, d.num_kv_heads,
                                                d.head_dim, odt, d.page_bytes))
        assert rc == oracle.OK
        assert L.lsc_kv_pool_required_bytes(d) == d.num_layers * Lo["region_bytes"]
        for l in range(d.num_layers):
            rc, v = L.lsc_kv_pool_layer_view(pool, l)
            assert rc == L.LSC_OK
            assert v.region == FAKE_BASE + l * Lo["region_bytes"]
            assert v.k == v.region and v.v - v.k == Lo["lane_stride_elems"] * (4 if dt == L.LSC_F32 else 2)
            assert list(v.shape) == [d.num_blocks, d.block_tokens, d.num_kv_heads, d.head_dim]
            assert list(v.strides) == [Lo["block_stride_elems"], d.num_kv_heads * d.head_dim, d.head_dim, 1]
            assert v.lane_stride == Lo["lane_stride_elems"] and v.payload_bytes == Lo["payload"]
            assert v.row_bytes == Lo["row_bytes"]
        assert L.lsc_kv_pool_layer_view(pool, d.num_layers)[0] == L.LSC_ERR_OUT_OF_RANGE
        assert L.lsc_kv_pool_destroy(pool) == L.LSC_OK


def test_block_stride_worked_example_through_the_abi(lsc):
    """§3.4: 48 fp16 elements in a 128 B page -> block stride 64 elements."""
    g = golden_kv("block_stride_example.txt")
    d = L.lsc_kv_pool_desc(1, 4, 3, 1, 16, L.LSC_F16, g["page_bytes"])
    pool = host_pool(d)
    rc, v = L.lsc_kv_pool_layer_view(pool, 0)
    assert v.strides[0] == g["block_stride_elements"]
    assert v.payload_bytes == g["logical_payload_bytes"]
    assert v.strides[0] - v.payload_bytes // g["element_bytes"] == g["gap_elements"]
    L.lsc_kv_pool_destroy(pool)


def test_descriptor_errors(lsc):
    bad = [(desc(layers=0), L.LSC_ERR_INVALID_ARG), (desc(dtype=7), L.LSC_ERR_INVALID_ARG),
           (desc(page=64), L.LSC_ERR_LAYOUT), (desc(page=136), L.LSC_ERR_MISALIGNED),
           (desc(dtype=L.LSC_F32, page=258), L.LSC_ERR_LAYOUT)]
    for d, want in bad:
        assert L.lsc_kv_pool_create(d, FAKE_BASE, 1 << 44)[0] == want
    assert L.lsc_kv_pool_create(desc(), FAKE_BASE + 8, 1 << 44)[0] == L.LSC_ERR_MISALIGNED
    assert L.lsc_kv_pool_create(desc(), FAKE_BASE, 16)[0] == L.LSC_ERR_NO_MEMORY


def test_copy_prefix_validation(lsc):
    pool = host_pool(desc())
    cases = [
        (([1, 2], [0, 0], [4, 4]), L.LSC_ERR_DUP_DST),
        (([1, 0], [0, 3], [4, 1]), L.LSC_ERR_SRC_IS_DST),
        (([1], [16], [1]), L.LSC_ERR_OUT_OF_RANGE),
        (([-1], [2], [1]), L.LSC_ERR_OUT_OF_RANGE),
        (([1], [2], [5]), L.LSC_ERR_INVALID_ARG),
        (([1], [2], [-1]), L.LSC_ERR_INVALID_ARG),
    ]
    for (s_, d_, n_), want in cases:
        assert L.lsc_copy_prefix(pool, L.kv_ops(s_, d_, n_))[0] == want, (s_, d_, n_)
    ops = L.kv_ops([1], [2], [1])
    ops["reserved"] = 1
    assert L.lsc_copy_prefix(pool, ops)[0] == L.LSC_ERR_INVALID_ARG
    # valid ops on a host-only pool: nothing to run them on (made only where no
    # GPU is visible: with one, the stand-in base would be dereferenced)
    if not gpu_present():
        assert L.lsc_copy_prefix(pool, L.kv_ops([1, 99], [2, 0], [3, 0]))[0] == L.LSC_ERR_CUDA
        assert L.lsc_copy_prefix(pool, L.kv_ops([], [], []))[0] == L.LSC_ERR_CUDA
    L.lsc_kv_pool_destroy(pool)
