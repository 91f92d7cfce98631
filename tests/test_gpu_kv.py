"""GPU parity of copy_prefix against the oracle: every byte of every attention
layer identical after the copy (rows past n_tokens, padding, sources and other
blocks untouched), with random bytes everywhere before the call; odd row sizes
(word and byte paths), more ops than one launch holds, the done event, and a
full-size pool on sampled blocks.

Sources: vLLM-Ascend "非连续 KV Cache" §3, §3.4; Kapitsa figure 2.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_lsc_gb300 import lsc as L

pytestmark = pytest.mark.gpu

ODT = {L.LSC_BF16: oracle.BF16, L.LSC_F32: oracle.F32, L.LSC_F16: oracle.F16}
ES = {L.LSC_BF16: 2, L.LSC_F32: 4, L.LSC_F16: 2}


class DevKv:
    def __init__(self, layers, blocks, bt, heads, hd, dtype, pad, seed=0):
        es = ES[dtype]
        payload = bt * heads * hd * es
        page = (payload + 15) // 16 * 16 + pad
        self.d = L.lsc_kv_pool_desc(layers, blocks, bt, heads, hd, dtype, page)
        self.nbytes = L.lsc_kv_pool_required_bytes(self.d)
        rng = np.random.default_rng(seed)
        self.host = rng.integers(0, 256, self.nbytes, dtype=np.uint8)
        self.buf = torch.from_numpy(self.host.copy()).cuda()
        rc, self.pool = L.lsc_kv_pool_create(self.d, self.buf, self.nbytes)
        assert rc == L.LSC_OK
        self.opool = oracle.KvPool(layers, blocks, bt, heads, hd, ODT[dtype], page)
        self.region = self.nbytes // layers

    def oracle_copy(self, src, dst, nt):
        regs = [self.host[l * self.region:(l + 1) * self.region].copy() for l in range(self.d.num_layers)]
        rc = oracle.copy_prefix(self.opool, regs, src, dst, nt)
        return rc, np.concatenate(regs)

    def close(self):
        assert L.lsc_kv_pool_destroy(self.pool) == L.LSC_OK


def random_ops(rng, blocks, bt, n):
    perm = rng.permutation(blocks)
    dst = perm[:n]
    src = rng.choice(perm[n:], n)            # sources never destinations; repeats allowed
    nt = rng.integers(0, bt + 1, n)
    return src.astype(np.int32), dst.astype(np.int32), nt.astype(np.int32)


SHAPES = [(3, 24, 4, 2, 8, L.LSC_BF16, 32), (2, 20, 5, 1, 3, L.LSC_F32, 16), (1, 12, 64, 2, 128, L.LSC_BF16, 512),
          (2, 10, 7, 3, 5, L.LSC_F16, 0)]


@pytest.mark.parametrize("shape", SHAPES, ids=["bf16", "f32-odd-rows", "bf16-64tok", "f16-odd"])
def test_copy_prefix_matches_oracle(lsc, shape):
    kv = DevKv(*shape, seed=1)
    rng = np.random.default_rng(2)
    src, dst, nt = random_ops(rng, shape[1], shape[2], 8)
    ev = torch.cuda.Event()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    rc, nbytes = L.lsc_copy_prefix(kv.pool, L.kv_ops(src, dst, nt), side, ev)
    assert rc == L.LSC_OK
    torch.cuda.current_stream().wait_event(ev)
    got = kv.buf.cpu().numpy()
    rc_o, want = kv.oracle_copy(src, dst, nt)
    assert rc_o == oracle.OK
    np.testing.assert_array_equal(got, want)
    v = L.lsc_kv_pool_layer_view(kv.pool, 0)[1]
    assert nbytes == int(nt.sum()) * v.row_bytes * 2 * shape[0]
    kv.close()


def test_copy_prefix_more_ops_than_one_launch(lsc):
    kv = DevKv(2, 6000, 2, 1, 8, L.LSC_BF16, 16, seed=3)
    rng = np.random.default_rng(4)
    src, dst, nt = random_ops(rng, 6000, 2, 3000)
    rc, _ = L.lsc_copy_prefix(kv.pool, L.kv_ops(src, dst, nt), torch.cuda.current_stream())
    assert rc == L.LSC_OK
    torch.cuda.synchronize()
    rc_o, want = kv.oracle_copy(src, dst, nt)
    np.testing.assert_array_equal(kv.buf.cpu().numpy(), want)
    kv.close()


@pytest.mark.big
def test_copy_prefix_full_size_sampled(lsc):
    """12 attention layers, 2048 blocks of 64 tokens x 2 kv heads x 256 dims bf16
    (64 KiB) in 64.5 KiB pages (3.2 GB); 16 prefixes of 31.5 blocks copied."""
    d = L.lsc_kv_pool_desc(12, 2048, 64, 2, 256, L.LSC_BF16, 65536 + 512)
    n = L.lsc_kv_pool_required_bytes(d)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    buf.view(torch.int32).random_(generator=g)
    rc, pool = L.lsc_kv_pool_create(d, buf, n)
    assert rc == L.LSC_OK
    rng = np.random.default_rng(6)
    perm = rng.permutation(2048)
    src, dst, nt = [], [], []
    for i in range(16):
        sb, db = perm[64 * i:64 * i + 32], perm[1024 + 64 * i:1024 + 64 * i + 32]
        src += list(sb)
        dst += list(db)
        nt += [64] * 31 + [32]
    page, lane = d.page_bytes, 2048 * d.page_bytes
    region = 2 * lane
    pages = buf.view(12, 2, 2048, page)
    before = pages[:, :, perm[1024:1088]].clone()     # the first prefix's destinations
    untouched = perm[32:64]                           # neither a source nor a destination
    keep = pages[:, :, untouched].clone()
    rc, nbytes = L.lsc_copy_prefix(pool, L.kv_ops(src, dst, nt), torch.cuda.current_stream())
    assert rc == L.LSC_OK
    torch.cuda.synchronize()
    row = 2 * 256 * 2
    for i in (0, 7, 15):
        for j in (0, 17, 31):
            s_, d_, n_ = src[32 * i + j], dst[32 * i + j], nt[32 * i + j]
            assert torch.equal(pages[:, :, d_, :n_ * row], pages[:, :, s_, :n_ * row])
    # the last (partial) block of prefix 0 keeps its rows past 32 and its padding
    assert torch.equal(pages[:, :, dst[31], 32 * row:], before[:, :, 31, 32 * row:])
    assert torch.equal(pages[:, :, untouched], keep)
    assert nbytes == sum(nt) * row * 2 * 12
    assert L.lsc_kv_pool_destroy(pool) == L.LSC_OK


def random_kv_shapes(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        out.append((int(rng.integers(1, 4)), int(rng.integers(8, 40)), int(rng.choice([1, 2, 3, 8, 16, 64])),
                    int(rng.integers(1, 5)), int(rng.choice([3, 8, 16, 64, 128, 256])),
                    int(rng.choice([L.LSC_BF16, L.LSC_F32, L.LSC_F16])), 16 * int(rng.integers(0, 9))))
    return out


KV_RANDOM = random_kv_shapes(2027, 12)


@pytest.mark.parametrize("shape", KV_RANDOM,
                         ids=["L{}-B{}-bt{}-h{}-d{}-t{}-pad{}".format(*s) for s in KV_RANDOM])
def test_copy_prefix_random_shape(lsc, shape):
    """Seeded random pools (layers, blocks, block tokens, kv heads, head dims,
    dtypes, page padding): every byte equals the oracle's after the copy."""
    kv = DevKv(*shape, seed=5)
    rng = np.random.default_rng(6)
    src, dst, nt = random_ops(rng, shape[1], shape[2], min(8, shape[1] // 2))
    rc, _ = L.lsc_copy_prefix(kv.pool, L.kv_ops(src, dst, nt), torch.cuda.current_stream())
    assert rc == L.LSC_OK
    torch.cuda.synchronize()
    rc_o, want = kv.oracle_copy(src, dst, nt)
    assert rc_o == oracle.OK
    np.testing.assert_array_equal(kv.buf.cpu().numpy(), want)
    kv.close()
