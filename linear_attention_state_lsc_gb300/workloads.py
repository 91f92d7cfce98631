"""Seeded synthetic workloads shared by the tests, the smoke check and bench.py.

This module holds no arithmetic of the method itself: no layout formula, no
restore decision, no conv or delta-rule math.  It draws seeded random inputs and
fills byte regions whose offsets the caller computes.  Page strides are literal
constants of each workload (their derivation is written next to them).

Workloads (shapes and value distributions from the task's configuration list):
  c0  tiny: layers GDN/attention/GDN, 16 slots, conv [64, 3] fp32,
      ssm [2, 16, 16] fp32, page padded to a 256 B multiple; 4 restore rows;
      one decode token per row.
  c1  restore at serving scale: 36 GDN + 12 attention layers (3 GDN then 1
      attention, repeated), 256 slots, conv [8192, 3] bf16, ssm [32, 128, 128]
      fp32, page rounded up to 4 KiB; 64 rows, all hits.
  c2  decode step: c1's shapes with bf16 ssm and 512 B of padding per page;
      256 live rows on a random permutation of the slots.
  c3  restore storm: c1's shapes, 1024 slots, 512 rows (40 % hit, 30 % miss,
      30 % no-op), one hot source slot, 0xA5 padding.
  c4  resume-after-restore prefill: 64 sequences of 64..2048 tokens on c1's
      pool, about half of them warm.
"""
from dataclasses import dataclass, field

import numpy as np

F32, BF16, F16 = "f32", "bf16", "f16"
ESIZE = {F32: 4, BF16: 2, F16: 2}
GDN, ATTN = "gdn", "attn"


@dataclass
class Workload:
    name: str
    layers: list
    num_slots: int
    conv_dim: int
    conv_width: int
    conv_dtype: str
    num_k_heads: int
    num_v_heads: int
    head_v_dim: int
    head_k_dim: int
    ssm_dtype: str
    page_bytes: int
    pad_byte: int = 0x00
    block_size: int = 16
    extra: dict = field(default_factory=dict)

    @property
    def gdn_layers(self):
        return [i for i, k in enumerate(self.layers) if k == GDN]


def _qwen_like_layers(n_gdn=36, n_attn=12):
    # three GDN layers followed by one attention layer, repeated
    out = []
    while len(out) < n_gdn + n_attn:
        out += [GDN, GDN, GDN, ATTN]
    return out


def get(name: str) -> Workload:
    if name == "c0":
        # conv 64*3*4 = 768 B, ssm 2*16*16*4 = 2048 B: 2816 B, already a multiple of 256
        return Workload("c0", [GDN, ATTN, GDN], 16, 64, 4, F32, 1, 2, 16, 16, F32, 2816,
                        pad_byte=0x00, block_size=16)
    if name == "c0p":
        # c0 with a page strictly larger than the payload (next 256 B multiple above
        # 2816) and a non-zero padding pattern
        return Workload("c0p", [GDN, ATTN, GDN], 16, 64, 4, F32, 1, 2, 16, 16, F32, 3072,
                        pad_byte=0xA5, block_size=16)
    if name == "c1":
        # conv 8192*3*2 = 49152 B, ssm 32*128*128*4 = 2097152 B: 2146304 B = 524 * 4096
        return Workload("c1", _qwen_like_layers(), 256, 8192, 4, BF16, 16, 32, 128, 128, F32,
                        2146304, pad_byte=0x00, block_size=64)
    if name == "c2":
        # conv 49152 B + ssm bf16 1048576 B = 1097728 B, plus 512 B of padding
        return Workload("c2", _qwen_like_layers(), 256, 8192, 4, BF16, 16, 32, 128, 128, BF16,
                        1098240, pad_byte=0xA5, block_size=64)
    if name == "c3":
        # c1's payload 2146304 B plus 512 B of padding
        return Workload("c3", _qwen_like_layers(), 1024, 8192, 4, BF16, 16, 32, 128, 128, F32,
                        2146816, pad_byte=0xA5, block_size=64)
    if name == "c4":
        return Workload("c4", _qwen_like_layers(), 256, 8192, 4, BF16, 16, 32, 128, 128, F32,
                        2146304, pad_byte=0x00, block_size=64)
    raise KeyError(name)


def small(name="s1", **kw) -> Workload:
    """Mid-size workloads for parity: several tiles and ragged tails, oracle in seconds."""
    base = dict(
        # Hk=2, Hv=4, dk=dv=32: conv 2*2*32 + 4*32 = 256 channels, W=4
        s1=Workload("s1", [GDN, GDN, ATTN, GDN], 24, 256, 4, BF16, 2, 4, 32, 32, F32,
                    # conv 256*3*2 = 1536 B, ssm 4*32*32*4 = 16384 B -> 17920 B, + 144 B pad
                    18064, pad_byte=0xA5, block_size=16),
        # dk = dv = 128 like the serving shapes, fewer heads: 2*2*128 + 4*128 = 1024
        s2=Workload("s2", [ATTN, GDN, GDN], 20, 1024, 4, BF16, 2, 4, 128, 128, BF16,
                    # conv 1024*3*2 = 6144 B, ssm 4*128*128*2 = 131072 B -> 137216 B, + 400 B pad
                    137616, pad_byte=0xA5, block_size=32),
        s3=Workload("s3", [GDN, ATTN], 12, 1024, 4, BF16, 2, 4, 128, 128, F32,
                    # conv 6144 B, ssm 4*128*128*4 = 262144 B -> 268288 B, + 256 B pad
                    268544, pad_byte=0x3C, block_size=32),
        # ragged byte counts: Hk=1, Hv=3, dk=16, dv=12 -> 2*16 + 3*12 = 68 channels;
        # conv 68*3*2 = 408 B (not a multiple of 16, so an 8 B gap precedes the ssm
        # view at 416), ssm 3*12*16*2 = 1152 B -> payload 1568 B, + 32 B pad
        s4=Workload("s4", [GDN, GDN], 10, 68, 4, BF16, 1, 3, 12, 16, BF16,
                    1600, pad_byte=0xA5, block_size=8),
    )[name]
    for k, v in kw.items():
        setattr(base, k, v)
    return base


# --------------------------------------------------------------------------
# random values

def _normal_f32(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def to_dtype_bytes(a_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Encode float32 values at `dtype`, returned as raw little-endian bytes (uint8).
    bf16/f16 use torch's CPU conversion (round to nearest even)."""
    a_f32 = np.ascontiguousarray(a_f32, np.float32)
    if dtype == F32:
        return a_f32.view(np.uint8).reshape(a_f32.shape[:-1] + (a_f32.shape[-1] * 4,))
    import torch
    t = torch.from_numpy(a_f32).to(torch.bfloat16 if dtype == BF16 else torch.float16)
    u = t.view(torch.int16).numpy().view(np.uint16)
    return u.view(np.uint8).reshape(a_f32.shape[:-1] + (a_f32.shape[-1] * 2,))


def from_dtype_bytes(b: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw bytes at `dtype` into float32 (exact)."""
    b = np.ascontiguousarray(b, np.uint8)
    if dtype == F32:
        return b.view(np.float32)
    import torch
    t = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16 if dtype == BF16 else torch.float16)
    return t.float().numpy()


def fill_region_host(region: np.ndarray, num_slots: int, page: int, views, pad_byte: int, seed: int):
    """Fill one layer region (uint8, num_slots*page bytes) on the host.

    views: list of (byte_offset_in_page, n_elems, dtype) -- the typed parts of a
    page; every other byte of every page gets pad_byte.  Values ~ N(0, 1).
    """
    rng = np.random.default_rng(seed)
    region[:] = pad_byte
    pages = region.reshape(num_slots, page)
    for off, n_elems, dtype in views:
        vals = _normal_f32(rng, (num_slots, n_elems))
        raw = to_dtype_bytes(vals, dtype)
        pages[:, off:off + raw.shape[1]] = raw


def fill_region_device(region, num_slots: int, page: int, views, pad_byte: int, seed: int):
    """Same as fill_region_host for a CUDA uint8 tensor, with torch's seeded
    generator on the device (used for the multi-GB pools)."""
    import torch
    tdt = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16}
    g = torch.Generator(device=region.device)
    g.manual_seed(seed)
    region.fill_(pad_byte)
    pages = region.view(num_slots, page)
    # fill in groups of slots to bound the temporary
    group = max(1, (256 << 20) // max(1, page))
    for off, n_elems, dtype in views:
        nb = n_elems * ESIZE[dtype]
        for s0 in range(0, num_slots, group):
            s1 = min(num_slots, s0 + group)
            vals = torch.randn((s1 - s0, n_elems), generator=g, device=region.device, dtype=torch.float32)
            raw = vals.to(tdt[dtype]).view(torch.uint8).view(s1 - s0, nb)
            pages[s0:s1, off:off + nb].copy_(raw)


# --------------------------------------------------------------------------
# restore rows

@dataclass
class RestoreRows:
    live: np.ndarray          # int32 linear_state_id
    src: np.ndarray           # int32 restore_src_slot_id
    restore_hash: np.ndarray  # uint64, carried
    save_hash: np.ndarray     # uint64, carried
    save_slot: np.ndarray     # int32, carried
    nkv: np.ndarray           # int32 n_kv_cache_tokens
    initialized: np.ndarray   # uint8 linear_state_initialized
    hs_prefill: np.ndarray    # uint8 has_initial_state default (row reused KV tokens)
    block_size: int


def _carried(rng, n, live):
    restore_hash = rng.integers(1, 2**63, size=n, dtype=np.int64).astype(np.uint64)
    save_hash = rng.integers(0, 2**63, size=n, dtype=np.int64).astype(np.uint64)
    save_slot = np.where(rng.random(n) < 0.5, live, -1).astype(np.int32)
    return restore_hash, save_hash, save_slot


def _rows(live, src, nkv, init, block_size, rng, restore_hash=None):
    live = np.asarray(live, np.int32)
    src = np.asarray(src, np.int32)
    nkv = np.asarray(nkv, np.int32)
    init = np.asarray(init, np.uint8)
    rh, sh, ss = _carried(rng, len(live), live)
    if restore_hash is not None:
        rh = np.asarray(restore_hash, np.uint64)
    hs = (nkv > 0).astype(np.uint8)
    return RestoreRows(live, src, rh, sh, ss, nkv, init, hs, block_size)


def restore_rows(name: str, seed: int = 0) -> RestoreRows:
    rng = np.random.default_rng(seed + 7919)
    w = get(name) if name in ("c0", "c0p", "c1", "c2", "c3", "c4") else None
    if name in ("c0", "c0p"):
        # one hit, one miss, one no-op, one more hit on the first hit's source
        perm = rng.permutation(16)
        live = perm[:4]
        src_slot = int(perm[4])
        src = [src_slot, -1, int(perm[5]), src_slot]
        nkv = [16, 32, 20, 32]
        init = [0, 0, 0, 0]
        return _rows(live, src, nkv, init, 16, rng)
    if name == "c1":
        perm = rng.permutation(w.num_slots)
        live, src = perm[:64], perm[64:128]
        nkv = 64 * rng.integers(1, 33, size=64)
        return _rows(live, src, nkv, np.zeros(64), 64, rng)
    if name == "c3":
        n = 512
        perm = rng.permutation(w.num_slots)
        live, ckpt = perm[:n], perm[n:]
        kinds = np.array([0] * 205 + [1] * 154 + [2] * 51 + [3] * 51 + [4] * 51)  # hit, miss, init, unaligned, zero
        rng.shuffle(kinds)
        hot = int(ckpt[0])
        src = np.full(n, -1, np.int64)
        nkv = 64 * rng.integers(1, 33, size=n)
        init = np.zeros(n, np.int64)
        hit_rows = np.nonzero(kinds == 0)[0]
        for j, r in enumerate(hit_rows):
            src[r] = hot if j % 2 == 0 else int(ckpt[rng.integers(1, len(ckpt))])
        init[kinds == 2] = 1
        src[kinds == 2] = ckpt[rng.integers(1, len(ckpt), size=int((kinds == 2).sum()))]
        un = kinds == 3
        nkv[un] = nkv[un] - rng.integers(1, 64, size=int(un.sum()))
        src[un] = ckpt[rng.integers(1, len(ckpt), size=int(un.sum()))]
        nkv[kinds == 4] = 0
        return _rows(live, src, nkv, init, 64, rng)
    raise KeyError(name)


def combo_rows(num_slots: int, block_size: int, seed: int = 0):
    """All 16 combinations nkv in {0, b, b+4, 2b} x initialized in {0, 1} x
    src in {-1, valid}, distinct live slots, sources outside the live set."""
    rng = np.random.default_rng(seed + 104729)
    assert num_slots >= 17
    perm = rng.permutation(num_slots)
    live, spare = perm[:16], perm[16:]
    combos = [(nk, ini, has) for nk in (0, block_size, block_size + 4, 2 * block_size)
              for ini in (0, 1) for has in (0, 1)]
    nkv = [c[0] for c in combos]
    init = [c[1] for c in combos]
    src = [int(spare[rng.integers(0, len(spare))]) if c[2] else -1 for c in combos]
    return _rows(live, src, nkv, init, block_size, rng)


# --------------------------------------------------------------------------
# decode and recurrence inputs

def decode_inputs(w: Workload, n_rows: int, seed: int = 0, layer: int = 0):
    """x ~ N(0,1), conv weights ~ N(0, 0.1), alpha = sigmoid(N(2,1)),
    beta = sigmoid(N(0,1)).  x and w are returned as float32 (the caller encodes
    them at the conv dtype)."""
    rng = np.random.default_rng(seed * 1000 + layer + 31)
    x = _normal_f32(rng, (n_rows, w.conv_dim))
    cw = (0.1 * _normal_f32(rng, (w.conv_dim, w.conv_width))).astype(np.float32)
    alpha = (1.0 / (1.0 + np.exp(-(2.0 + _normal_f32(rng, (n_rows, w.num_v_heads)))))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-_normal_f32(rng, (n_rows, w.num_v_heads))))).astype(np.float32)
    return x, cw, alpha, beta


def seq_lengths(n_seq: int, lo: int, hi: int, seed: int = 0):
    rng = np.random.default_rng(seed + 15485863)
    return rng.integers(lo, hi + 1, size=n_seq).astype(np.int32)


def prefill_inputs(w: Workload, lengths, seed: int = 0, layer: int = 0):
    """Inputs of the prefill conv: cu_seqlens int32, x ~ N(0,1) [T, conv_dim] and
    conv weights ~ N(0, 0.1) [conv_dim, conv_width], float32 (the caller encodes
    them at the conv dtype)."""
    rng = np.random.default_rng(seed * 1000 + layer + 43)
    lengths = np.asarray(lengths, np.int64)
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    x = _normal_f32(rng, (int(lengths.sum()), w.conv_dim))
    cw = (0.1 * _normal_f32(rng, (w.conv_dim, w.conv_width))).astype(np.float32)
    return cu, x, cw


def recurrent_inputs(w: Workload, lengths, seed: int = 0, layer: int = 0):
    """q, k ~ N(0,1) scaled to unit L2 norm per head; v ~ N(0,1);
    alpha = sigmoid(N(2,1)), beta = sigmoid(N(0,1)); cu_seqlens int32."""
    rng = np.random.default_rng(seed * 1000 + layer + 17)
    lengths = np.asarray(lengths, np.int64)
    T = int(lengths.sum())
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    q = _normal_f32(rng, (T, w.num_k_heads, w.head_k_dim))
    k = _normal_f32(rng, (T, w.num_k_heads, w.head_k_dim))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = _normal_f32(rng, (T, w.num_v_heads, w.head_v_dim))
    alpha = (1.0 / (1.0 + np.exp(-(2.0 + _normal_f32(rng, (T, w.num_v_heads)))))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-_normal_f32(rng, (T, w.num_v_heads))))).astype(np.float32)
    return cu, q.astype(np.float32), k.astype(np.float32), v, alpha, beta
