"""Shared test helpers: workload -> oracle pool, seeded host regions, golden files."""
import os

import numpy as np

import oracle
from linear_attention_state_lsc_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ODT = {W.F32: oracle.F32, W.BF16: oracle.BF16, W.F16: oracle.F16}


def oracle_pool(w: W.Workload, layers=None) -> oracle.Pool:
    kinds = [oracle.GDN if k == W.GDN else oracle.ATTENTION for k in (layers or w.layers)]
    return oracle.Pool(kinds, w.num_slots, w.conv_dim, w.conv_width, ODT[w.conv_dtype],
                       w.num_v_heads, w.head_v_dim, w.head_k_dim, ODT[w.ssm_dtype], w.page_bytes)


def oracle_layout(w: W.Workload):
    rc, L = oracle.layout(oracle_pool(w))
    assert rc == oracle.OK, rc
    return L


def views(w: W.Workload, L):
    """(offset, n_elems, dtype) of the conv and ssm views inside a page."""
    return [(0, L["conv_elems"], w.conv_dtype), (L["ssm_offset"], L["ssm_elems"], w.ssm_dtype)]


def host_regions(w: W.Workload, seed: int = 0, random_padding: bool = False):
    """{layer: uint8 region} filled with N(0,1) state and the workload's pad byte
    (or random bytes everywhere outside the views when random_padding)."""
    L = oracle_layout(w)
    out = {}
    for l in w.gdn_layers:
        reg = np.empty(w.num_slots * w.page_bytes, np.uint8)
        W.fill_region_host(reg, w.num_slots, w.page_bytes, views(w, L), w.pad_byte, seed * 1000 + l)
        if random_padding:
            rng = np.random.default_rng(seed * 7777 + l)
            noise = rng.integers(0, 256, size=reg.shape, dtype=np.uint8)
            pages, npg = reg.reshape(w.num_slots, w.page_bytes), noise.reshape(w.num_slots, w.page_bytes)
            mask = np.ones(w.page_bytes, bool)
            for off, n, dt in views(w, L):
                mask[off:off + n * W.ESIZE[dt]] = False
            pages[:, mask] = npg[:, mask]
        out[l] = reg
    return out


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def golden_kv(name):
    return {k: int(v) for k, v in read_golden(name)}


def payload_mask(w: W.Workload, L):
    """bool[page]: True on bytes that belong to the conv or ssm view."""
    m = np.zeros(w.page_bytes, bool)
    for off, n, dt in views(w, L):
        m[off:off + n * W.ESIZE[dt]] = True
    return m


LDT = {W.F32: 0, W.BF16: 1, W.F16: 2}


def lib_desc(w: W.Workload, layers=None):
    """Library pool description of a workload (include/lsc.h lsc_pool_desc)."""
    from linear_attention_state_lsc_gb300 import lsc
    kinds = [lsc.LSC_LAYER_GDN if k == W.GDN else lsc.LSC_LAYER_ATTENTION for k in (layers or w.layers)]
    return lsc.make_pool_desc(kinds, w.num_slots, w.conv_dim, w.conv_width, LDT[w.conv_dtype],
                              w.num_v_heads, w.head_v_dim, w.head_k_dim, LDT[w.ssm_dtype], w.page_bytes)


def ops_of(rows):
    from linear_attention_state_lsc_gb300 import lsc
    return lsc.ops_array(rows.live, rows.src, rows.restore_hash, rows.save_hash, rows.save_slot)


def gpu_present():
    """True when a CUDA device is visible.  Tests that build host-only pools on
    a stand-in base address make a valid (enqueuing) call only when this is
    False: with a device present the pool would be a device pool and the
    stand-in address would be dereferenced."""
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
