"""GPU: both copy forms of the restore -- 1-D TMA bulk copies through shared
memory (the default when the copied ranges are 16-byte multiples) and 16-byte
vectors through registers (LSC_RESTORE_COPY=vector, and shapes whose ranges
are not 16-byte multiples) -- are bit-exact against the oracle, padding and
untouched slots included."""
import numpy as np
import pytest

import oracle
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool
from test_gpu_parity import oracle_restore, run_restore, workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["default", "vector"])
@pytest.mark.parametrize("name", ["c0", "c0p", "s2", "s3", "s4"])
def test_restore_copy_forms_match_oracle(lsc, name, mode, monkeypatch):
    if mode == "vector":
        monkeypatch.setenv("LSC_RESTORE_COPY", "vector")
    else:
        monkeypatch.delenv("LSC_RESTORE_COPY", raising=False)
    w = workload(name, num_slots=max(W.get(name).num_slots if name.startswith("c") else 0, 24))
    rows = W.combo_rows(w.num_slots, w.block_size, seed=23)
    with DevPool(w, seed=5, random_padding=True) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        rc, rep, hs = run_restore(P, rows, w.block_size)
        assert rc == L.LSC_OK and rep.launches == 1
        rc_o, regions, hs_o = oracle_restore(w, P, pre, rows, w.block_size)
        assert rc_o == oracle.OK
        np.testing.assert_array_equal(hs, hs_o)
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])
        assert P.status() == L.LSC_OK


def test_bulk_restore_many_units_per_cta(lsc, monkeypatch):
    """128 hits over 3 GDN layers, about 11 units of 32 KiB per CTA (the
    ring of stages wraps several times): bit-exact against the oracle."""
    monkeypatch.delenv("LSC_RESTORE_COPY", raising=False)
    w = workload("s3", num_slots=256, layers=[W.GDN, W.GDN, W.ATTN, W.GDN])
    rng = np.random.default_rng(7)
    perm = rng.permutation(w.num_slots)
    n = 128
    rows = W._rows(perm[:n], perm[n:2 * n], [w.block_size] * n, [0] * n, w.block_size, rng)
    with DevPool(w, seed=6, random_padding=True) as P:
        pre = {l: P.host[l].copy() for l in P.gdn_layers}
        rc, rep, hs = run_restore(P, rows, w.block_size)
        assert rc == L.LSC_OK and rep.n_hit == n
        rc_o, regions, hs_o = oracle_restore(w, P, pre, rows, w.block_size)
        assert rc_o == oracle.OK
        np.testing.assert_array_equal(hs, hs_o)
        for l in P.gdn_layers:
            np.testing.assert_array_equal(P.download(l), regions[l])
        assert P.status() == L.LSC_OK
