"""CPU checks of the scaled-row inputs that the dynamic-range GPU tests use.

Scaling a source row by a power of two 2^k (the generator's ``mag`` option)
must give records that decode (oracle) to exactly 2^k times the records of
the unit row: for fp8 with fp32 scales the codes are unchanged and every
scale is multiplied by 2^k; for fp8 with ue8m0 scales the codes are
unchanged and every scale byte grows by k. This pins the generator's scaling
and the oracle's decoding of records far from unit scale (scale exponents
that f16 cannot hold), with no GPU involved.
"""
import numpy as np
import pytest
import torch

import oracle
from swa_paged_decode_gb300 import workloads as W


@pytest.mark.parametrize("fmt", [W.FMT_FP8_528, W.FMT_FP8_528_UE8M0])
@pytest.mark.parametrize("k", [-20, -10, 10, 16])
def test_scaled_records_decode_to_scaled_rows(fmt, k):
    g0 = torch.Generator().manual_seed(3)
    g1 = torch.Generator().manual_seed(3)
    unit = W.make_cache(64, 64, fmt, g0, "cpu")
    scaled = W.make_cache(64, 64, fmt, g1, "cpu", mag=(k,))
    a = unit.data.view(-1, 528).numpy()
    b = scaled.data.view(-1, 528).numpy()
    assert np.array_equal(a[:, :512], b[:, :512])            # same e4m3 codes
    if fmt == W.FMT_FP8_528_UE8M0:
        assert np.array_equal(b[:, 512:].astype(np.int64), a[:, 512:].astype(np.int64) + k)
    else:
        sa = a[:, 512:].copy().view(np.float32)
        sb = b[:, 512:].copy().view(np.float32)
        assert np.array_equal(sb, sa * np.float32(2.0 ** k))
    for r in range(0, 64, 7):
        da = oracle.dequant_record(a[r], fmt)
        db = oracle.dequant_record(b[r], fmt)
        assert np.array_equal(db, da * 2.0 ** k)


def test_mixed_magnitudes_cycle_per_slot():
    g = torch.Generator().manual_seed(5)
    c = W.make_cache(192, 64, W.FMT_FP8_528, g, "cpu", mag=(-20, -10, 0))
    s = c.data.view(-1, 528)[:, 512:].clone().view(torch.float32)   # [slots, 4]
    e = torch.log2(s.amax(dim=1)).round()
    # unit rows have block scales near 2^-7 (absmax of 128 N(0,1) ~ 3 / 448)
    assert torch.all((e[0::3] < -24) & (e[1::3] < -14) & (e[1::3] > -20) & (e[2::3] > -10))


def test_q_scale_is_exact():
    kw = dict(T=3, H=16, swa=dict(width=8, lens="full", fmt=W.FMT_FP8_528, page=64, slots=256))
    a = W.make_workload(seed=9, **kw)
    b = W.make_workload(seed=9, q_log2=-12, **kw)
    assert torch.equal(b.q.float(), a.q.float() * 2.0 ** -12)
    assert torch.equal(a.swa.ids, b.swa.ids) and torch.equal(a.swa_cache.data, b.swa_cache.data)
