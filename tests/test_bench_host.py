"""Host-side pieces of the benchmark (no GPU): the algorithmic accounting
the roofline divides by, the traffic record's scaling, and the V4.1 form of
a workload drawing the same inputs as the plain one."""
import torch

import bench
from swa_paged_decode_gb300 import workloads as W


def tiny(**kw):
    return W.make_workload(T=3, H=16, seed=5, sink=True, rope=True,
                           swa=dict(width=8, lens=(2, 8), fmt=W.FMT_FP8_528, page=4, slots=64),
                           extra=dict(width=5, lens=(0, 5), fmt=W.FMT_NVFP4_288, page=8,
                                      slots=128, invalid=0.3), **kw)


def test_algorithmic_counts_by_hand():
    w = tiny()
    rows = bytes_ = 0
    for cache, lst in ((w.swa_cache, w.swa), (w.extra_cache, w.extra)):
        for t in range(w.T):
            lim = min(max(int(lst.lens[t]), 0), lst.width)
            for r in range(lim):
                sid = int(lst.ids[t, r])
                if 0 <= sid < cache.num_slots:
                    rows += 1
                    bytes_ += cache.record_bytes
    a = bench.algorithmic(w)
    assert a["rows"] == rows and a["gathered_bytes"] == bytes_
    assert a["flops"] == 2 * 2 * 512 * w.H * rows
    ids = 4 * (8 + 5) * w.T
    q = w.T * w.H * 512 * 2
    lse = w.T * w.H * 4
    assert a["total_bytes"] == bytes_ + ids + q + w.T * w.H * 512 * 2 + lse
    m = bench.algorithmic(w, mx=True)
    assert m["total_bytes"] == bytes_ + ids + q + w.T * w.H * (512 + 16) + lse


def test_traffic_record_scales_with_rows_and_is_keyed_to_the_sources():
    full = bench.NCU_TRAFFIC["rows_per_launch"]
    if bench.sources_hash() == bench.NCU_TRAFFIC["sources"]:
        assert bench.ncu_traffic(full) == bench.NCU_TRAFFIC["bytes_per_launch"]
        assert abs(bench.ncu_traffic(4 * full) - 4 * bench.NCU_TRAFFIC["bytes_per_launch"]) <= 4
    else:
        assert bench.ncu_traffic(full) is None


def test_v41_form_draws_the_same_inputs():
    a = W.make_config(2, T=8)
    b = W.make_config(2, T=8, v41=True)
    assert b.swa_cache.fmt == W.FMT_FP8_528_UE8M0 and b.extra_cache.fmt == W.FMT_FP8_528_UE8M0
    assert b.rope_style == W.ROPE_GPTJ and b.name.endswith("_v41")
    for x, y in ((a.q, b.q), (a.swa.ids, b.swa.ids), (a.swa.lens, b.swa.lens),
                 (a.extra.ids, b.extra.ids), (a.extra.lens, b.extra.lens), (a.sink, b.sink)):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
    assert a.swa_cache.data.shape == b.swa_cache.data.shape


class _FakeDec:
    """CPU stand-in for the decoder buffers the parity record reads."""

    def __init__(self, out, lse, kept, chk):
        self.out, self.lse, self._k, self._c = out, lse, kept, chk

    def selection(self):
        return self._k, self._c


class _FakeStep:
    def __init__(self, w, dec):
        self.w, self.dec = w, dec


def test_parity_record_passes_on_oracle_output_and_catches_errors():
    import numpy as np

    import oracle
    w = tiny()
    a = W.oracle_args(w)
    res = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"], sink=a["sink"],
                        positions=a["positions"], cos_sin=a["cos_sin"], rope_style=a["rope_style"])
    tok = np.arange(w.T)
    ref = (tok, *res)
    out = torch.from_numpy(res[0]).to(torch.bfloat16)
    lse = torch.from_numpy(res[1]).float()
    kept = torch.from_numpy(res[2])
    chk = torch.from_numpy(res[3].view(np.int32))
    rec = bench.parity_record(_FakeStep(w, _FakeDec(out, lse, kept, chk)), ref, mx=False)
    assert rec["pass"] and rec["tokens_checked"] == w.T and rec["selection_exact"]
    bad = out.clone()
    bad[1, 2, 7] += 0.05                       # one element past the 2e-2 bound
    assert not bench.parity_record(_FakeStep(w, _FakeDec(bad, lse, kept, chk)), ref, False)["pass"]
    kb = kept.clone()
    kb[0] += 1                                 # selection off by one row
    assert not bench.parity_record(_FakeStep(w, _FakeDec(out, lse, kb, chk)), ref, False)["pass"]
    lb = lse.clone()
    lb[2, 0] += 2e-3
    assert not bench.parity_record(_FakeStep(w, _FakeDec(out, lb, kept, chk)), ref, False)["pass"]
