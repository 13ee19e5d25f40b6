"""run + combine captured into a CUDA graph and replayed: the path allocates
nothing, never synchronizes and sets its kernels up once per device, so a
captured step must reproduce the direct call bit for bit, replay after
replay (a workload with split tokens, so the combine launch is captured
too)."""
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_graph_replay_matches_direct_call():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    B.load()
    w = W.make_config(3, device="cuda")
    dec = B.Decoder(w)
    assert dec.plan.ctas_per_group > 1            # the combine kernel runs
    out, lse = dec(w)                             # direct call (also does the one-time set-up)
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec(w)
    for _ in range(2):
        dec.out.fill_(float("nan"))
        dec.lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dec.out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(dec.lse.view(torch.int32), ref_lse.view(torch.int32))
        assert B.dsa_decode_read_status(dec.workspace) == 0


def test_graph_replay_v41_mxfp8():
    # run_v41 + combine_v41 + the MXFP8 cast, captured and replayed
    BLD.build()
    B.load()
    w = W.make_config(3, device="cuda", v41=True)
    dec = B.Decoder(w, mx_group=8)
    assert dec.plan.ctas_per_group > 1
    mx, lse = dec(w)
    torch.cuda.synchronize()
    ref = (mx.data.clone(), mx.scale.clone(), lse.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec(w)
    for _ in range(2):
        mx.data.fill_(0x7F)
        mx.scale.fill_(-1)
        dec.lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(mx.data, ref[0]) and torch.equal(mx.scale, ref[1])
        assert torch.equal(dec.lse.view(torch.int32), ref[2].view(torch.int32))
        assert B.dsa_decode_read_status(dec.workspace) == 0
