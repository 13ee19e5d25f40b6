"""dsa_decode_run_noalloc: run + combine on the library's own static device
scratch. Collected last (file name). The GPU tests compare it, call after
call, with the caller-workspace entry points (dsa_decode_run then
dsa_decode_combine) on the same inputs; both launch the same kernels with
the same plan, so the results must agree bit for bit. The CPU tests check the
host-side refusals, which come before any CUDA call."""
import ctypes

import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W

MAX_BYTES = 48 * 1024 * 1024
DSA_ERR_INVALID_ARG, DSA_ERR_WORKSPACE, DSA_ERR_PLAN = -1, -4, -7


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.load()


def _call_raw(lib, plan):
    # Every pointer is NULL: only the plan checks run, no CUDA call is made.
    return lib.dsa_decode_run_noalloc(ctypes.byref(plan), None, 0, 0, None, None, 0, None, None,
                                      None, 0, None, None, None, None, 0, 1.0, None, None, None,
                                      None)


def test_noalloc_refuses_plan_above_limit(lib):
    # 2000 SMs' worth of split-KV partial slots: 2000 * 64 heads * 4 KiB > 48 MiB
    plan, nbytes = B.dsa_decode_plan(4096, 64, 128, 4096, num_sms=2000)
    assert nbytes > MAX_BYTES
    assert _call_raw(lib, plan) == DSA_ERR_WORKSPACE


def test_noalloc_refuses_bad_plan(lib):
    plan = B.Plan()
    assert _call_raw(lib, plan) == DSA_ERR_PLAN


def test_noalloc_limit_covers_measured_shapes():
    # every measured configuration on a 152-SM GB300 fits the static scratch
    for k, T in [(1, None), (2, None), (3, None), (4, None), (5, 1024)]:
        c = W.CONFIGS[k]
        Tk = c["T"] if T is None else T
        ew = 0 if c["extra"] is None else c["extra"]["width"]
        _, nbytes = B.dsa_decode_plan(Tk, c["H"], c["swa"]["width"], ew, num_sms=152)
        assert nbytes <= MAX_BYTES, (k, nbytes)


def _reference(w):
    dec = B.Decoder(w)
    out, lse = dec(w)
    torch.cuda.synchronize()
    return out.clone(), lse.clone(), dec.plan


def _noalloc(w, plan):
    out = torch.full((w.T, w.H, W.HEAD_DIM), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    B.dsa_decode_run_noalloc(plan, w.q, w.swa_cache, w.swa.ids, w.swa.lens, w.extra_cache,
                             None if w.extra is None else w.extra.ids,
                             None if w.extra is None else w.extra.lens, w.sink, w.positions,
                             w.cos_sin, w.scale, out, lse, device_status=st)
    torch.cuda.synchronize()
    return out, lse, int(st.item())


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_call_after_call(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    # workload 3 splits tokens across CTAs (partials + combine); workload 2
    # has another plan layout; then workload 3 again on the reused scratch.
    w3 = W.make_config(3, device="cuda")
    w2 = W.make_config(2, device="cuda")
    ref3 = _reference(w3)
    ref2 = _reference(w2)
    assert ref3[2].ctas_per_group > 1
    for w, (ro, rl, plan) in [(w3, ref3), (w2, ref2), (w3, ref3)]:
        out, lse, status = _noalloc(w, plan)
        assert status == B.DSA_OK
        assert torch.equal(out.view(torch.int16), ro.view(torch.int16)), w.name
        assert torch.equal(lse.view(torch.int32), rl.view(torch.int32)), w.name


@pytest.mark.gpu
def test_noalloc_repeated_calls_same_inputs(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = W.make_config(5, T=64, device="cuda")
    ro, rl, plan = _reference(w)
    a = _noalloc(w, plan)
    b = _noalloc(w, plan)
    for out, lse, status in (a, b):
        assert status == B.DSA_OK
        assert torch.equal(out.view(torch.int16), ro.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), rl.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_reports_kernel_status_then_clears_it(lib):
    """A condition the kernel records (a position outside the cos/sin table:
    DSA_ERR_INVALID_ARG) reaches the caller's status word through the shared
    scratch, and the next valid call reports DSA_OK again (the word is
    cleared per call, not left from the last one)."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = W.make_config(5, T=8, device="cuda")
    ro, rl, plan = _reference(w)
    good = w.positions.clone()
    w.positions[3] = w.cos_sin.shape[0] + 5
    _, _, status = _noalloc(w, plan)
    assert status == DSA_ERR_INVALID_ARG
    w.positions.copy_(good)
    out, lse, status = _noalloc(w, plan)
    assert status == B.DSA_OK
    assert torch.equal(out.view(torch.int16), ro.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), rl.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_zero_tokens_writes_ok_status(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    plan, _ = B.dsa_decode_plan(0, 64, 128, 0)
    st = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    rc = lib.dsa_decode_run_noalloc(ctypes.byref(plan), None, 0, 0, None, None, 0, None, None,
                                    None, 0, None, None, None, None, 0, 1.0, None, None,
                                    ctypes.c_void_p(st.data_ptr()), None)
    torch.cuda.synchronize()
    assert rc == B.DSA_OK and int(st.item()) == B.DSA_OK
