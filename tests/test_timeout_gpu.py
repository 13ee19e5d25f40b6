"""Failure detection on the GPU without a fault: every device wait in the
tensor-core kernel is bounded, and a wait that runs out records
DSA_ERR_TIMEOUT in the status word, the kernel still returns (no trap, no
hang), and the device stays usable.

The test makes the waits run out on purpose: the plan's wait budget comes
from the DSA_DECODE_WAIT_BUDGET environment variable (read at planning time
only), set to one SM cycle, so the first wait that does not find its phase
already complete gives up. The kernel then stops issuing MMAs, lets every
role walk to the end, waits (with the full default budget) for the MMAs it
had issued, and frees its TMEM. The next call, planned without the variable,
must report DSA_OK and match the oracle.
"""
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import compare, oracle_ref, run_gpu

DSA_ERR_TIMEOUT = -6


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.load()


def test_budget_knob_goes_into_the_plan(lib, monkeypatch):
    plan, _ = B.dsa_decode_plan(4, 64, 128, 256, num_sms=152)
    assert plan.wait_budget_cycles == 0          # default: the kernel's ~2 s budget
    monkeypatch.setenv("DSA_DECODE_WAIT_BUDGET", "1")
    plan, _ = B.dsa_decode_plan(4, 64, 128, 256, num_sms=152)
    assert plan.wait_budget_cycles == 1


@pytest.mark.gpu
@pytest.mark.parametrize("cfg,T", [(5, 8), (3, None), (1, None)])
def test_expired_wait_reports_timeout_then_next_call_is_clean(lib, monkeypatch, cfg, T):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = W.make_config(cfg, T=T, device="cuda")
    monkeypatch.setenv("DSA_DECODE_WAIT_BUDGET", "1")
    dec = B.Decoder(w)
    monkeypatch.delenv("DSA_DECODE_WAIT_BUDGET")
    assert dec.plan.wait_budget_cycles == 1 and dec.plan.kernel == 1
    for _ in range(2):                                  # twice: the status word restarts per call
        dec(w)
        torch.cuda.synchronize()
        assert B.dsa_decode_read_status(dec.workspace) == DSA_ERR_TIMEOUT
    dec2, out, lse, kept, chk = run_gpu(w)              # asserts DSA_OK
    assert dec2.plan.wait_budget_cycles == 0
    tok = list(range(min(w.T, 8)))
    compare(out, lse, kept, chk, oracle_ref(w, tok), tokens=tok, what=f"after timeout {w.name}")
