"""The checking build (libdsa_decode_debug.so, compiled with DSA_DEBUG): every
record, slot-id, Q and table read, every output and partial store and every
store into the shared-memory tiles is bounds-checked in the kernels; a failed
check skips the access and records DSA_ERR_BOUNDS (kind of check in word 1 of
the status block) instead of trapping.

Small cases (one token, 16 heads, list widths 1-3, every record format) and a
few larger ones run through it against the oracle: no check may fire and the
results must match. The negative case shrinks the extent the record check
uses (a test knob of the checking build, DSA_DEBUG_CHECK_EXTENT, read per
call) below the real cache: records past it are reported and skipped, never
read, so nothing outside the real allocation is touched."""
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import compare, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu
DSA_ERR_BOUNDS = -8
FORMATS = (W.FMT_FP8_528, W.FMT_NVFP4_288, W.FMT_FP8_528_UE8M0, W.FMT_MODEL1_584)


@pytest.fixture(scope="module", autouse=True)
def checking_build():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    BLD.build(debug=True)
    B.load()
    B.use_checking_build(True)
    yield
    B.use_checking_build(False)


def wl(seed, *, T=1, H=16, swa_w=3, extra_w=2, swa_fmt=W.FMT_FP8_528, extra_fmt=W.FMT_NVFP4_288,
       lens="full", rope_style=W.ROPE_NEOX):
    lens_s = lens if lens == "full" else (0, swa_w)
    lens_e = lens if lens == "full" else (0, extra_w)
    return W.make_workload(
        T=T, H=H, seed=seed, sink=True, rope=True, device="cuda", rope_style=rope_style,
        swa=dict(width=swa_w, lens=lens_s, fmt=swa_fmt, page=64, slots=1024),
        extra=None if extra_w == 0 else dict(width=extra_w, lens=lens_e, fmt=extra_fmt, page=64,
                                              slots=1024, invalid=0.2))


@pytest.mark.parametrize("swa_w,extra_w", [(1, 0), (2, 1), (3, 3), (1, 3)])
@pytest.mark.parametrize("fmt", FORMATS)
def test_small_cases_no_check_fires(swa_w, extra_w, fmt):
    w = wl(1000 + 10 * swa_w + extra_w + 100 * fmt, swa_w=swa_w, extra_w=extra_w, swa_fmt=fmt,
           extra_fmt=FORMATS[(fmt + 1) % 4],
           rope_style=W.ROPE_GPTJ if fmt == W.FMT_FP8_528_UE8M0 else W.ROPE_NEOX)
    dec, out, lse, kept, chk = run_gpu(w)                    # asserts status DSA_OK
    compare(out, lse, kept, chk, oracle_ref(w), what=f"checking build {swa_w},{extra_w} fmt{fmt}")


@pytest.mark.parametrize("H,num_sms", [(64, 7), (128, 0), (32, 1000)])
def test_split_and_head_groups_no_check_fires(H, num_sms):
    w = wl(1100 + H, T=5, H=H, swa_w=128, extra_w=300, lens="ragged")
    dec, out, lse, kept, chk = run_gpu(w, num_sms=num_sms)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"checking build H={H}")


def test_mxfp8_output_no_check_fires():
    w = wl(1200, T=3, H=16, swa_w=64, extra_w=0, swa_fmt=W.FMT_FP8_528_UE8M0,
           rope_style=W.ROPE_GPTJ)
    dec = B.Decoder(w, num_sms=5, mx_group=4)
    dec(w)
    torch.cuda.synchronize()
    assert B.dsa_decode_read_status(dec.workspace) == 0


def test_record_check_fires_and_skips(monkeypatch):
    w = wl(1300, T=4, H=16, swa_w=64, extra_w=0)
    cache_bytes = w.swa_cache.data.numel()
    monkeypatch.setenv("DSA_DEBUG_CHECK_EXTENT", str(cache_bytes // 2))
    dec = B.Decoder(w)
    dec(w)
    torch.cuda.synchronize()
    assert B.dsa_decode_read_status(dec.workspace) == DSA_ERR_BOUNDS
    assert int(dec.workspace[4:8].view(torch.int32).item()) == 1      # kind: a record read
    monkeypatch.delenv("DSA_DEBUG_CHECK_EXTENT")
    dec2, out, lse, kept, chk = run_gpu(w)                  # the full extent again: clean
    compare(out, lse, kept, chk, oracle_ref(w), what="after the narrowed extent")
