"""GPU parity over the dynamic range of the KV records.

The kernel writes each fp8 row into its f16 tile normalized by 2^-e (e the
exponent of the row's largest block scale) and puts 2^e back in the softmax,
so rows of any magnitude keep f16 precision. These cases draw the source rows
at 2^k times unit scale (k = -20, -10, +10, +16; a token's rows all small, or
mixed per slot) for both fp8 record forms (fp32 scales per 128 dims, ue8m0
scales per 32 dims, whose exponents then fall far outside f16's range), and
NVFP4 rows whose e4m3 block scales are subnormal. Where Q is scaled by 2^-k
the scores stay in the unit range, as in a real layer; the absolute bound on
out then applies to out * 2^-k (the bound is stated for unit-scale rows), the
cosine, lse and selection bounds unchanged.
"""
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import compare, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

FP8 = (W.FMT_FP8_528, W.FMT_FP8_528_UE8M0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    B.load()


def wl(seed, *, fmt, mag, q_log2=0, extra=None, H=64, T=6, lens=(1, 128), sink=True):
    return W.make_workload(
        T=T, H=H, seed=seed, sink=sink, rope=True, device="cuda", q_log2=q_log2,
        rope_style=W.ROPE_GPTJ if fmt == W.FMT_FP8_528_UE8M0 else W.ROPE_NEOX,
        swa=dict(width=128, lens=lens, fmt=fmt, page=64, slots=4096, mag=mag), extra=extra)


@pytest.mark.parametrize("fmt", FP8)
@pytest.mark.parametrize("k", [-20, -10])
def test_small_rows_unit_q(fmt, k):
    """Every kept row of every token is small: scores near 0, so the softmax
    is near uniform and out is an average of 2^k-scale rows."""
    w = wl(400 + k, fmt=fmt, mag=(k,))
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"fmt{fmt} rows 2^{k}", out_scale=2.0 ** -k)


@pytest.mark.parametrize("fmt", FP8)
@pytest.mark.parametrize("k", [-20, -10, 10, 16])
def test_scaled_rows_unit_scores(fmt, k):
    """Rows at 2^k, Q at 2^-k: scores in the unit range, out at 2^k."""
    w = wl(500 + k, fmt=fmt, mag=(k,), q_log2=-k)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"fmt{fmt} rows 2^{k} q 2^{-k}",
            out_scale=2.0 ** -k)


@pytest.mark.parametrize("fmt", FP8)
@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_mixed_magnitudes_per_slot(fmt, H):
    """Slots cycle through 2^-20, 2^-10, 2^0: every token mixes magnitudes
    (the output follows its unit-scale rows)."""
    extra = dict(width=300, lens=(0, 300), fmt=W.FMT_NVFP4_288, page=128, slots=8192,
                 mag=(0, -6, -8))
    w = wl(600 + H, fmt=fmt, mag=(-20, -10, 0), H=H, extra=extra)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"fmt{fmt} mixed H={H}")


@pytest.mark.parametrize("fmt", FP8)
def test_small_rows_split_schedule(fmt):
    """Rows at 2^-20 with the work split over many CTAs (partials + combine)."""
    extra = dict(width=1000, lens=(500, 1000), fmt=fmt, page=64, slots=8192, mag=(-20,))
    w = wl(700, fmt=fmt, mag=(-20,), q_log2=20, extra=extra, T=3)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=40)
    assert dec.plan.ctas_per_group > w.T
    compare(out, lse, kept, chk, oracle_ref(w), what=f"fmt{fmt} split 2^-20", out_scale=2.0 ** 20)


@pytest.mark.parametrize("k", [-6, -8])
def test_nvfp4_subnormal_block_scales(k):
    """NVFP4 rows at 2^-6 and 2^-8: their e4m3 block scales (absmax / 6) are
    e4m3 subnormals; e2m1 times such a scale is still an exact f16 normal."""
    extra = dict(width=512, lens=(1, 512), fmt=W.FMT_NVFP4_288, page=256, slots=8192, mag=(k,))
    w = wl(800 - k, fmt=W.FMT_FP8_528, mag=(k,), q_log2=-k, extra=extra)
    codes = w.extra_cache.data.view(-1, 288)[:, 256:]
    assert bool(((codes & 0x78) == 0).any()), "expected e4m3 subnormal scale codes"
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"nvfp4 2^{k}", out_scale=2.0 ** -k)
