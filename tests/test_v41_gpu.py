"""GPU parity of the V4.1 variants through the C ABI against the fp64 oracle:
fp8-528 records with ue8m0 scales, GPT-J RoPE, and the MXFP8 output epilogue
(inverse GPT-J RoPE, ue8m0 scale per head and 32 dims, e4m3 codes, o-fused
layout), on the tensor-core kernel (16/32/64 heads per CTA), the CUDA-core
kernel (48 heads per CTA) and the combine kernel (forced split schedules).

MXFP8 codes are decisions taken in fp32 on the kernel's output, which differs
from the oracle's exact output within the decode tolerance; the comparison is
therefore on dequantized values (decode tolerance plus half an e4m3 step), on
the validity of every chunk's scale, and bit for bit where the kernel's fp32
output is exact: tokens with a single kept row, no sink and no RoPE, whose
output is that row's dequantized record.
"""
import numpy as np
import pytest
import torch

import oracle
from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import OUT_ATOL, compare, oracle_ref

pytestmark = pytest.mark.gpu

E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    B.load()


def v41(seed, *, T=6, H=64, swa_fmt=W.FMT_FP8_528_UE8M0, extra_fmt=W.FMT_NVFP4_288,
        swa_lens="full", extra_lens=(1, 300), extra_w=300, sink=True, rope=True,
        rope_style=W.ROPE_GPTJ, invalid=0.1):
    return W.make_workload(
        T=T, H=H, seed=seed, sink=sink, rope=rope, rope_style=rope_style, device="cuda",
        swa=dict(width=128, lens=swa_lens, fmt=swa_fmt, page=64, slots=1024),
        extra=None if extra_w == 0 else dict(width=extra_w, lens=extra_lens, fmt=extra_fmt,
                                             page=64, slots=4096, invalid=invalid))


def run(w, num_sms=0, mx_group=None):
    dec = B.Decoder(w, num_sms=num_sms, mx_group=mx_group)
    out, lse = dec(w)
    kept, chk = dec.selection()
    torch.cuda.synchronize()
    assert B.dsa_decode_read_status(dec.workspace) == 0
    return dec, out, lse, kept, chk


def fused(x, G):
    """[n, H, 512] -> o-fused [n, H/G, G*512] (slot ka = chunk * G + h % G)."""
    n, H, _ = x.shape
    return x.reshape(n, H // G, G, 16, 32).transpose(0, 1, 3, 2, 4).reshape(n, H // G, G * 512)


def mx_check(dec, w, ref, G, what):
    """GPU MXFP8 output against the oracle epilogue of the oracle's output."""
    r_out = ref[0]
    pos = None if w.positions is None else w.positions.cpu().numpy()
    cs = None if w.cos_sin is None else w.cos_sin.cpu()
    c_ref, s_ref, x_ref = oracle.mxfp8_epilogue(r_out, group_size=G, positions=pos, cos_sin=cs,
                                                rope_style=w.rope_style)
    codes = dec.mx.data.cpu().numpy()
    sc = dec.mx.scale_bytes().cpu().numpy()
    assert codes.shape == c_ref.shape and sc.shape == s_ref.shape
    E = sc.astype(np.int64) - 127
    step = np.repeat(np.ldexp(1.0, E), 32, axis=-1)               # per element of a slot
    v = E4M3[codes] * step
    x = fused(x_ref.astype(np.float64), G)
    # scales: a chunk's scaled amax lies in (224, 448], so its largest code is
    # in [224, 448] (values just above 224 round to 224), or the chunk is 0
    mag = np.abs(E4M3[codes]).reshape(*codes.shape[:2], -1, 32).max(axis=-1)
    zero = mag == 0
    assert np.all((mag[~zero] >= 224.0) & (mag[~zero] <= 448.0)), f"{what}: chunk scale"
    assert np.all(np.abs(sc.astype(np.int64) - s_ref.astype(np.int64)) <= 1), f"{what}: scale byte"
    # values: decode tolerance plus half an e4m3 step at the element's size
    tol = OUT_ATOL + np.abs(x) * 2.0 ** -4 * 1.001 + step * 2.0 ** -10
    err = np.abs(v - x)
    assert np.all(err <= tol), f"{what}: max excess {(err - tol).max()}"
    return float(err.max())


@pytest.mark.parametrize("fmts", [(2, 2), (2, 1), (0, 2)])
def test_ue8m0_records_bf16(fmts):
    w = v41(500 + fmts[0] * 3 + fmts[1], swa_fmt=fmts[0], extra_fmt=fmts[1],
            rope_style=W.ROPE_NEOX)
    dec, out, lse, kept, chk = run(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"ue8m0 formats {fmts}")


@pytest.mark.parametrize("H,num_sms", [(16, 0), (64, 0), (128, 0), (64, 1000), (48, 0),
                                       (96, 7)])
def test_gptj_rope_bf16(H, num_sms):
    w = v41(510 + H + num_sms, H=H, T=5)
    dec, out, lse, kept, chk = run(w, num_sms=num_sms)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"GPT-J H={H} sms={num_sms}")


@pytest.mark.parametrize("H,G,num_sms", [(64, 8, 0), (64, 1, 1000), (16, 4, 0), (16, 16, 37),
                                         (128, 2, 0), (48, 6, 0), (48, 3, 1000), (32, 8, 5)])
def test_mxfp8_output(H, G, num_sms):
    w = v41(520 + H + G + num_sms, H=H, T=5)
    dec, out, lse, kept, chk = run(w, num_sms=num_sms, mx_group=G)
    ref = oracle_ref(w)
    # lse and row selection as in the bf16 path
    r_out, r_lse, r_kept, r_chk = ref
    assert np.array_equal(kept.cpu().numpy(), r_kept)
    assert np.array_equal(chk.cpu().numpy().view(np.uint32), r_chk)
    l = lse.cpu().double().numpy()
    assert np.array_equal(np.isfinite(l), np.isfinite(r_lse))
    fin = np.isfinite(r_lse)
    assert np.abs(l[fin] - r_lse[fin]).max() <= 1e-3
    mx_check(dec, w, ref, G, f"MXFP8 H={H} G={G} sms={num_sms}")


def test_mxfp8_without_rope():
    w = v41(540, rope=False, T=4)
    dec, *_ = run(w, num_sms=300, mx_group=4)
    mx_check(dec, w, oracle_ref(w), 4, "MXFP8 without RoPE")


@pytest.mark.parametrize("H,num_sms", [(64, 0), (64, 1000), (48, 0), (16, 300)])
def test_mxfp8_single_row_bit_exact(H, num_sms):
    # One kept row per token, no sink, no RoPE: the output is the row itself,
    # exact in the kernel (f16 tiles are exact for these records), so codes
    # and scales must equal the oracle's bit for bit (+0 and -0 alike).
    w = v41(550 + H + num_sms, H=H, T=8, swa_lens=(1, 1), extra_w=0, sink=False, rope=False)
    G = 4
    dec, *_ = run(w, num_sms=num_sms, mx_group=G)
    ref = oracle_ref(w)
    c_ref, s_ref, _ = oracle.mxfp8_epilogue(ref[0], group_size=G)
    codes = dec.mx.data.cpu().numpy()
    canon = lambda c: np.where(c == 0x80, 0, c)
    assert np.array_equal(canon(codes), canon(c_ref))
    assert np.array_equal(dec.mx.scale_bytes().cpu().numpy(), s_ref)


def test_mxfp8_strided_buffers():
    # Padded token/group strides and scale words two apart: only the addressed
    # bytes change, with the same values as in a dense buffer.
    w = v41(560, H=64, T=4, swa_lens=(1, 1), extra_w=0, sink=False, rope=False)
    G = 8
    dense = B.Decoder(w, mx_group=G)
    dense(w)
    mx = B.MxOut(w.T, w.H, G, "cuda")
    data = torch.full((w.T, w.H // G + 1, G * 512 + 64), 0xA5, dtype=torch.uint8, device="cuda")
    scale = torch.full((w.T, w.H // G + 1, 2 * G * 4), 0x5A5A5A5A, dtype=torch.int32,
                       device="cuda")
    mx.data = data[:, :w.H // G, :G * 512]
    mx.scale = scale[:, :w.H // G, ::2]
    dec = B.Decoder(w, mx_group=G)
    dec.mx = mx
    dec(w)
    torch.cuda.synchronize()
    assert torch.equal(mx.data, dense.mx.data)
    assert torch.equal(mx.scale, dense.mx.scale)
    assert torch.all(data[:, w.H // G:, :] == 0xA5) and torch.all(data[:, :, G * 512:] == 0xA5)
    assert torch.all(scale[:, :, 1::2] == 0x5A5A5A5A) and torch.all(scale[:, w.H // G:, :] == 0x5A5A5A5A)


def test_cuda_core_kernel_v41(monkeypatch):
    monkeypatch.setenv("DSA_DECODE_KERNEL", "simt")
    w = v41(570, H=64, T=4)
    dec, out, lse, kept, chk = run(w, num_sms=5)
    assert dec.plan.kernel == 0
    compare(out, lse, kept, chk, oracle_ref(w), what="simt GPT-J ue8m0")
    dec, *_ = run(w, num_sms=5, mx_group=8)
    mx_check(dec, w, oracle_ref(w), 8, "simt MXFP8")
