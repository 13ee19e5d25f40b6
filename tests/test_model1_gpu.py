"""GPU parity of the MODEL1 record (584 B: 448 e4m3 dims with a ue8m0 scale
per 64, 64 bf16 RoPE dims, 1 unused byte; FlashMLA's sparse_decode.h page)
against the fp64 oracle, through the C ABI.

Records sit 8 bytes off the 16-byte grid at odd slots, so every case mixes
aligned and unaligned records. Cases: either list, both lists, every head
count (16/32/64/128 on tensor cores, 48/96 on the CUDA-core kernel), split
schedules, NeoX and GPT-J RoPE, rows at 2^-20 .. 2^10 scale, a RoPE part much
larger or smaller than the fp8 part (the row exponent takes both parts into
account), the CUDA-core cross-check and MXFP8 output."""
import numpy as np
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import compare, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu
M1 = W.FMT_MODEL1_584


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    B.load()


def wl(seed, *, H=64, T=6, swa_fmt=M1, extra_fmt=W.FMT_NVFP4_288, extra_w=300, swa_mag=(0,),
       extra_mag=(0,), q_log2=0, rope_style=W.ROPE_NEOX, sink=True):
    return W.make_workload(
        T=T, H=H, seed=seed, sink=sink, rope=True, device="cuda", q_log2=q_log2,
        rope_style=rope_style,
        swa=dict(width=128, lens=(1, 128), fmt=swa_fmt, page=64, slots=4096, mag=swa_mag),
        extra=None if extra_w == 0 else dict(width=extra_w, lens=(0, extra_w), fmt=extra_fmt,
                                             page=128, slots=8192, invalid=0.05, mag=extra_mag))


@pytest.mark.parametrize("fmts", [(M1, W.FMT_NVFP4_288), (W.FMT_FP8_528, M1), (M1, M1),
                                  (M1, W.FMT_FP8_528_UE8M0)])
def test_model1_in_either_list(fmts):
    w = wl(900 + fmts[1], swa_fmt=fmts[0], extra_fmt=fmts[1])
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"formats {fmts}")


@pytest.mark.parametrize("H", [16, 32, 48, 64, 96, 128])
def test_model1_every_head_count(H):
    w = wl(910 + H, H=H, T=3)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"MODEL1 H={H}")


@pytest.mark.parametrize("num_sms", [3, 40])
def test_model1_split_schedules(num_sms):
    w = wl(920 + num_sms, T=4, extra_fmt=M1, extra_w=900)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=num_sms)
    assert dec.plan.ctas_per_group > 1
    compare(out, lse, kept, chk, oracle_ref(w), what=f"MODEL1 num_sms={num_sms}")


def test_model1_gptj_rope():
    w = wl(930, rope_style=W.ROPE_GPTJ)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what="MODEL1 GPT-J")


@pytest.mark.parametrize("k", [-20, -10, 10])
def test_model1_scaled_rows(k):
    w = wl(940 + k, swa_mag=(k,), extra_fmt=M1, extra_mag=(k, 0) if k < 0 else (k,),
           q_log2=-k if k > 0 else 0)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"MODEL1 rows 2^{k}",
            out_scale=2.0 ** -k if k > 0 else 1.0)


@pytest.mark.parametrize("rope_log2", [-16, 12])
def test_model1_rope_part_far_from_fp8_part(rope_log2):
    """The bf16 RoPE dims drawn at 2^rope_log2 times the fp8 dims' scale:
    with a large RoPE part the row exponent comes from the bf16 values (the
    f16 tile would overflow otherwise); with a small one from the scales."""
    w = wl(950, extra_w=0, T=5, H=32, q_log2=-rope_log2 if rope_log2 > 0 else 0)
    g = torch.Generator(device="cuda").manual_seed(77)
    slots = w.swa_cache.num_slots
    x = torch.randn((slots, 512), generator=g, device="cuda")
    x[:, 448:] *= 2.0 ** rope_log2
    w.swa_cache.data[:, :64 * 584] = W.encode_model1_records(x).view(-1, 64 * 584)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"MODEL1 rope 2^{rope_log2}",
            out_scale=2.0 ** -rope_log2 if rope_log2 > 0 else 1.0)


@pytest.mark.parametrize("H", [16, 64])
def test_model1_cuda_core_cross_check(monkeypatch, H):
    monkeypatch.setenv("DSA_DECODE_KERNEL", "simt")
    w = wl(960 + H, H=H, T=4, extra_fmt=M1)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=5)
    assert dec.plan.kernel == 0
    compare(out, lse, kept, chk, oracle_ref(w), what=f"MODEL1 simt H={H}")


def test_model1_mxfp8_output_single_rows_exact():
    """Tokens with one kept row, no sink, no RoPE: the output is that row's
    decoded record, so the MXFP8 codes and scales must equal the oracle
    epilogue's bit for bit."""
    import oracle
    w = W.make_workload(T=5, H=16, seed=970, sink=False, rope=False, device="cuda",
                        swa=dict(width=16, lens=(1, 1), fmt=M1, page=64, slots=4096))
    G = 4
    dec = B.Decoder(w, mx_group=G)
    mx, lse = dec(w)
    torch.cuda.synchronize()
    assert B.dsa_decode_read_status(dec.workspace) == 0
    r_out = oracle_ref(w)[0]
    codes, scales, _ = oracle.mxfp8_epilogue(r_out, group_size=G)
    canon = lambda c: np.where(c == 0x80, 0, c)                # +0 and -0 alike
    assert np.array_equal(canon(mx.data.cpu().numpy()), canon(codes))
    assert np.array_equal(mx.scale_bytes().cpu().numpy(), scales)
