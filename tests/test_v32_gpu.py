"""GPU parity of the V3.2 record (656 B: the fp8-528 record of key dims
0..511 plus 64 bf16 key dims 512..575; 576-dim Q and keys, 512-dim values;
FlashMLA's sparse_decode.h page) against the fp64 oracle, through the C ABI.

Records sit 16 bytes off the 32-byte grid at odd slots, so every case mixes
both load paths (and padded pages the 16-byte fallback). Cases: every
supported head count (groups of at most 32 heads), ragged and empty lists,
split schedules, with and without a sink, rows at 2^-20 .. 2^10 scale, bf16
dims much larger or smaller than the fp8 ones (the row exponent takes both
into account), and a sampled workload at the size of the 128-token
configuration."""
import numpy as np
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import compare, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu
V32 = W.FMT_V32_656


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    B.load()


def wl(seed, *, H=64, T=6, swa_w=200, extra_w=300, swa_mag=(0,), extra_mag=(0,), q_log2=0,
       sink=True, page_pad=0):
    return W.make_workload(
        T=T, H=H, seed=seed, sink=sink, rope=False, device="cuda", q_log2=q_log2,
        page_pad=page_pad,
        swa=dict(width=swa_w, lens=(0, swa_w + 2), fmt=V32, page=64, slots=4096, mag=swa_mag),
        extra=None if extra_w == 0 else dict(width=extra_w, lens=(0, extra_w + 2), fmt=V32,
                                             page=128, slots=8192, invalid=0.05, mag=extra_mag))


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_v32_every_head_count(H):
    w = wl(1000 + H, H=H, T=3)
    dec, out, lse, kept, chk = run_gpu(w)
    assert dec.plan.d_qk == 576 and dec.plan.heads_per_group <= 32
    compare(out, lse, kept, chk, oracle_ref(w), what=f"V3.2 H={H}")


@pytest.mark.parametrize("sink", [False, True])
@pytest.mark.parametrize("page_pad", [0, 16])
def test_v32_load_paths_and_sink(sink, page_pad):
    w = wl(1010 + 2 * page_pad + sink, sink=sink, page_pad=page_pad)
    w.swa.lens[1] = 0
    w.extra.lens[1] = 0                                   # token 1: nothing kept
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"V3.2 pad {page_pad} sink {sink}")


@pytest.mark.parametrize("num_sms", [8, 40])
def test_v32_split_schedules(num_sms):
    w = wl(1030 + num_sms, T=4, extra_w=900)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=num_sms)
    assert dec.plan.ctas_per_group > 1
    compare(out, lse, kept, chk, oracle_ref(w), what=f"V3.2 num_sms={num_sms}")


def test_v32_single_list_ragged():
    w = wl(1040, extra_w=0, swa_w=5, T=7)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what="V3.2 one list, width 5")


@pytest.mark.parametrize("k", [-20, -10, 10])
def test_v32_scaled_rows(k):
    w = wl(1050 + k, swa_mag=(k,), extra_mag=(k, 0) if k < 0 else (k,),
           q_log2=-k if k > 0 else 0)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"V3.2 rows 2^{k}",
            out_scale=2.0 ** -k if k > 0 else 1.0)


@pytest.mark.parametrize("tail_log2", [-16, 12])
def test_v32_bf16_dims_far_from_fp8_dims(tail_log2):
    """Key dims 512..575 drawn at 2^tail_log2 times the fp8 dims: with large
    bf16 dims the row exponent comes from them (the f16 tile would overflow
    otherwise); with small ones from the scales."""
    w = wl(1060, extra_w=0, T=5, H=32, q_log2=-tail_log2 if tail_log2 > 0 else 0)
    g = torch.Generator(device="cuda").manual_seed(78)
    slots = w.swa_cache.num_slots
    x = torch.randn((slots, 576), generator=g, device="cuda")
    x[:, 512:] *= 2.0 ** tail_log2
    w.swa_cache.data[:, :64 * 656] = W.encode_v32_records(x).view(-1, 64 * 656)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"V3.2 tail 2^{tail_log2}")


def test_v32_config3_size_sampled():
    """The 128-token, 64-head configuration with every list in the V3.2 form
    (widths 128 and 2048, 2^20 extra slots), tokens sampled."""
    w = W.make_config(3, device="cuda", v32=True)
    tok = np.sort(np.random.default_rng(3).choice(w.T, size=12, replace=False))
    dec, out, lse, kept, chk = run_gpu(w)
    assert dec.plan.heads_per_group == 32 and dec.plan.head_groups == 2
    compare(out, lse, kept, chk, oracle_ref(w, tok), tokens=tok, what="config3 V3.2")
