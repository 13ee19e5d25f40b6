"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Sizes: the five measured configurations at their full shapes (all tokens where
the oracle finishes in seconds, a seeded sample of tokens otherwise, with the
same launch configuration the benchmark times), plus edge cases: empty and
invalid lists, ragged widths, every supported head count, forced split-KV
schedules, strided Q, padded pages, infinite sinks, run-to-run determinism.
"""
import numpy as np
import pytest
import torch

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD
from swa_paged_decode_gb300 import workloads as W
from tests._parity import compare, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    BLD.build()
    B.load()


def sample_tokens(T, n, seed=0):
    if T <= n:
        return np.arange(T)
    g = np.random.default_rng(seed)
    return np.sort(g.choice(T, size=n, replace=False))


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_config_full(cfg):
    w = W.make_config(cfg, device="cuda")
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"config{cfg}")


def test_config4_sampled():
    w = W.make_config(4, device="cuda")
    tok = sample_tokens(w.T, 24, seed=4)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w, tok), tokens=tok, what="config4")


@pytest.mark.parametrize("T", W.CONFIG5_BATCHES)
def test_config5_batches(T):
    w = W.make_config(5, T=T, device="cuda")
    tok = sample_tokens(T, 16, seed=T)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w, tok), tokens=tok, what=f"config5 T={T}")


def small(seed, *, T=6, H=32, swa_w=128, extra_w=256, swa_lens=(0, 128), extra_lens=(0, 256),
          swa_fmt=W.FMT_FP8_528, extra_fmt=W.FMT_NVFP4_288, sink=True, rope=True, invalid=0.1,
          page_pad=0, swa_slots=4096, extra_slots=8192):
    return W.make_workload(
        T=T, H=H, seed=seed, sink=sink, rope=rope, device="cuda", page_pad=page_pad,
        swa=dict(width=swa_w, lens=swa_lens, fmt=swa_fmt, page=64, slots=swa_slots),
        extra=None if extra_w == 0 else dict(width=extra_w, lens=extra_lens, fmt=extra_fmt,
                                             page=128, slots=extra_slots, invalid=invalid))


@pytest.mark.parametrize("H", [16, 32, 48, 64, 96, 128])
def test_every_head_count(H):
    w = small(100 + H, H=H, T=3)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"H={H}")


@pytest.mark.parametrize("swa_w,extra_w", [(1, 0), (7, 0), (100, 0), (129, 3), (128, 300),
                                           (255, 257), (5, 1000)])
def test_ragged_widths(swa_w, extra_w):
    w = small(7 + swa_w + extra_w, swa_w=swa_w, extra_w=extra_w, swa_lens=(0, swa_w + 2),
              extra_lens=(0, extra_w + 2))
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"widths {swa_w},{extra_w}")


@pytest.mark.parametrize("fmts", [(0, 0), (1, 1), (1, 0)])
def test_record_format_mixes(fmts):
    w = small(21, swa_fmt=fmts[0], extra_fmt=fmts[1])
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"formats {fmts}")


def test_empty_invalid_and_out_of_range_entries():
    w = small(31, T=8)
    S = w.swa_cache.num_slots
    w.swa.lens[0] = 0
    w.extra.lens[0] = 0                                  # token 0: nothing kept
    w.swa.ids[1, :] = -1                                 # token 1: all invalid
    w.extra.ids[1, :] = -1
    w.swa.ids[2, :40] = torch.tensor([-1, -7, S, S + 1, 2 ** 31 - 1] * 8, dtype=torch.int32)
    w.swa.lens[3] = 10 ** 6                              # clamp to width
    w.extra.lens[3] = -5                                 # clamp to 0
    w.swa.lens[4] = 1                                    # single row
    w.extra.lens[4] = 0
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what="edge entries")
    assert torch.all(out[:2] == 0) and torch.all(torch.isneginf(lse[:2]))


def test_single_row_lse_is_the_score():
    w = small(32, T=4, extra_w=0, swa_lens=(1, 1), rope=False, sink=False)
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what="length-1 lists")


@pytest.mark.parametrize("num_sms", [1, 3, 37, 1000])
def test_forced_split_schedules(num_sms):
    w = small(41, T=5, H=64)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=num_sms)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"num_sms={num_sms}")


@pytest.mark.parametrize("long_lists", [False, True])
def test_q_staging_forms_at_64_heads(long_lists):
    """Both forms of the 64-head kernel on the same kind of inputs: the
    producers stage Q and issue a token's first QK when the schedule gives
    few tiles per token segment (short lists), the softmax warps do with
    many (long lists on few CTAs)."""
    if long_lists:
        w = small(45, T=8, H=64, swa_w=128, extra_w=4096, extra_lens=(3000, 4096),
                  extra_slots=1 << 16)
        dec, out, lse, kept, chk = run_gpu(w, num_sms=2)
        assert dec.plan.producer_q == 0
    else:
        w = small(46, T=8, H=64, extra_lens=(1, 256))
        dec, out, lse, kept, chk = run_gpu(w, num_sms=3)
        assert dec.plan.producer_q == 1 and dec.plan.ctas_per_group > 1
    assert dec.plan.heads_per_group == 64
    compare(out, lse, kept, chk, oracle_ref(w), what=f"64 heads, long lists {long_lists}")


@pytest.mark.parametrize("num_sms", [16, 1000])
def test_split_tokens_merged_in_run_or_by_combine(num_sms):
    """Tokens of 72 tiles split over CTAs: on 16 SMs each spans a few CTAs and
    the run kernel merges it (the CTA that completes its units); on 1000 a
    token spans more than 64 CTAs and the combine kernel merges it."""
    w = small(47, T=8, H=64, extra_w=9000, extra_lens=(8000, 9000), extra_slots=1 << 16)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=num_sms)
    assert dec.plan.split_tokens > 0
    assert dec.plan.merge_in_run == (1 if num_sms == 16 else 0)
    compare(out, lse, kept, chk, oracle_ref(w), what=f"merge, num_sms={num_sms}")


def test_split_with_empty_partials():
    # Lengths so short that most split parts see no row at all.
    w = small(42, T=3, H=16, swa_lens=(0, 3), extra_lens=(0, 2))
    dec, out, lse, kept, chk = run_gpu(w, num_sms=1000)
    assert dec.plan.ctas_per_group > w.T
    compare(out, lse, kept, chk, oracle_ref(w), what="empty partials")


def test_strided_q_and_padded_pages():
    w = small(51, page_pad=32)
    big = torch.randn((w.T, w.H + 16, 520), device="cuda").to(torch.bfloat16)
    big[:, 3:3 + w.H, :512] = w.q
    w.q = big[:, 3:3 + w.H, :512]                     # strides (H+16)*520, 520
    assert w.q.stride(1) == 520
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what="strided q, padded pages")


def test_infinite_sinks():
    w = small(61, H=16)
    w.sink[:4] = float("inf")
    w.sink[4:8] = float("-inf")
    w.sink[8:] = 30.0
    dec, out, lse, kept, chk = run_gpu(w, num_sms=7)
    compare(out, lse, kept, chk, oracle_ref(w), what="infinite sinks")
    assert torch.all(out[:, :4] == 0)


def test_rope_table_edges():
    w = small(71)
    w.positions[:] = torch.tensor([0, 1, W.ROPE_TABLE_ROWS - 1, 65536, 12345, 7],
                                  device="cuda")[: w.T]
    dec, out, lse, kept, chk = run_gpu(w)
    compare(out, lse, kept, chk, oracle_ref(w), what="rope positions")


def test_deterministic_bitwise():
    w = small(81, T=5, H=64)
    dec = B.Decoder(w, num_sms=11)
    o1, l1 = [x.clone() for x in dec(w)]
    o2, l2 = dec(w)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_stream_and_workspace_reuse_across_shapes():
    s = torch.cuda.Stream()
    w1 = small(91, T=2, H=16)
    w2 = small(92, T=7, H=64, extra_w=0)
    with torch.cuda.stream(s):
        d1, o1, l1, k1, c1 = run_gpu(w1)
        d2, o2, l2, k2, c2 = run_gpu(w2)
    s.synchronize()
    compare(o1, l1, k1, c1, oracle_ref(w1), what="stream w1")
    compare(o2, l2, k2, c2, oracle_ref(w2), what="stream w2")


def test_default_kernel_is_tensor_core():
    for H in (16, 32, 64, 128):
        plan, _ = B.dsa_decode_plan(4, H, 128, 256, 0)
        assert plan.kernel == 1, H
    for H in (48, 96):
        plan, _ = B.dsa_decode_plan(4, H, 128, 256, 0)
        assert plan.kernel == 0, H


@pytest.mark.parametrize("H", [16, 64, 128])
def test_cuda_core_cross_check_kernel(monkeypatch, H):
    monkeypatch.setenv("DSA_DECODE_KERNEL", "simt")
    w = small(200 + H, H=H, T=4)
    dec, out, lse, kept, chk = run_gpu(w, num_sms=5)
    assert dec.plan.kernel == 0
    compare(out, lse, kept, chk, oracle_ref(w), what=f"simt H={H}")


def test_position_outside_table_sets_status():
    w = small(300, T=2)
    w.positions[1] = W.ROPE_TABLE_ROWS + 5
    dec = B.Decoder(w)
    dec(w)
    assert B.dsa_decode_read_status(dec.workspace) == -1


@pytest.mark.parametrize("cfg,T", [(3, None), (4, None), (3, 512)])
def test_work_balanced_ranges(cfg, T):
    """When the plan asks for it, the run kernel places the CTA boundaries so
    that every CTA gets the same work: 4 units per live tile plus 10 per
    token with a live tile (charged at its first live tile). The published
    ranges partition [0, U) and their work differs by at most the rounding
    of two boundaries to unit edges."""
    w = W.make_config(cfg, T=T, device="cuda")
    dec, out, lse, kept, chk = run_gpu(w)
    plan = dec.plan
    assert plan.balance_live == 1
    tok = sample_tokens(w.T, 24)
    compare(out, lse, kept, chk, oracle_ref(w, tokens=tok), tokens=tok, what=w.name)
    C = plan.ctas_per_group
    nb = (C + 1) * 8
    b = dec.workspace[plan.ws_bounds_offset: plan.ws_bounds_offset + nb].view(torch.int64).cpu().numpy()
    assert b[0] == 0 and b[-1] == plan.total_units and np.all(np.diff(b) > 0)
    tpt = plan.tiles_per_token
    cost = np.zeros(plan.total_units, dtype=np.int64)
    lists = [(w.swa, 0)] + ([(w.extra, plan.tiles_swa)] if w.extra is not None else [])
    lim = [(l.lens.clamp(0, l.width).cpu().numpy(), off) for l, off in lists]
    for t in range(w.T):
        first = None
        for lm, off in lim:
            nlive = -(-int(lm[t]) // 128)
            cost[t * tpt + off: t * tpt + off + nlive] = 4
            if nlive and first is None:
                first = t * tpt + off
        if first is not None:
            cost[first] += 10
    per = np.array([cost[b[c]:b[c + 1]].sum() for c in range(C)])
    assert per.max() - per.min() <= 2 * 14, (per.min(), per.max())
