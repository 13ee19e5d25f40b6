"""Pins of the fp64 oracle against facts it does not compute itself.

Each test uses something other than the oracle's own formula: a library
routine (torch float8 conversion, torch SDPA, logsumexp), a published value
table, a closed form, an invariant, or a brute-force Python loop.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from swa_paged_decode_gb300 import workloads as W
from tests import _indep as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(w, tokens=None, **over):
    a = W.oracle_args(w)
    a.update(over)
    return oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"], sink=a["sink"],
                         positions=a["positions"], cos_sin=a["cos_sin"], rope_style=a["rope_style"], tokens=tokens,
                         nthreads=2)


def small(seed=0, *, T=3, H=4, sink=True, rope=True, swa_w=16, extra_w=24, invalid=0.2,
          swa_fmt=W.FMT_FP8_528, extra_fmt=W.FMT_NVFP4_288, page_pad=0, swa_lens=(0, 20),
          extra_lens=(1, 24)):
    return W.make_workload(
        T=T, H=H, seed=seed, sink=sink, rope=rope, page_pad=page_pad,
        swa=dict(width=swa_w, lens=swa_lens, fmt=swa_fmt, page=16, slots=256),
        extra=None if extra_w == 0 else dict(width=extra_w, lens=extra_lens, fmt=extra_fmt,
                                             page=32, slots=512, invalid=invalid))


# ---------------------------------------------------------------- decoders

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = I.lib_e4m3(codes)
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])


def test_e2m1_all_codes_match_ocp_table():
    got = np.array([oracle.e2m1_value(c) for c in range(16)])
    assert np.array_equal(got, I.E2M1_TABLE)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_e4m3_spec_values_golden():
    # Values printed in the OCP 8-bit floating point spec (E4M3 column).
    for code, val in _golden_rows("e4m3_spec_values.txt"):
        assert oracle.e4m3_value(int(code, 16)) == float(val)


def test_fp8_record_layout_matches_library_decode():
    rng = np.random.default_rng(1)
    for _ in range(20):
        codes = rng.integers(0, 256, 512, dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x10  # no NaN codes
        scales = rng.uniform(1e-3, 3.0, 4).astype("<f4")
        rec = np.concatenate([codes, np.frombuffer(scales.tobytes(), dtype=np.uint8)])
        assert np.array_equal(oracle.dequant_record(rec, 0), I.lib_dequant(rec, 0))


def test_fp8_record_block_scale_index():
    # Block b of 128 dims must take the b-th scale: codes all 1.0, scales 1,2,4,8.
    rec = np.full(528, 0x38, dtype=np.uint8)
    rec[512:] = np.frombuffer(np.array([1, 2, 4, 8], dtype="<f4").tobytes(), dtype=np.uint8)
    k = oracle.dequant_record(rec, 0)
    assert np.array_equal(k, np.repeat([1.0, 2.0, 4.0, 8.0], 128))


def test_nvfp4_record_layout_matches_table_decode():
    rng = np.random.default_rng(2)
    for _ in range(20):
        data = rng.integers(0, 256, 256, dtype=np.uint8)
        sc = rng.integers(0, 256, 32, dtype=np.uint8)
        sc[(sc & 0x7F) == 0x7F] = 0x30
        rec = np.concatenate([data, sc])
        assert np.array_equal(oracle.dequant_record(rec, 1), I.lib_dequant(rec, 1))


def test_nvfp4_nibble_order_and_scale_index():
    # byte i = (hi << 4) | lo: element 2i is lo, 2i+1 is hi.
    rec = np.zeros(288, dtype=np.uint8)
    rec[:256] = (0x7 << 4) | 0x2          # even dims 1.0, odd dims 6.0
    rec[256:288] = 0x38                     # all scales 1.0
    rec[256 + 5] = 0x40                     # block 5 (dims 80..95) scale 2.0
    k = oracle.dequant_record(rec, 1)
    want = np.tile([1.0, 6.0], 256)
    want[80:96] *= 2.0
    assert np.array_equal(k, want)


# ------------------------------------------------------------- generator

def test_generator_fp8_roundtrip_within_e4m3_rounding():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(64, 512, generator=g)
    recs = W.encode_fp8_records(x).numpy()
    for i in range(64):
        k = oracle.dequant_record(recs[i], 0)
        sc = np.frombuffer(recs[i, 512:].tobytes(), dtype="<f4").astype(np.float64)
        s = np.repeat(sc, 128)
        err = np.abs(k - x[i].double().numpy())
        # half an e4m3 ulp: 2^-4 relative for normals, 2^-10 absolute (in code units) below
        assert np.all(err <= s * np.maximum(np.abs(x[i].double().numpy()) / s * 2.0 ** -4, 2.0 ** -10) * 1.0001)


def test_generator_nvfp4_roundtrip_within_e2m1_rounding():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(64, 512, generator=g)
    recs = W.encode_nvfp4_records(x).numpy()
    for i in range(64):
        k = oracle.dequant_record(recs[i], 1)
        s = np.repeat(I.lib_e4m3(recs[i, 256:]), 16)
        xi = x[i].double().numpy()
        err = np.abs(k - xi)
        # e2m1 half-gap (0.25 below 2, 0.5 below 4, 1 above) in scale units, plus
        # saturation at 6 when the e4m3 scale rounded down (at most 1/16 of absmax).
        y = np.abs(xi) / s
        half_gap = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
        assert np.all(err <= s * (half_gap + np.maximum(y - 6.0, 0.0)) * 1.0001 + 1e-12)
        assert np.dot(k, xi) / np.linalg.norm(k) / np.linalg.norm(xi) > 0.98


def test_rope_table_against_numpy():
    tab = W.rope_table(4096).double().numpy()
    p = np.arange(4096)[:, None]
    w = 10000.0 ** (-np.arange(32) * 2.0 / 64.0)
    ref = np.concatenate([np.cos(p * w), np.sin(p * w)], axis=1)
    assert np.all(np.abs(tab - ref) <= np.abs(ref) * 2.0 ** -24 + 1e-30)


# ------------------------------------------------------- attention core

def test_matches_torch_sdpa_fp64():
    w = small(5)
    out, lse, kept, chk = run(w)
    for t in range(w.T):
        K, keys = I.gather_rows(w, t)
        q = I.q_rows(w, t)
        assert kept[t] == len(keys)
        if len(keys) == 0:
            continue
        qt = torch.from_numpy(q)[None, :, None, :]
        Kt = torch.from_numpy(K)[None, None].expand(1, w.H, -1, -1)
        # sink = an extra key of logit `sink`, value 0: append a 513th dim.
        sk = w.sink.double().numpy()
        q2 = torch.cat([qt, torch.ones(1, w.H, 1, 1, dtype=torch.float64)], -1)
        K2 = torch.cat([Kt, torch.zeros(1, w.H, K.shape[0], 1, dtype=torch.float64)], -1)
        ksink = torch.zeros(1, w.H, 1, 513, dtype=torch.float64)
        ksink[0, :, 0, 512] = torch.from_numpy(sk) / w.scale
        K3 = torch.cat([K2, ksink], 2)
        V3 = torch.cat([K2[..., :512], torch.zeros(1, w.H, 1, 512, dtype=torch.float64)], 2)
        ref = F.scaled_dot_product_attention(q2, K3, V3, scale=w.scale)[0, :, 0]
        np.testing.assert_allclose(out[t], ref.numpy(), rtol=0, atol=1e-12)
        ref_lse = torch.logsumexp(w.scale * (qt[0, :, 0] @ torch.from_numpy(K).T), dim=-1)
        np.testing.assert_allclose(lse[t], ref_lse.numpy(), rtol=0, atol=1e-12)


def test_no_sink_matches_sdpa():
    w = small(6, sink=False, rope=False)
    out, lse, kept, _ = run(w)
    for t in range(w.T):
        K, _ = I.gather_rows(w, t)
        if K.shape[0] == 0:
            continue
        q = torch.from_numpy(I.q_rows(w, t))[None, :, None]
        Kt = torch.from_numpy(K)[None, None].expand(1, w.H, -1, -1)
        ref = F.scaled_dot_product_attention(q, Kt, Kt, scale=w.scale)[0, :, 0]
        np.testing.assert_allclose(out[t], ref.numpy(), rtol=0, atol=1e-12)


def test_bruteforce_python_loops_tiny():
    for seed in range(4):
        w = small(10 + seed, T=2, H=2, swa_w=3, extra_w=4, swa_lens=(0, 4), extra_lens=(0, 5),
                  invalid=0.3)
        out, lse, kept, chk = run(w)
        for t in range(w.T):
            K, keys = I.gather_rows(w, t)
            q = I.q_rows(w, t)
            assert kept[t] == len(keys) and int(chk[t]) == I.checksum(keys)
            for h in range(w.H):
                s = [w.scale * sum(q[h, d] * K[j, d] for d in range(512)) for j in range(len(keys))]
                if not s:
                    assert lse[t, h] == -math.inf and not out[t, h].any()
                    continue
                z = sum(math.exp(x) for x in s)
                den = z + math.exp(float(w.sink[h]))
                o = [sum(math.exp(s[j]) * K[j, d] for j in range(len(s))) / den for d in range(512)]
                assert abs(lse[t, h] - math.log(z)) < 1e-12
                np.testing.assert_allclose(out[t, h], o, rtol=0, atol=1e-12)


def test_two_key_closed_form():
    # q = e_0, two rows whose dim 0 decodes to a and b: out_0 = (e^{sa} a + e^{sb} b) / (e^{sa}+e^{sb}+e^{sink}).
    w = small(7, T=1, H=1, swa_w=2, extra_w=0, rope=False, swa_lens=(2, 2))
    w.q.zero_()
    w.q[0, 0, 0] = 1.0
    ids = w.swa.ids[0].tolist()
    out, lse, _, _ = run(w)
    a, b = (I.lib_dequant(I.cache_record(w.swa_cache, i), 0)[0] for i in ids)
    sa, sb, sk = w.scale * a, w.scale * b, float(w.sink[0])
    assert abs(lse[0, 0] - math.log(math.exp(sa) + math.exp(sb))) < 1e-14
    want = (math.exp(sa) * a + math.exp(sb) * b) / (math.exp(sa) + math.exp(sb) + math.exp(sk))
    assert abs(out[0, 0, 0] - want) < 1e-14


# ---------------------------------------------------- special cases / invariants

def test_constant_rows_give_that_row():
    w = small(8, sink=False)
    for c in (w.swa_cache, w.extra_cache):
        rb = c.record_bytes
        recs = c.data[:, :c.page_size * rb].view(c.num_pages, c.page_size, rb)
        recs[:] = recs[0, 0].clone()
    out, lse, kept, _ = run(w)
    row_fp8 = I.lib_dequant(I.cache_record(w.swa_cache, 0), 0)
    row_fp4 = I.lib_dequant(I.cache_record(w.extra_cache, 0), 1)
    for t in range(w.T):
        K, keys = I.gather_rows(w, t)
        if not keys:
            continue
        lids = {k[0] for k in keys}
        if lids == {0}:
            np.testing.assert_allclose(out[t], np.broadcast_to(row_fp8, out[t].shape), atol=1e-12)
        elif lids == {1}:
            np.testing.assert_allclose(out[t], np.broadcast_to(row_fp4, out[t].shape), atol=1e-12)


def test_length_one_list_returns_that_row():
    w = small(9, sink=False, extra_w=0, swa_lens=(1, 1))
    w.swa.ids[:, 0] = torch.tensor([3, 70, 255])[: w.T].to(torch.int32)
    out, lse, kept, _ = run(w)
    for t in range(w.T):
        k = I.lib_dequant(I.cache_record(w.swa_cache, int(w.swa.ids[t, 0])), 0)
        np.testing.assert_allclose(out[t], np.broadcast_to(k, out[t].shape), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[t], w.scale * I.q_rows(w, t) @ k, rtol=0, atol=1e-12)


def test_sink_scales_output_by_mass_ratio():
    w = small(11)
    out_s, lse_s, _, _ = run(w)
    out_n, lse_n, _, _ = run(w, sink=None)
    np.testing.assert_array_equal(lse_s, lse_n)      # lse excludes the sink
    z = np.exp(lse_n)
    ratio = z / (z + np.exp(w.sink.double().numpy())[None, :])
    np.testing.assert_allclose(out_s, out_n * ratio[..., None], rtol=0, atol=1e-13)


def test_sink_infinities():
    w = small(12)
    out_n, lse_n, _, _ = run(w, sink=None)
    out_p, lse_p, _, _ = run(w, sink=torch.full((w.H,), math.inf))
    out_m, lse_m, _, _ = run(w, sink=torch.full((w.H,), -math.inf))
    assert not out_p.any()
    np.testing.assert_array_equal(out_m, out_n)
    np.testing.assert_array_equal(lse_p, lse_n)


def test_rope_position_zero_is_identity():
    w = small(13)
    w.positions.zero_()
    out_r, lse_r, _, _ = run(w)
    out_n, lse_n, _, _ = run(w, cos_sin=None, positions=None)
    np.testing.assert_allclose(out_r, out_n, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse_r, lse_n, rtol=0, atol=1e-15)


def test_split_invariance_via_combine():
    w = small(14, T=2, swa_lens=(16, 16), extra_lens=(24, 24), invalid=0.0)
    out_full, lse_full, _, _ = run(w)
    # Partition the 40 candidate rows of each token into 3 parts by masking ids.
    parts = [(0, 0, 10), (0, 10, 16), (1, 0, 24)]
    p_out, p_lse = [], []
    for which in range(3):
        a = W.oracle_args(w)
        for li, l in enumerate(a["lists"]):
            ids = l["ids"].clone()
            keep = torch.zeros_like(ids, dtype=torch.bool)
            lid, r0, r1 = parts[which]
            if lid == li:
                keep[:, r0:r1] = True
            l["ids"] = torch.where(keep, ids, torch.full_like(ids, -1))
        o, l_, _, _ = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"],
                                    positions=a["positions"], cos_sin=a["cos_sin"], rope_style=a["rope_style"])
        p_out.append(o)
        p_lse.append(l_)
    out_c, lse_c = oracle.combine(p_out, p_lse, sink=w.sink.double().numpy()[None, :])
    np.testing.assert_allclose(out_c, out_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_c, lse_full, rtol=0, atol=1e-12)


def test_combine_with_empty_parts():
    o = np.random.default_rng(0).normal(size=(3, 2, 512))
    l = np.array([[0.5, -np.inf], [-np.inf, -np.inf], [1.0, -np.inf]])
    out, lse = oracle.combine(o, l)
    assert lse[1] == -np.inf and not out[1].any()
    w = np.exp([0.5, 1.0])
    np.testing.assert_allclose(out[0], (w[0] * o[0, 0] + w[1] * o[2, 0]) / w.sum(), atol=1e-14)


def test_permutation_invariance():
    w = small(15, swa_lens=(16, 16), extra_lens=(24, 24), invalid=0.1)
    out, lse, kept, chk = run(w)
    g = torch.Generator().manual_seed(0)
    for lst in (w.swa, w.extra):
        perm = torch.randperm(lst.width, generator=g)
        lst.ids[:] = lst.ids[:, perm]
    out2, lse2, kept2, chk2 = run(w)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)
    assert np.array_equal(kept, kept2)


def test_minus_one_and_out_of_range_equal_deletion():
    w = small(16, swa_lens=(16, 16), extra_lens=(24, 24), invalid=0.0)
    base_out, base_lse, base_kept, _ = run(w)
    # Deleting positions 3..5 of the sliding-window list (shift left, len -= 3)
    w2 = small(16, swa_lens=(16, 16), extra_lens=(24, 24), invalid=0.0)
    ids = w2.swa.ids.clone()
    w2.swa.ids[:] = torch.cat([ids[:, :3], ids[:, 6:], torch.full_like(ids[:, :3], -1)], 1)
    w2.swa.lens[:] = 13
    del_out, del_lse, del_kept, _ = run(w2)
    for bad in (-1, -7, 256, 257, 2 ** 31 - 1):        # 256 = number of slots
        w3 = small(16, swa_lens=(16, 16), extra_lens=(24, 24), invalid=0.0)
        w3.swa.ids[:, 3:6] = bad
        o3, l3, k3, _ = run(w3)
        np.testing.assert_allclose(o3, del_out, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l3, del_lse, rtol=0, atol=1e-13)
        assert np.array_equal(k3, base_kept - 3)


def test_lens_clamped_to_width_and_zero():
    w = small(17, invalid=0.0, swa_lens=(16, 16), extra_lens=(24, 24))
    o1, l1, k1, _ = run(w)
    w.swa.lens[:] = 1000
    w.extra.lens[:] = 24 + 5
    o2, l2, k2, _ = run(w)
    np.testing.assert_array_equal(o1, o2)
    w.swa.lens[:] = -5
    w.extra.lens[:] = 0
    o3, l3, k3, _ = run(w)
    assert not o3.any() and np.all(l3 == -np.inf) and not k3.any()


def test_page_padding_does_not_change_result():
    a = small(18, page_pad=0)
    b = small(18, page_pad=48)
    assert b.swa_cache.page_stride == 16 * 528 + 48
    oa, la, _, _ = run(a)
    ob, lb, _, _ = run(b)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


def test_token_subset_matches_full_run():
    w = small(19, T=5)
    out, lse, kept, chk = run(w)
    o2, l2, k2, c2 = run(w, tokens=[4, 1])
    np.testing.assert_array_equal(o2, out[[4, 1]])
    np.testing.assert_array_equal(c2, chk[[4, 1]])
