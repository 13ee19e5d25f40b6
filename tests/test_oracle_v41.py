"""Pins of the oracle's V4.1 pieces (the swapab page's fp8 record with ue8m0
scales, GPT-J RoPE, and the output epilogue: inverse RoPE, MXFP8 cast,
o-fused layout) against facts the oracle does not compute itself: library
routines (torch's float8 conversion, numpy ldexp and complex arithmetic),
closed forms, invariants and an independent torch implementation of the
cast and layout.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from swa_paged_decode_gb300 import workloads as W
from tests import _indep as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ------------------------------------------------------ ue8m0 fp8 records

def test_ue8m0_spec_values_golden():
    # E8M0 values printed in the OCP Microscaling (MX) spec.
    for code, val in _golden_rows("e8m0_spec_values.txt"):
        got = oracle.ue8m0_value(int(code, 16))
        if val == "NaN":
            assert math.isnan(got)
        else:
            assert got == float.fromhex(val)


def test_ue8m0_all_bytes_match_ldexp():
    for b in range(255):
        assert oracle.ue8m0_value(b) == np.ldexp(1.0, b - 127)
    assert math.isnan(oracle.ue8m0_value(255))


def test_ue8m0_record_matches_library_decode():
    rng = np.random.default_rng(11)
    for _ in range(20):
        codes = rng.integers(0, 256, 512, dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x10   # no NaN codes
        sc = rng.integers(100, 150, 16, dtype=np.uint8)
        rec = np.concatenate([codes, sc])
        assert np.array_equal(oracle.dequant_record(rec, 2), I.lib_dequant(rec, 2))


def test_ue8m0_record_scale_index():
    # Dims 32g .. 32g+31 take scale byte g: codes all 1.0, byte g = 119 + g.
    rec = np.full(528, 0x38, dtype=np.uint8)
    rec[512:] = 119 + np.arange(16, dtype=np.uint8)
    k = oracle.dequant_record(rec, 2)
    assert np.array_equal(k, np.repeat(np.ldexp(1.0, np.arange(16) - 8), 32))
    rec[512 + 5] = 0xFF                                 # NaN scale: exactly group 5
    k = oracle.dequant_record(rec, 2)
    assert np.isnan(k[160:192]).all() and not np.isnan(np.delete(k, np.s_[160:192])).any()


def test_generator_ue8m0_roundtrip_and_exponent_rule():
    g = torch.Generator().manual_seed(12)
    x = torch.randn(32, 512, generator=g) * 3.0
    recs = W.encode_fp8_ue8m0_records(x).numpy()
    xs = x.double().numpy()
    for i in range(32):
        k = oracle.dequant_record(recs[i], 2)
        e = recs[i, 512:].astype(np.int64) - 127
        amax = np.abs(xs[i].reshape(16, 32)).max(axis=1)
        # the smallest power of two with amax / 2^e <= 448
        assert np.all(amax <= 448.0 * np.ldexp(1.0, e))
        assert np.all(amax > 448.0 * np.ldexp(1.0, e - 1))
        s = np.ldexp(1.0, np.repeat(e, 32))
        err = np.abs(k - xs[i])
        assert np.all(err <= s * np.maximum(np.abs(xs[i]) / s * 2.0 ** -4, 2.0 ** -10) * 1.0001)


# ------------------------------------------------------------------ RoPE

def _rotated_q(style, q_bf16, row):
    """Rotated Q read back through the oracle: token t keeps one row whose key
    is the unit vector of dim 448 + t, and with scale 1 its lse is q_rot[448+t]."""
    n = 64
    recs = np.zeros((n, 528), dtype=np.uint8)
    recs[np.arange(n), 448 + np.arange(n)] = 0x38                    # 1.0
    recs[:, 512:] = np.frombuffer(np.ones(4, dtype="<f4").tobytes(), dtype=np.uint8)
    caches = [dict(bytes=recs.reshape(-1), num_pages=n, page_size=1, page_stride=528, format=0)]
    lists = [dict(ids=np.arange(n, dtype=np.int32)[:, None], lens=np.ones(n, dtype=np.int32),
                  width=1)]
    q = q_bf16.reshape(1, 1, 512).expand(n, 1, 512).contiguous()
    _, lse, _, _ = oracle.decode(q, caches, lists, scale=1.0,
                                 positions=np.zeros(n, dtype=np.int64),
                                 cos_sin=row.reshape(1, 64).astype(np.float32),
                                 rope_style=style, nthreads=2)
    return lse[:, 0]


@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_GPTJ])
def test_rope_matches_complex_rotation(style):
    g = torch.Generator().manual_seed(13 + style)
    q = torch.randn(512, generator=g).to(torch.bfloat16)
    ang = torch.rand(32, generator=g, dtype=torch.float64) * 2 * math.pi
    row = np.concatenate([np.cos(ang.numpy()), np.sin(ang.numpy())]).astype(np.float32)
    got = _rotated_q(style, q, row)
    want = q.double().numpy().copy()
    I.rotate_rope(want, row.astype(np.float64), style)
    assert np.allclose(got, want[448:], rtol=1e-12, atol=1e-12)


def test_gptj_and_neox_pair_different_dims():
    # Quarter turn on pair 0 only: GPT-J sends q[448] to -q[449], NeoX to -q[480].
    q = torch.zeros(512, dtype=torch.bfloat16)
    q[448], q[449], q[480] = 1.0, 2.0, 4.0
    row = np.zeros(64, dtype=np.float32)
    row[:32] = 1.0
    row[0], row[32] = 0.0, 1.0
    gj = _rotated_q(oracle.ROPE_GPTJ, q, row)
    nx = _rotated_q(oracle.ROPE_NEOX, q, row)
    assert gj[0] == pytest.approx(-2.0, abs=1e-12) and gj[1] == pytest.approx(1.0, abs=1e-12)
    assert nx[0] == pytest.approx(-4.0, abs=1e-12) and nx[32] == pytest.approx(1.0, abs=1e-12)


def test_gptj_workload_matches_independent_attention():
    w = W.make_workload(T=3, H=2, seed=14, sink=True, rope=True, rope_style=W.ROPE_GPTJ,
                        swa=dict(width=16, lens=(4, 16), fmt=W.FMT_FP8_528_UE8M0, page=16,
                                 slots=256),
                        extra=dict(width=24, lens=(1, 24), fmt=W.FMT_NVFP4_288, page=32,
                                   slots=512, invalid=0.2))
    a = W.oracle_args(w)
    out, lse, kept, _ = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"],
                                      sink=a["sink"], positions=a["positions"],
                                      cos_sin=a["cos_sin"], rope_style=a["rope_style"])
    for t in range(w.T):
        K, keys = I.gather_rows(w, t)
        assert kept[t] == len(keys)
        qr = I.q_rows(w, t)
        s = w.scale * qr @ K.T                                        # [H, n]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True) + np.exp(w.sink.double().numpy()[:, None] - m)
        assert np.allclose(lse[t], m[:, 0] + np.log(e.sum(axis=1)), rtol=1e-12, atol=1e-12)
        assert np.allclose(out[t], (e / den) @ K, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------- MXFP8 pieces

def test_e4m3_encode_matches_torch():
    codes = torch.arange(127, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).double()
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(15)
    ys = np.concatenate([vals.numpy(), mids.numpy(), np.nextafter(mids.numpy(), 0),
                         np.nextafter(mids.numpy(), 1000), rng.uniform(-460, 460, 4000),
                         rng.normal(0, 1e-2, 500), [0.0, -0.0, 1e-30, -1e-30, 463.9]])
    ys = ys.astype(np.float32)          # the cast's input is fp32
    ys = np.concatenate([ys, -ys])
    ref = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(y)) for y in ys], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_ue8m0_ceil_closed_forms():
    for k in range(-40, 40):
        p = math.ldexp(1.0, k)
        assert oracle.ue8m0_ceil(p) == 127 + k                       # exact power of two
        up = float(np.nextafter(np.float32(p), np.float32(np.inf)))
        assert oracle.ue8m0_ceil(up) == 128 + k                      # just above it
    rng = np.random.default_rng(16)
    for v in rng.lognormal(0, 8, 2000).astype(np.float32):
        b = oracle.ue8m0_ceil(float(v))
        assert math.ldexp(1.0, b - 128) < v <= math.ldexp(1.0, b - 127)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_mxfp8_matches_independent_cast_and_layout(G):
    rng = np.random.default_rng(17 + G)
    x = rng.normal(0, 1, (3, 4, 512)) * np.exp(rng.normal(0, 3, (3, 4, 1)))
    x[0, 1, 64:96] = 0.0                                            # all-zero chunk
    codes, scales, xo = oracle.mxfp8_epilogue(x, group_size=G)
    assert np.array_equal(xo, x.astype(np.float32))                 # no RoPE: rounding only
    rc, rs = I.lib_mxfp8(xo, G)
    assert np.array_equal(scales, rs)
    # +0 and -0 are the same value; everything else bit for bit
    assert np.array_equal(codes & np.where(codes == 0x80, 0, 0xFF), rc & np.where(rc == 0x80, 0, 0xFF))


def test_mxfp8_chunk_properties():
    rng = np.random.default_rng(18)
    x = rng.normal(0, 1, (4, 2, 512)) * np.exp(rng.normal(0, 4, (4, 2, 1)))
    codes, scales, xo = oracle.mxfp8_epilogue(x, group_size=1)
    table = I.lib_e4m3(np.arange(256, dtype=np.uint8))
    for r in range(4):
        for h in range(2):
            for cc in range(16):
                ka = cc
                e = int(scales[r, h, ka]) - 127
                cv = table[codes[r, h, ka * 32:(ka + 1) * 32]]
                xs = xo[r, h, 32 * cc:32 * cc + 32].astype(np.float64) * 2.0 ** -e
                amax = np.abs(xs).max()
                assert 224.0 < amax <= 448.0 * (1 + 2 ** -20)
                # each code is the nearest grid point of the scaled value
                grid = table[:127]
                best = np.abs(grid[None, :] - np.abs(xs)[:, None]).min(axis=1)
                assert np.allclose(np.abs(cv - xs), best, rtol=0, atol=0)


def test_mxfp8_scale_closed_forms():
    x = np.zeros((1, 1, 512))
    x[0, 0, 0:32] = 0.5
    x[0, 0, 3] = 448.0 * 2.0 ** -3                 # chunk max exactly 448 * 2^-3
    x[0, 0, 40] = float(np.nextafter(np.float32(448.0 * 4), np.float32(1e9)))   # just above 448 * 2^2
    codes, scales, _ = oracle.mxfp8_epilogue(x, group_size=1)
    assert scales[0, 0, 0] == 127 - 3 and codes[0, 0, 3] == 0x7E
    assert scales[0, 0, 1] == 127 + 3 and codes[0, 0, 32 + 8] == 0x76      # 224.0001 -> 224
    assert scales[0, 0, 2] == oracle.ue8m0_ceil(np.float32(1e-10) * np.float32(1.0 / 448.0))
    assert (codes[0, 0, 64:] == 0).all()


def test_mxfp8_o_fused_positions():
    # Head h, chunk cc holds the single value (h + 1) * 2^cc at dim 32cc + 7:
    # its scale lands at [h // G][cc*G + h%G], its code at byte 7 of that slot.
    H, G = 6, 3
    x = np.zeros((1, H, 512))
    for h in range(H):
        for cc in range(16):
            x[0, h, 32 * cc + 7] = (h + 1) * 2.0 ** cc
    codes, scales, _ = oracle.mxfp8_epilogue(x, group_size=G)
    for h in range(H):
        for cc in range(16):
            g, ka = h // G, cc * G + h % G
            assert scales[0, g, ka] == oracle.ue8m0_ceil(np.float32((h + 1) * 2.0 ** cc) * np.float32(1 / 448))
            slot = codes[0, g, ka * 32:(ka + 1) * 32]
            assert slot[7] != 0 and np.count_nonzero(slot) == 1


@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_GPTJ])
def test_inverse_rope_undoes_forward(style):
    rng = np.random.default_rng(19 + style)
    v = rng.normal(0, 1, (2, 3, 512))
    ang = rng.uniform(0, 2 * np.pi, (5, 32))
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    pos = np.array([4, 1], dtype=np.int64)
    fwd = v.copy()
    for r in range(2):
        I.rotate_rope(fwd[r], cs[pos[r]].astype(np.float64), style)
    _, _, xo = oracle.mxfp8_epilogue(fwd, group_size=1, positions=pos, cos_sin=cs,
                                     rope_style=style)
    assert np.allclose(xo, v, rtol=0, atol=1e-6)
    # dims below 448 untouched
    assert np.array_equal(xo[..., :448], fwd[..., :448].astype(np.float32))
