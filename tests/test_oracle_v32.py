"""Pins of the oracle's V3.2 record (FlashMLA's sparse_decode.h page:
bytes_per_token = 512 + 64*2 + (512/128)*4 for d_qk = 576, d_v = 512; read
as the 528-byte fp8 record -- 512 e4m3 codes, 4 little-endian fp32 scales,
one per 128 dims -- followed by the 64 further key dims as bf16).

Independent checks: a torch decode of the same bytes (float8_e4m3fn and
bfloat16 views, numpy's little-endian fp32), the scale index, the generator
round trip, and a brute-force fp64 attention written here from the
definition (576-dim scores, 512-dim values, the sink in the denominator)
against the whole oracle on small workloads; the oracle refuses a RoPE
table or a mix of record forms with this record."""
import numpy as np
import pytest
import torch

import oracle
from swa_paged_decode_gb300 import workloads as W


def torch_decode_v32(rec: np.ndarray) -> np.ndarray:
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    t = torch.from_numpy(rec.copy())
    codes = t[:512].view(torch.float8_e4m3fn).double().numpy()
    scales = np.frombuffer(rec[512:528].tobytes(), dtype="<f4").astype(np.float64)
    tail = t[528:656].clone().view(torch.bfloat16).double().numpy()
    return np.concatenate([codes * np.repeat(scales, 128), tail])


def random_record(rng):
    rec = rng.integers(0, 256, size=656, dtype=np.uint8)
    rec[:512] = rng.integers(0, 0x7F, size=512)                      # finite codes
    sc = (rng.standard_normal(4) * 2.0 ** rng.integers(-20, 20, size=4)).astype("<f4")
    rec[512:528] = np.frombuffer(sc.tobytes(), dtype=np.uint8)
    bf = rng.standard_normal(64).astype(np.float32) * np.float32(2.0 ** rng.integers(-8, 8))
    rec[528:656] = torch.from_numpy(bf).to(torch.bfloat16).view(torch.uint8).numpy()
    return rec


def test_record_size_is_the_pages_byte_count():
    assert W.RECORD_BYTES[W.FMT_V32_656] == 512 + 64 * 2 + (512 // 128) * 4 == 656
    assert oracle.RECORD_BYTES[oracle.FMT_V32_656] == 656
    assert W.FMT_V32_656 == oracle.FMT_V32_656


def test_decode_matches_torch_views():
    rng = np.random.default_rng(11)
    for _ in range(50):
        rec = random_record(rng)
        d = oracle.dequant_record(rec, oracle.FMT_V32_656)
        assert d.shape == (576,)
        np.testing.assert_array_equal(d, torch_decode_v32(rec))


def test_scale_index_and_tail():
    rng = np.random.default_rng(12)
    rec = random_record(rng)
    rec[:512] = rng.integers(1, 0x7E, size=512)
    base = oracle.dequant_record(rec, oracle.FMT_V32_656)
    for m in range(4):
        r2 = rec.copy()
        s = np.frombuffer(r2[512 + 4 * m:516 + 4 * m].tobytes(), dtype="<f4") * np.float32(2)
        r2[512 + 4 * m:516 + 4 * m] = np.frombuffer(s.tobytes(), dtype=np.uint8)
        d = oracle.dequant_record(r2, oracle.FMT_V32_656)
        blk = slice(128 * m, 128 * m + 128)
        np.testing.assert_array_equal(d[blk], 2 * base[blk])
        mask = np.ones(576, bool)
        mask[blk] = False
        np.testing.assert_array_equal(d[mask], base[mask])
    r3 = rec.copy()
    r3[528 + 2 * 7:528 + 2 * 8] = torch.tensor([3.0], dtype=torch.bfloat16).view(torch.uint8).numpy()
    d3 = oracle.dequant_record(r3, oracle.FMT_V32_656)
    assert d3[512 + 7] == 3.0
    mask = np.ones(576, bool)
    mask[512 + 7] = False
    np.testing.assert_array_equal(d3[mask], base[mask])


def test_generator_round_trip():
    g = torch.Generator().manual_seed(13)
    x = torch.randn((200, 576), generator=g) * torch.exp2(torch.randint(-12, 12, (200, 1), generator=g).float())
    recs = W.encode_v32_records(x).numpy()
    xd = x.double().numpy()
    for i in range(200):
        d = oracle.dequant_record(recs[i], oracle.FMT_V32_656)
        np.testing.assert_array_equal(d[512:], x[i, 512:].to(torch.bfloat16).double().numpy())
        for m in range(4):
            blk = slice(128 * m, 128 * m + 128)
            sc = np.abs(xd[i, blk]).max() / 448                      # the block's scale
            err = np.abs(d[blk] - xd[i, blk])
            assert np.all(err <= np.maximum(np.abs(xd[i, blk]) * 2.0 ** -4, sc * 2.0 ** -10) * 1.001)


def brute_force(w, tokens):
    """Attention written from the definition: kept rows of both lists, 576-dim
    scores, values = the rows' first 512 dims, sink in the denominator."""
    q = w.q.double().numpy()
    outs, lses = [], []
    for t in tokens:
        rows = []
        for cache, lst in ((w.swa_cache, w.swa), (w.extra_cache, w.extra)):
            if lst is None:
                continue
            data = cache.data.numpy()
            lim = min(max(int(lst.lens[t]), 0), lst.width)
            for r in range(lim):
                sid = int(lst.ids[t, r])
                if 0 <= sid < cache.num_slots:
                    page, off = divmod(sid, cache.page_size)
                    rows.append(torch_decode_v32(data[page, off * 656:(off + 1) * 656]))
        K = np.array(rows).reshape(-1, 576)
        s = w.scale * q[t] @ K.T                                     # [H, n]
        if K.shape[0] == 0:
            outs.append(np.zeros((w.H, 512)))
            lses.append(np.full(w.H, -np.inf))
            continue
        mx = s.max(axis=1, keepdims=True)
        e = np.exp(s - mx)
        z = e.sum(axis=1)
        den = z + (np.exp(w.sink.double().numpy() - mx[:, 0]) if w.sink is not None else 0.0)
        outs.append((e @ K[:, :512]) / den[:, None])
        lses.append(mx[:, 0] + np.log(z))
    return np.array(outs), np.array(lses)


@pytest.mark.parametrize("sink", [False, True])
def test_decode_against_brute_force(sink):
    w = W.make_workload(T=4, H=4, seed=14 + sink, sink=sink,
                        swa=dict(width=40, lens=(0, 40), fmt=W.FMT_V32_656, page=16, slots=256),
                        extra=dict(width=70, lens=(1, 70), fmt=W.FMT_V32_656, page=32, slots=512,
                                   invalid=0.2))
    assert w.q.shape == (4, 4, 576) and abs(w.scale - 576 ** -0.5) < 1e-15
    a = W.oracle_args(w)
    out, lse, _, _ = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"], sink=a["sink"])
    ro, rl = brute_force(w, range(4))
    np.testing.assert_allclose(out, ro, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)


def test_extra_dims_matter():
    # the 64 extra key dims enter the scores: zeroing Q's extra dims changes lse
    w = W.make_workload(T=2, H=2, seed=16,
                        swa=dict(width=8, lens=(8, 8), fmt=W.FMT_V32_656, page=16, slots=64))
    a = W.oracle_args(w)
    _, lse, _, _ = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"])
    q2 = w.q.clone()
    q2[..., 512:] = 0
    _, lse2, _, _ = oracle.decode(q2, a["caches"], a["lists"], scale=a["scale"])
    assert np.all(np.abs(lse - lse2) > 1e-6)


def test_rejects_rope_and_mixed_forms():
    w = W.make_workload(T=2, H=2, seed=17,
                        swa=dict(width=8, lens=(8, 8), fmt=W.FMT_V32_656, page=16, slots=64))
    a = W.oracle_args(w)
    with pytest.raises(ValueError):
        oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"],
                      positions=torch.zeros(2, dtype=torch.int64), cos_sin=W.rope_table(4))
    w2 = W.make_workload(T=2, H=2, seed=18,
                         swa=dict(width=8, lens=(8, 8), fmt=W.FMT_FP8_528, page=16, slots=64))
    b = W.oracle_args(w2)
    with pytest.raises((ValueError, AssertionError)):
        oracle.decode(a["q"], [a["caches"][0], b["caches"][0]], [a["lists"][0], b["lists"][0]],
                      scale=a["scale"])
