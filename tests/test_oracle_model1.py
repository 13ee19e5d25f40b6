"""Pins of the oracle's MODEL1 record (FlashMLA's sparse_decode.h page:
bytes_per_token = 448 + 64*2 + (448/64)*1 + 1 for d_qk = d_v = 512, read in
the order the terms are summed: 448 e4m3 codes, 64 bf16 values, 7 scale
bytes of one per 64 fp8 dims, 1 unused byte).

Independent checks: a torch decode of the same bytes (float8_e4m3fn and
bfloat16 views, numpy ldexp for the ue8m0 scales), the scale index (one byte
scales exactly its 64 dims), NaN poisoning, the unused byte, the generator
round trip and the decode path through the whole oracle (a length-1 list
returns the record's row, lse = its score)."""
import numpy as np
import torch

import oracle
from swa_paged_decode_gb300 import workloads as W


def torch_decode_model1(rec: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(rec.copy())
    codes = t[:448].view(torch.float8_e4m3fn).double().numpy()
    sc = np.ldexp(1.0, rec[576:583].astype(np.int64) - 127).astype(np.float64)
    sc[rec[576:583] == 0xFF] = np.nan
    nope = codes * np.repeat(sc, 64)
    rope = t[448:576].clone().view(torch.bfloat16).double().numpy()
    return np.concatenate([nope, rope])


def random_record(rng):
    rec = rng.integers(0, 256, size=584, dtype=np.uint8)
    rec[576:583] = rng.integers(100, 150, size=7)                     # scales 2^-27 .. 2^22
    bf = rng.standard_normal(64).astype(np.float32) * np.float32(2.0 ** rng.integers(-8, 8))
    rec[448:576] = torch.from_numpy(bf).to(torch.bfloat16).view(torch.uint8).numpy()
    return rec


def test_record_size_is_the_pages_byte_count():
    assert W.RECORD_BYTES[W.FMT_MODEL1_584] == 448 + 64 * 2 + (448 // 64) * 1 + 1 == 584
    assert oracle.RECORD_BYTES[oracle.FMT_MODEL1_584] == 584


def test_decode_matches_torch_views():
    rng = np.random.default_rng(1)
    for _ in range(50):
        rec = random_record(rng)
        np.testing.assert_array_equal(oracle.dequant_record(rec, 3), torch_decode_model1(rec))


def test_scale_index_nan_and_unused_byte():
    rng = np.random.default_rng(2)
    rec = random_record(rng)
    rec[:448] = rng.integers(1, 0x7E, size=448)                      # finite, non-zero codes
    base = oracle.dequant_record(rec, 3)
    for m in range(7):
        r2 = rec.copy()
        r2[576 + m] += 1                                             # doubles dims 64m..64m+63
        d = oracle.dequant_record(r2, 3)
        np.testing.assert_array_equal(d[64 * m:64 * m + 64], 2 * base[64 * m:64 * m + 64])
        mask = np.ones(512, bool)
        mask[64 * m:64 * m + 64] = False
        np.testing.assert_array_equal(d[mask], base[mask])
        r3 = rec.copy()
        r3[576 + m] = 0xFF                                           # E8M0 NaN: exactly those dims
        d3 = oracle.dequant_record(r3, 3)
        assert np.all(np.isnan(d3[64 * m:64 * m + 64])) and not np.any(np.isnan(d3[mask]))
    r4 = rec.copy()
    r4[583] ^= 0xA5
    np.testing.assert_array_equal(oracle.dequant_record(r4, 3), base)


def test_generator_round_trip():
    g = torch.Generator().manual_seed(3)
    x = torch.randn((200, 512), generator=g) * torch.exp2(torch.randint(-12, 12, (200, 1), generator=g).float())
    recs = W.encode_model1_records(x).numpy()
    xd = x.double().numpy()
    for i in range(200):
        d = oracle.dequant_record(recs[i], 3)
        np.testing.assert_array_equal(d[448:], x[i, 448:].to(torch.bfloat16).double().numpy())
        for m in range(7):
            blk = slice(64 * m, 64 * m + 64)
            e = int(recs[i, 576 + m]) - 127
            amax = np.abs(xd[i, blk]).max()
            assert 224 < amax / 2.0 ** e <= 448                      # ceil(log2(amax / 448))
            err = np.abs(d[blk] - xd[i, blk])
            assert np.all(err <= np.maximum(np.abs(xd[i, blk]) * 2.0 ** -4, 2.0 ** (e - 10)) * 1.0001)
        assert recs[i, 583] == 0


def test_length_one_list_returns_the_row():
    w = W.make_workload(T=3, H=16, seed=4, swa=dict(width=4, lens=(1, 1), fmt=W.FMT_MODEL1_584,
                                                    page=64, slots=256))
    a = W.oracle_args(w)
    out, lse, kept, _ = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"])
    recs = w.swa_cache.data.view(-1, 584).numpy()
    q = w.q.double().numpy()
    for t in range(3):
        row = torch_decode_model1(recs[int(w.swa.ids[t, 0])])
        assert kept[t] == 1
        np.testing.assert_allclose(out[t], np.broadcast_to(row, (16, 512)), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], w.scale * q[t] @ row, rtol=1e-12, atol=1e-12)
