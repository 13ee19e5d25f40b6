"""Independent test-side helpers (not the oracle, not the CUDA path).

Record decoding here goes through torch's own float8_e4m3fn conversion and
the e2m1 value table printed in the OCP Microscaling spec, so it shares no
code with the oracle's bit-field decoders. The row gather is a plain Python
loop written from the selection rule (a second, independent loop nest).
"""
import numpy as np
import torch

# OCP MX spec, FP4 E2M1 value table (codes 0..15).
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                       -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def lib_e4m3(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def lib_dequant(rec: np.ndarray, fmt: int) -> np.ndarray:
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    if fmt == 0:
        codes = lib_e4m3(rec[:512])
        scales = np.frombuffer(rec[512:528].tobytes(), dtype="<f4").astype(np.float64)
        return codes * np.repeat(scales, 128)
    nib = np.empty(512, dtype=np.uint8)
    nib[0::2] = rec[:256] & 0xF
    nib[1::2] = rec[:256] >> 4
    return E2M1_TABLE[nib] * np.repeat(lib_e4m3(rec[256:288]), 16)


def cache_record(cache, sid: int) -> np.ndarray:
    data = cache.data.cpu().numpy()
    page, off = divmod(int(sid), cache.page_size)
    rb = cache.record_bytes
    return data[page, off * rb:(off + 1) * rb]


def gather_rows(w, t: int):
    """(K [n, 512] fp64, list of (list_id, position, id)) for token t."""
    rows, keys = [], []
    pairs = [(w.swa_cache, w.swa)] + ([(w.extra_cache, w.extra)] if w.extra is not None else [])
    for lid, (cache, lst) in enumerate(pairs):
        ln = int(lst.lens[t])
        limit = min(max(ln, 0), lst.width)
        for r in range(limit):
            sid = int(lst.ids[t, r])
            if 0 <= sid < cache.num_slots:
                rows.append(lib_dequant(cache_record(cache, sid), cache.fmt))
                keys.append((lid, r, sid))
    K = np.array(rows, dtype=np.float64).reshape(len(rows), 512)
    return K, keys


def q_rows(w, t: int) -> np.ndarray:
    """[H, 512] fp64 bf16 values of Q, RoPE applied via complex multiplication
    (NeoX: dims 448..479 are the real parts, 480..511 the imaginary parts)."""
    q = w.q[t].to(torch.float64).numpy().copy()
    if w.cos_sin is not None:
        row = w.cos_sin[int(w.positions[t])].to(torch.float64).numpy()
        rot = row[:32] + 1j * row[32:]
        z = (q[:, 448:480] + 1j * q[:, 480:512]) * rot[None, :]
        q[:, 448:480] = z.real
        q[:, 480:512] = z.imag
    return q


def fmix32(h: int) -> int:
    h &= 0xFFFFFFFF
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h


def checksum(keys) -> int:
    s = 0
    for lid, r, sid in keys:
        s = (s + fmix32((sid * 0x9E3779B1 + 2 * r + lid) & 0xFFFFFFFF)) & 0xFFFFFFFF
    return s
