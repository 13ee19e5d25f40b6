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
    if fmt == 2:   # ue8m0 byte b = 2^(b - 127), one per 32 dims
        codes = lib_e4m3(rec[:512])
        return np.ldexp(codes, np.repeat(rec[512:528].astype(np.int64) - 127, 32))
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
        rotate_rope(q, row, getattr(w, "rope_style", 0))
    return q


def rotate_rope(x: np.ndarray, row: np.ndarray, style: int, inverse: bool = False) -> None:
    """In place on x [..., 512]: the rope dims as complex numbers times
    cos + i sin (conjugate for the inverse). NeoX (style 0): real parts are
    dims 448..479, imaginary parts 480..511; GPT-J (style 1): real parts the
    even dims of 448..511, imaginary parts the odd ones."""
    rot = row[:32] + 1j * row[32:]
    if inverse:
        rot = np.conj(rot)
    if style == 0:
        re, im = slice(448, 480), slice(480, 512)
    else:
        re, im = slice(448, 512, 2), slice(449, 512, 2)
    z = (x[..., re] + 1j * x[..., im]) * rot
    x[..., re] = z.real
    x[..., im] = z.imag


def lib_mxfp8(x: np.ndarray, G: int):
    """MXFP8 cast and o-fused layout of fp32 values x [n, H, 512] with torch
    ops: per (head, 32 dims) amax (floor 1e-10) times fp32(1/448) in fp32,
    exponent = ceil(log2) of that (float64 log2 of an fp32 value), codes by
    torch's round-to-nearest-even float8_e4m3fn conversion of x * 2^-exponent
    (clamped to +-448: a saturating cast). Returns (codes [n, H/G, G*512],
    scale bytes [n, H/G, G*16])."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    n, H, _ = t.shape
    c = t.reshape(n, H, 16, 32)
    amax = c.abs().amax(dim=-1).clamp(min=1e-10)
    v = amax * torch.tensor(1.0 / 448.0, dtype=torch.float32)
    e = torch.ceil(torch.log2(v.double()))
    y = (c.double() * torch.exp2(-e)[..., None]).clamp(-448.0, 448.0).float()
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)          # [n, H, 16, 32]
    sc = (e + 127).clamp(0, 254).to(torch.uint8)                  # [n, H, 16]
    # o-fused: group g = h // G, slot ka = chunk * G + h % G
    codes = codes.reshape(n, H // G, G, 16, 32).permute(0, 1, 3, 2, 4).reshape(n, H // G, G * 512)
    sc = sc.reshape(n, H // G, G, 16).permute(0, 1, 3, 2).reshape(n, H // G, G * 16)
    return codes.numpy(), sc.numpy()


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
