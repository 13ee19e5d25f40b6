"""Seeded synthetic inputs for paged sparse/sliding-window MQA decode.

This module only DRAWS inputs: random source rows quantized into cache
records, slot lists, lengths, Q, sink logits, positions and the RoPE table.
It holds none of the decode arithmetic (no dequantization, selection or
attention), so both the CUDA library's tests and the fp64 oracle can be fed
from it without sharing the method's code.

Record encodings (the decode side reads these; definitions as stated for the
workloads of this method):
  * fp8-528:  512 e4m3 codes, then 4 little-endian fp32 scales, one per 128
    dims; scale = block absmax / 448, code = e4m3 round-to-nearest-even of
    x / scale (saturated at +-448).
  * NVFP4-288: 256 bytes of e2m1 nibbles (element 2i in the low nibble of byte
    i, 2i+1 in the high nibble), then 32 e4m3 scales, one per 16 dims;
    scale = e4m3(block absmax / 6), code = e2m1 round-to-nearest-even of
    x / scale, saturated at +-6.
  * fp8-528 with ue8m0 scales (the V4.1 record of the swapab page): 512 e4m3
    codes, then 16 ue8m0 bytes, one per 32 dims; scale = 2^ceil(log2(group
    absmax / 448)) (the page's rule for its MXFP8 output, taken for the cache
    too), byte = exponent + 127, code = e4m3 round-to-nearest-even of
    x / scale.
  * MODEL1-584 (FlashMLA's sparse_decode.h page gives the byte counts
    448 + 64*2 + 448/64 + 1 for d_qk = d_v = 512; read in that order): the
    e4m3 codes of dims 0..447 with one ue8m0 scale per 64 dims (same rule as
    above, per 64 dims), dims 448..511 (the RoPE part) as little-endian bf16
    (round to nearest even), the 7 scale bytes, one zero pad byte.
  * V3.2-656 (same page: 512 + 64*2 + (512/128)*4 bytes for d_qk = 576,
    d_v = 512): the fp8-528 record of the first 512 source dims, then the
    64 further key dims as little-endian bf16 (round to nearest even); the
    source rows have 576 dims, Q too, and no RoPE is applied to Q.

The five named workloads follow the configurations the method is measured on
(T tokens, H query heads, one shared 512-dim KV row per slot). Seeds: workload
k uses seed k-1 unless told otherwise. Draw order: caches (sliding window,
then extra), Q, lengths, slot ids, invalid-entry mask, sink, positions.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

HEAD_DIM = 512
FMT_FP8_528 = 0
FMT_NVFP4_288 = 1
FMT_FP8_528_UE8M0 = 2
FMT_MODEL1_584 = 3
FMT_V32_656 = 4
RECORD_BYTES = {FMT_FP8_528: 528, FMT_NVFP4_288: 288, FMT_FP8_528_UE8M0: 528,
                FMT_MODEL1_584: 584, FMT_V32_656: 656}
FMT_NAMES = {FMT_FP8_528: "fp8_528", FMT_NVFP4_288: "nvfp4_288",
             FMT_FP8_528_UE8M0: "fp8_528_ue8m0", FMT_MODEL1_584: "model1_584",
             FMT_V32_656: "v32_656"}
KEY_DIMS_V32 = 576   # key / query dims with V3.2 records (values keep 512)
ROPE_NEOX = 0   # dim 448+i pairs with 480+i
ROPE_GPTJ = 1   # dim 448+2i pairs with 449+2i
ROPE_TABLE_ROWS = 131072
ROPE_THETA = 10000.0


@dataclasses.dataclass
class PagedCache:
    """A paged cache: ``data`` is uint8 [num_pages, page_stride]; the record of
    slot s sits at page s // page_size, byte offset (s % page_size) * record."""
    data: torch.Tensor
    page_size: int
    fmt: int

    @property
    def num_pages(self) -> int:
        return int(self.data.shape[0])

    @property
    def page_stride(self) -> int:
        return int(self.data.stride(0))

    @property
    def record_bytes(self) -> int:
        return RECORD_BYTES[self.fmt]

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size

    def to(self, device) -> "PagedCache":
        return PagedCache(self.data.to(device), self.page_size, self.fmt)


@dataclasses.dataclass
class SlotList:
    """Slot ids [T, width] int32 (-1 = unused) and lengths [T] int32."""
    ids: torch.Tensor
    lens: torch.Tensor
    width: int

    def to(self, device) -> "SlotList":
        return SlotList(self.ids.to(device), self.lens.to(device), self.width)


@dataclasses.dataclass
class Workload:
    name: str
    T: int
    H: int
    scale: float
    q: torch.Tensor                      # bf16 [T, H, 512]
    swa_cache: PagedCache
    swa: SlotList
    extra_cache: Optional[PagedCache] = None
    extra: Optional[SlotList] = None
    sink: Optional[torch.Tensor] = None  # fp32 [H]
    positions: Optional[torch.Tensor] = None  # int64 [T]
    cos_sin: Optional[torch.Tensor] = None    # fp32 [ROPE_TABLE_ROWS, 64]
    rope_style: int = ROPE_NEOX

    def to(self, device) -> "Workload":
        f = lambda x: None if x is None else x.to(device)
        return Workload(self.name, self.T, self.H, self.scale, f(self.q),
                        self.swa_cache.to(device), self.swa.to(device),
                        None if self.extra_cache is None else self.extra_cache.to(device),
                        None if self.extra is None else self.extra.to(device),
                        f(self.sink), f(self.positions), f(self.cos_sin), self.rope_style)


# --------------------------------------------------------------------------
# encoders
# --------------------------------------------------------------------------

def encode_fp8_records(x: torch.Tensor) -> torch.Tensor:
    """[n, 512] float -> [n, 528] uint8 fp8-528 records."""
    n = x.shape[0]
    xb = x.float().reshape(n, 4, 128)
    scale = (xb.abs().amax(dim=-1) / 448.0).float()            # [n, 4]
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    y = (xb / safe[..., None]).clamp(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, 512)
    sbytes = scale.contiguous().view(torch.uint8).reshape(n, 16)  # little endian
    return torch.cat([codes, sbytes], dim=1)


def encode_fp8_ue8m0_records(x: torch.Tensor) -> torch.Tensor:
    """[n, 512] float -> [n, 528] uint8 fp8-528 records with ue8m0 scales."""
    n = x.shape[0]
    xb = x.float().reshape(n, 16, 32)
    amax = xb.abs().amax(dim=-1).double()                       # [n, 16]
    ex = torch.where(amax > 0, torch.ceil(torch.log2(amax / 448.0)), torch.zeros_like(amax))
    ex = ex.clamp(-127, 127)
    y = (xb.double() / torch.exp2(ex)[..., None]).clamp(-448.0, 448.0).float()
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, 512)
    sbytes = (ex + 127).to(torch.uint8)
    return torch.cat([codes, sbytes], dim=1)


def encode_model1_records(x: torch.Tensor) -> torch.Tensor:
    """[n, 512] float -> [n, 584] uint8 MODEL1 records."""
    n = x.shape[0]
    xb = x[:, :448].float().reshape(n, 7, 64)
    amax = xb.abs().amax(dim=-1).double()                       # [n, 7]
    ex = torch.where(amax > 0, torch.ceil(torch.log2(amax / 448.0)), torch.zeros_like(amax))
    ex = ex.clamp(-127, 127)
    y = (xb.double() / torch.exp2(ex)[..., None]).clamp(-448.0, 448.0).float()
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, 448)
    rope = x[:, 448:].float().to(torch.bfloat16).contiguous().view(torch.uint8).reshape(n, 128)
    sbytes = (ex + 127).to(torch.uint8)
    pad = torch.zeros((n, 1), dtype=torch.uint8, device=x.device)
    return torch.cat([codes, rope, sbytes, pad], dim=1)


def encode_v32_records(x: torch.Tensor) -> torch.Tensor:
    """[n, 576] float -> [n, 656] uint8 V3.2 records."""
    n = x.shape[0]
    tail = x[:, HEAD_DIM:].float().to(torch.bfloat16).contiguous().view(torch.uint8).reshape(n, 128)
    return torch.cat([encode_fp8_records(x[:, :HEAD_DIM]), tail], dim=1)


def _e2m1_codes(y: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even onto e2m1 magnitudes {0,.5,1,1.5,2,3,4,6}, saturating
    at 6; returns 4-bit codes (sign in bit 3) as uint8."""
    a = y.abs()
    idx = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
           + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
           + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    sign = (y < 0).to(torch.uint8) << 3
    return idx | torch.where(idx > 0, sign, torch.zeros_like(sign))


def encode_nvfp4_records(x: torch.Tensor) -> torch.Tensor:
    """[n, 512] float -> [n, 288] uint8 NVFP4-288 records."""
    n = x.shape[0]
    xb = x.float().reshape(n, 32, 16)
    sc8 = (xb.abs().amax(dim=-1) / 6.0).clamp(max=448.0).to(torch.float8_e4m3fn)   # [n, 32]
    scf = sc8.float()
    safe = torch.where(scf > 0, scf, torch.ones_like(scf))
    codes = _e2m1_codes(xb / safe[..., None])
    codes = torch.where((scf > 0)[..., None], codes, torch.zeros_like(codes))
    codes = codes.reshape(n, 256, 2)
    packed = codes[..., 0] | (codes[..., 1] << 4)
    return torch.cat([packed, sc8.view(torch.uint8)], dim=1)


def make_cache(num_slots: int, page_size: int, fmt: int, gen: torch.Generator,
               device, page_pad: int = 0, chunk: int = 1 << 18, mag=(0,)) -> PagedCache:
    """N(0,1) source rows, quantized to records, laid out in pages.
    ``page_pad`` extra bytes (multiple of 16) separate consecutive pages.
    ``mag``: powers of two; the source row of slot s is scaled by
    2^mag[s % len(mag)] before it is quantized (default: unit rows)."""
    assert num_slots % page_size == 0 and page_pad % 16 == 0
    rb = RECORD_BYTES[fmt]
    num_pages = num_slots // page_size
    stride = page_size * rb + page_pad
    data = torch.zeros((num_pages, stride), dtype=torch.uint8, device=device)
    recs = data[:, :page_size * rb].view(num_pages, page_size, rb)
    enc = {FMT_FP8_528: encode_fp8_records, FMT_NVFP4_288: encode_nvfp4_records,
           FMT_FP8_528_UE8M0: encode_fp8_ue8m0_records,
           FMT_MODEL1_584: encode_model1_records, FMT_V32_656: encode_v32_records}[fmt]
    dk = KEY_DIMS_V32 if fmt == FMT_V32_656 else HEAD_DIM
    chunk = max(page_size, chunk - chunk % page_size)
    for s0 in range(0, num_slots, chunk):
        s1 = min(num_slots, s0 + chunk)          # both multiples of page_size
        x = torch.randn((s1 - s0, dk), generator=gen, device=device)
        if tuple(mag) != (0,):
            m = torch.tensor([float(k) for k in mag], dtype=torch.float32, device=device)
            sl = torch.arange(s0, s1, device=device) % len(mag)
            x = x * torch.exp2(m[sl])[:, None]
        recs[s0 // page_size: s1 // page_size] = enc(x).view(-1, page_size, rb)
    return PagedCache(data, page_size, fmt)


def sample_distinct(T: int, k: int, n: int, gen: torch.Generator, device) -> torch.Tensor:
    """[T, k] int32: per row, k distinct ids drawn uniformly from [0, n), in
    random order (sampling without replacement)."""
    assert 0 <= k <= n
    if k == 0:
        return torch.zeros((T, 0), dtype=torch.int32, device=device)
    if 4 * k > n:
        keys = torch.rand((T, n), generator=gen, device=device)
        return keys.argsort(dim=1)[:, :k].to(torch.int32)
    ids = torch.randint(0, n, (T, k), generator=gen, device=device, dtype=torch.int64)
    for _ in range(200):
        s, order = ids.sort(dim=1)
        dup_sorted = torch.zeros_like(ids, dtype=torch.bool)
        dup_sorted[:, 1:] = s[:, 1:] == s[:, :-1]
        if not bool(dup_sorted.any()):
            return ids.to(torch.int32)
        dup = torch.zeros_like(dup_sorted).scatter_(1, order, dup_sorted)
        cnt = int(dup.sum())
        ids[dup] = torch.randint(0, n, (cnt,), generator=gen, device=device,
                                 dtype=torch.int64)
    raise RuntimeError("could not draw distinct slot ids")


def rope_table(rows: int = ROPE_TABLE_ROWS, device="cpu") -> torch.Tensor:
    """fp32 [rows, 64]: row p = [cos(p w_i) for i<32 | sin(p w_i) for i<32],
    w_i = theta^(-2i/64), computed in fp64 and rounded once to fp32."""
    i = torch.arange(32, dtype=torch.float64)
    w = ROPE_THETA ** (-2.0 * i / 64.0)
    p = torch.arange(rows, dtype=torch.float64)[:, None]
    ang = p * w[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).float().to(device)


def _lens(T, width, lens, gen, device):
    if lens == "full":
        return torch.full((T,), width, dtype=torch.int32, device=device)
    lo, hi = lens
    return torch.randint(lo, hi + 1, (T,), generator=gen, device=device,
                         dtype=torch.int64).to(torch.int32)


def make_workload(*, T: int, H: int, swa: dict, extra: Optional[dict] = None,
                  sink: bool = False, rope: bool = False, seed: int = 0,
                  device="cpu", name: str = "custom", page_pad: int = 0,
                  scale: Optional[float] = None, rope_style: int = ROPE_NEOX,
                  q_log2: int = 0) -> Workload:
    """Build a workload.

    swa / extra: dict(width, lens=(lo, hi) inclusive or "full", fmt, page,
    slots, invalid=fraction of in-range entries replaced by -1 (default 0),
    mag=powers of two scaling the source rows per slot, see make_cache).
    q_log2: Q is drawn N(0,1) and scaled by 2^q_log2 (exact in bf16).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    specs = [swa] + ([extra] if extra is not None else [])
    caches = [make_cache(s["slots"], s["page"], s["fmt"], gen, device, page_pad,
                         mag=s.get("mag", (0,))) for s in specs]
    v32 = [s["fmt"] == FMT_V32_656 for s in specs]
    assert not any(v32) or (all(v32) and not rope), "V3.2 records: every list, no RoPE"
    dk = KEY_DIMS_V32 if any(v32) else HEAD_DIM
    q = torch.randn((T, H, dk), generator=gen, device=device)
    if q_log2:
        q = q * 2.0 ** q_log2
    q = q.to(torch.bfloat16)
    lens = [_lens(T, s["width"], s.get("lens", "full"), gen, device) for s in specs]
    ids = [sample_distinct(T, s["width"], s["slots"], gen, device) for s in specs]
    lists = []
    for s, l, i in zip(specs, lens, ids):
        r = torch.arange(s["width"], device=device)[None, :]
        inr = r < l.to(torch.int64)[:, None]
        frac = float(s.get("invalid", 0.0))
        if frac > 0:
            drop = torch.rand(i.shape, generator=gen, device=device) < frac
            i = torch.where(drop & inr, torch.full_like(i, -1), i)
        i = torch.where(inr, i, torch.full_like(i, -1))
        lists.append(SlotList(i.contiguous(), l, s["width"]))
    sk = torch.randn((H,), generator=gen, device=device) if sink else None
    pos = cs = None
    if rope:
        pos = torch.randint(0, ROPE_TABLE_ROWS, (T,), generator=gen, device=device,
                            dtype=torch.int64)
        cs = rope_table(ROPE_TABLE_ROWS, device)
    return Workload(name, T, H, scale if scale is not None else dk ** -0.5, q,
                    caches[0], lists[0],
                    caches[1] if extra is not None else None,
                    lists[1] if extra is not None else None, sk, pos, cs, rope_style)


# The five measured configurations (sizes as stated; the open choices -- full
# sliding-window lengths, page 64 and 2^16 slots for the sliding-window caches
# of workloads 3-5 -- are the plainest readings).
def _spec(width, lens, fmt, page, slots, invalid=0.0):
    return dict(width=width, lens=lens, fmt=fmt, page=page, slots=slots, invalid=invalid)


CONFIGS = {
    1: dict(T=4, H=16, swa=_spec(128, (1, 128), FMT_FP8_528, 64, 4096), extra=None,
            sink=False, rope=False),
    2: dict(T=64, H=32, swa=_spec(128, (1, 128), FMT_FP8_528, 64, 1 << 16),
            extra=_spec(512, (0, 512), FMT_FP8_528, 64, 1 << 18, invalid=0.05),
            sink=True, rope=False),
    3: dict(T=128, H=64, swa=_spec(128, "full", FMT_FP8_528, 128, 1 << 16),
            extra=_spec(2048, (256, 2048), FMT_NVFP4_288, 256, 1 << 20),
            sink=True, rope=False),
    4: dict(T=256, H=128, swa=_spec(128, "full", FMT_FP8_528, 64, 1 << 16),
            extra=_spec(2048, (1024, 2048), FMT_FP8_528, 64, 1 << 21),
            sink=True, rope=True),
    5: dict(T=1024, H=64, swa=_spec(128, "full", FMT_FP8_528, 64, 1 << 16),
            extra=_spec(4096, "full", FMT_NVFP4_288, 256, 1 << 22),
            sink=True, rope=True),
}
CONFIG5_BATCHES = (1, 8, 64, 256, 1024)


def make_config(k: int, *, T: Optional[int] = None, device="cpu",
                seed: Optional[int] = None, page_pad: int = 0, v41: bool = False,
                model1: bool = False, v32: bool = False) -> Workload:
    """Measured configuration k. ``v41``: the same shapes and draws in the
    V4.1 form -- every fp8-528 list holds ue8m0-scaled records, RoPE pairs
    dims GPT-J style. ``model1``: every fp8-528 list holds MODEL1 records
    instead (same draws, same RoPE). ``v32``: every list holds V3.2 records
    (576-dim keys and Q, no RoPE; same widths, lengths and caches' slot
    counts and pages)."""
    c = dict(CONFIGS[k])
    if T is not None:
        c["T"] = T
    name = f"config{k}_T{c['T']}_H{c['H']}"
    if v32:
        for key in ("swa", "extra"):
            if c[key] is not None:
                c[key] = dict(c[key], fmt=FMT_V32_656)
        c["rope"] = False
        name += "_v32"
    if model1:
        for key in ("swa", "extra"):
            if c[key] is not None and c[key]["fmt"] == FMT_FP8_528:
                c[key] = dict(c[key], fmt=FMT_MODEL1_584)
        name += "_model1"
    if v41:
        for key in ("swa", "extra"):
            if c[key] is not None and c[key]["fmt"] == FMT_FP8_528:
                c[key] = dict(c[key], fmt=FMT_FP8_528_UE8M0)
        c["rope_style"] = ROPE_GPTJ
        name += "_v41"
    return make_workload(seed=(k - 1) if seed is None else seed, device=device,
                         name=name, page_pad=page_pad, **c)


def workload_summary(w: Workload) -> dict:
    """Shape description (no selection arithmetic)."""
    def cache(c):
        return None if c is None else dict(
            fmt=FMT_NAMES[c.fmt], page=c.page_size, slots=c.num_slots,
            bytes=int(c.data.numel()))
    return dict(workload=w.name, T=w.T, H=w.H, swa_width=w.swa.width,
                extra_width=0 if w.extra is None else w.extra.width,
                swa_cache=cache(w.swa_cache), extra_cache=cache(w.extra_cache),
                sink=w.sink is not None, rope=w.cos_sin is not None,
                rope_style=["neox", "gptj"][w.rope_style])


def oracle_args(w: Workload) -> dict:
    """Arguments for ``oracle.decode`` (CPU copies; plain data, no arithmetic)."""
    w = w.to("cpu")
    caches = [dict(bytes=w.swa_cache.data.reshape(-1), num_pages=w.swa_cache.num_pages,
                   page_size=w.swa_cache.page_size, page_stride=w.swa_cache.page_stride,
                   format=w.swa_cache.fmt)]
    lists = [dict(ids=w.swa.ids, lens=w.swa.lens, width=w.swa.width)]
    if w.extra is not None:
        caches.append(dict(bytes=w.extra_cache.data.reshape(-1),
                           num_pages=w.extra_cache.num_pages,
                           page_size=w.extra_cache.page_size,
                           page_stride=w.extra_cache.page_stride,
                           format=w.extra_cache.fmt))
        lists.append(dict(ids=w.extra.ids, lens=w.extra.lens, width=w.extra.width))
    return dict(q=w.q, caches=caches, lists=lists, scale=w.scale, sink=w.sink,
                positions=w.positions, cos_sin=w.cos_sin, rope_style=w.rope_style)
