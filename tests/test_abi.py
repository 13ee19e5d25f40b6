"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, plans correctly, and rejects bad arguments before any launch.

Every rejected call below is invalid in at least one checked way, so none of
them reaches a CUDA call (the validation happens first)."""
import ctypes
import os
import re

import pytest

from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import build as BLD

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "dsa_decode.h")


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_decode_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(B.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_every_declared_call_cites_its_definition():
    """Each entry point's comment block (the comment right before its
    declaration) names the passage of the pages that defines the operation
    ("Defined by: ...", with a page and an identifier on it), or says that
    the pages have no counterpart."""
    src = open(HEADER).read()
    pages = ("swapab page", "sparse_decode.h page", "production.py page")
    for name in declared_functions():
        m = re.search(r"(/\*(?:(?!\*/).)*\*/)\s*[\w\s\*]*?\b" + name + r"\s*\(", src, flags=re.S)
        assert m, f"{name}: no comment before its declaration"
        doc = " ".join(m.group(1).split())
        if "counterpart" in doc:
            continue
        assert "Defined by:" in doc, f"{name}: no citation"
        cited = doc.split("Defined by:", 1)[1]
        assert any(p in cited for p in pages), f"{name}: citation names no page"


def test_abi_version_matches_header(lib):
    m = re.search(r"#define DSA_DECODE_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.dsa_decode_abi_version() == int(m.group(1))


def test_status_strings(lib):
    for code in B.STATUS_NAMES:
        assert lib.dsa_decode_status_string(code)
    assert lib.dsa_decode_status_string(12345) == b"unknown status"


def test_plan_struct_size_matches_header():
    # 16 int32 + 8 int64 + 14 reserved int64
    assert ctypes.sizeof(B.Plan) == 16 * 4 + 8 * 8 + 14 * 8


@pytest.mark.parametrize("T,H,ws,we,sms", [
    (4, 16, 128, 0, 152), (64, 32, 128, 512, 152), (128, 64, 128, 2048, 152),
    (256, 128, 128, 2048, 152), (1, 64, 128, 4096, 152), (1024, 64, 128, 4096, 152),
    (3, 48, 100, 300, 7), (5, 96, 1, 1, 1), (2, 16, 129, 0, 1000)])
def test_plan_schedule_covers_every_unit_once(lib, T, H, ws, we, sms):
    plan, nbytes = B.dsa_decode_plan(T, H, ws, we, sms)
    assert plan.num_tokens == T and plan.num_heads == H
    assert plan.head_groups * plan.heads_per_group == H
    assert plan.heads_per_group % 16 == 0 and plan.heads_per_group <= 64
    tpt = -(-ws // 128) + -(-we // 128)
    assert plan.tiles_per_token == tpt and plan.total_units == T * tpt
    C, upc = plan.ctas_per_group, plan.units_per_cta
    assert C * plan.head_groups <= max(sms, plan.head_groups) or C == plan.total_units
    assert (C - 1) * upc < plan.total_units <= C * upc          # no empty CTA
    owner = [u // upc for u in range(plan.total_units)]
    assert owner == sorted(owner) and len(set(owner)) == C
    # per CTA at most two partial tokens -> slots 2c, 2c+1
    for c in range(C):
        u0, u1 = c * upc, min(plan.total_units, (c + 1) * upc)
        toks = range(u0 // tpt, (u1 - 1) // tpt + 1)
        partial = [t for t in toks if not (u0 <= t * tpt and (t + 1) * tpt <= u1)]
        assert len(partial) <= 2 and all(t in (toks[0], toks[-1]) for t in partial)
    # workspace regions are ordered, aligned and inside the total
    offs = [plan.ws_sel_offset, plan.ws_part_lse_offset, plan.ws_part_sel_offset,
            plan.ws_part_o_offset, plan.workspace_bytes]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs) and nbytes == offs[-1]
    assert plan.ws_part_sel_offset - plan.ws_part_lse_offset >= 4 * 2 * C * H
    assert nbytes - plan.ws_part_o_offset >= 4 * 2 * C * H * 512


def test_plan_rejects_bad_shapes(lib):
    for args, code in [((4, 20, 128, 0, 1), -2), ((4, 256, 128, 0, 1), -2),
                       ((4, 0, 128, 0, 1), -2), ((-1, 16, 128, 0, 1), -1),
                       ((4, 16, 0, 0, 1), -1), ((4, 16, 128, -1, 1), -1),
                       ((4, 16, 128, 0, -3), -1)]:
        with pytest.raises(B.DsaError) as e:
            B.dsa_decode_plan(*args)
        assert e.value.status == code, args
    plan = B.Plan()
    n = ctypes.c_size_t()
    assert lib.dsa_decode_plan(4, 16, 128, 0, 1, None, ctypes.byref(n)) == -1
    assert lib.dsa_decode_plan(4, 16, 128, 0, 1, ctypes.byref(plan), None) == -1


def test_zero_tokens_is_a_no_op(lib):
    plan, nbytes = B.dsa_decode_plan(0, 16, 128, 0, 4)
    assert nbytes == 0
    # run/combine return OK without touching any pointer
    assert lib.dsa_decode_run(ctypes.byref(plan), None, 0, None, 0, 0, None, None, 0, None,
                              None, None, 0, None, None, None, None, 0, 1.0, None, None,
                              None) == 0
    assert lib.dsa_decode_combine(ctypes.byref(plan), None, 0, None, None, None, None) == 0


# ---------------------------------------------------------------- validation
FAKE = 1 << 40          # 256-aligned fake device addresses: never dereferenced


class Args:
    """A fully described call whose pointers are fake; each test breaks one
    field, so validation fails before anything is launched."""

    def __init__(self, H=16, T=4, ws=128, we=0):
        self.plan, self.nbytes = B.dsa_decode_plan(T, H, ws, we, 4)
        self.T, self.H = T, H
        self.swa = B.CacheDesc(FAKE, 64, 64 * 528, 64, 0)
        self.extra = B.CacheDesc(FAKE, 64, 64 * 288, 64, 1) if we else None
        self.kw = dict(ws=FAKE, ws_bytes=self.nbytes, q=FAKE, q_st=H * 512, q_sh=512,
                       swa_idx=FAKE, swa_stride=ws + (-ws) % 4, swa_lens=FAKE,
                       extra_idx=FAKE if we else None, extra_stride=we + (-we) % 4 if we else 0,
                       extra_lens=FAKE if we else None, sink=None, pos=None, cs=None, cs_rows=0,
                       scale=0.044, out=FAKE, lse=FAKE)

    def call(self, lib, **over):
        k = dict(self.kw)
        k.update(over)
        plan = over.get("plan", self.plan)
        swa = over.get("swa_desc", self.swa)
        extra = over.get("extra_desc", self.extra)
        return lib.dsa_decode_run(
            ctypes.byref(plan) if plan is not None else None, k["ws"], k["ws_bytes"], k["q"],
            k["q_st"], k["q_sh"], ctypes.byref(swa) if swa is not None else None,
            k["swa_idx"], k["swa_stride"], k["swa_lens"],
            ctypes.byref(extra) if extra is not None else None, k["extra_idx"],
            k["extra_stride"], k["extra_lens"], k["sink"], k["pos"], k["cs"], k["cs_rows"],
            k["scale"], k["out"], k["lse"], None)


def test_run_rejects_bad_plan(lib):
    a = Args()
    bad = B.Plan()
    ctypes.memmove(ctypes.byref(bad), ctypes.byref(a.plan), ctypes.sizeof(bad))
    bad.magic = 0
    assert a.call(lib, plan=bad) == -7
    assert a.call(lib, plan=None) == -7
    assert lib.dsa_decode_combine(ctypes.byref(bad), FAKE, a.nbytes, None, FAKE, FAKE, None) == -7


@pytest.mark.parametrize("field,value,code", [
    ("q", None, -1), ("out", None, -1), ("lse", None, -1), ("scale", float("nan"), -1),
    ("scale", float("inf"), -1), ("q_sh", 256, -1), ("q_st", 512, -1),
    ("q", FAKE + 8, -3), ("q_st", 16 * 512 + 4, -3), ("out", FAKE + 4, -3), ("lse", FAKE + 2, -3),
    ("ws", None, -4), ("ws_bytes", 16, -4), ("ws", FAKE + 128, -4),
    ("swa_idx", None, -1), ("swa_lens", None, -1), ("swa_stride", 64, -1),
    ("swa_idx", FAKE + 2, -3), ("swa_lens", FAKE + 2, -3),
    ("pos", FAKE, -1), ("cs", FAKE, -1), ("sink", FAKE + 1, -3),
    ("extra_idx", FAKE, -1), ("extra_lens", FAKE, -1),
])
def test_run_rejects_bad_argument(lib, field, value, code):
    a = Args()
    assert a.call(lib, **{field: value}) == code


def test_run_rejects_bad_cache_descriptors(lib):
    a = Args()
    base = dict(base=FAKE, num_pages=64, page_stride_bytes=64 * 528, page_size=64, format=0)
    cases = [(dict(page_size=48), -1), (dict(page_size=0), -1), (dict(num_pages=0), -1),
             (dict(page_stride_bytes=64 * 528 - 16), -1), (dict(format=7), -2),
             (dict(base=None), -1), (dict(base=FAKE + 8), -3),
             (dict(page_stride_bytes=64 * 528 + 8), -3)]
    for over, code in cases:
        d = dict(base)
        d.update(over)
        desc = B.CacheDesc(d["base"], d["num_pages"], d["page_stride_bytes"], d["page_size"],
                           d["format"])
        assert a.call(lib, swa_desc=desc) == code, over
    assert a.call(lib, swa_desc=None) == -1


def test_run_extra_list_presence_must_match_plan(lib):
    a = Args(we=256)
    assert a.call(lib, extra_desc=None) == -1
    assert a.call(lib, extra_idx=None) == -1
    assert a.call(lib, extra_lens=None) == -1
    b = Args(we=0)
    assert b.call(lib, extra_desc=B.CacheDesc(FAKE, 64, 64 * 288, 64, 1), extra_idx=FAKE,
                  extra_lens=FAKE, extra_stride=256) == -1


def test_rope_needs_both_pointers_and_rows(lib):
    a = Args()
    assert a.call(lib, pos=FAKE) == -1
    assert a.call(lib, cs=FAKE) == -1
    assert a.call(lib, pos=FAKE, cs=FAKE, cs_rows=0) == -1
    assert a.call(lib, pos=FAKE, cs=FAKE + 4, cs_rows=10) == -3


def test_combine_and_selection_validation(lib):
    a = Args(T=3, we=512)                      # 15 units over 4 CTAs: tokens are split
    assert a.plan.ctas_per_group > 1 and a.plan.split_tokens > 0
    assert lib.dsa_decode_combine(ctypes.byref(a.plan), None, 0, None, FAKE, FAKE, None) == -4
    assert lib.dsa_decode_combine(ctypes.byref(a.plan), FAKE, a.nbytes, None, None, FAKE, None) == -1
    assert lib.dsa_decode_combine(ctypes.byref(a.plan), FAKE, a.nbytes, None, FAKE + 2, FAKE,
                                  None) == -3
    assert lib.dsa_decode_selection(ctypes.byref(a.plan), None, FAKE, FAKE, None) == -1
    assert lib.dsa_decode_read_status(None, None, None) == -1


@pytest.mark.parametrize("T,sms", [(1, 152), (64, 152), (128, 152), (256, 152), (1024, 152), (4, 1)])
def test_plan_live_balancing_flag_and_bounds_slot(lib, T, sms):
    """Work balancing is planned for >= 16 tokens of >= 8 tiles each; the
    CTA-range array (C + 1 int64) sits inside the workspace, after the
    partials, 256-byte aligned."""
    plan, nbytes = B.dsa_decode_plan(T, 64, 128, 2048, sms)
    C = plan.ctas_per_group
    assert plan.balance_live == (1 if T >= 16 and plan.tiles_per_token >= 8 else 0)
    narrow, _ = B.dsa_decode_plan(T, 64, 128, 512, sms)   # 5 tiles per token
    assert narrow.balance_live == 0
    assert plan.ws_bounds_offset % 256 == 0
    assert plan.ws_bounds_offset >= plan.ws_part_o_offset
    assert plan.ws_bounds_offset + 8 * (C + 1) <= nbytes


def test_split_tokens_zero_only_when_every_token_is_whole(lib):
    """An even split whose CTAs hold whole tokens splits nothing, so the plan
    says split_tokens = 0 and combine launches nothing; otherwise it is the
    upper bound C - 1."""
    p, _ = B.dsa_decode_plan(4, 16, 128, 0, num_sms=152)      # 1 tile per token, 4 CTAs
    assert p.ctas_per_group == 4 and p.units_per_cta % p.tiles_per_token == 0
    assert p.balance_live == 0 and p.split_tokens == 0
    p, _ = B.dsa_decode_plan(1, 64, 128, 4096, num_sms=152)   # one token over 33 CTAs
    assert p.split_tokens == p.ctas_per_group - 1 > 0
    p, _ = B.dsa_decode_plan(1024, 64, 128, 4096, num_sms=152)   # balanced ranges
    assert p.balance_live == 1 and p.split_tokens == p.ctas_per_group - 1
    p, _ = B.dsa_decode_plan(400, 16, 128, 0, num_sms=152)     # 3 whole tokens per CTA
    assert p.units_per_cta == 3 and p.split_tokens == 0


@pytest.mark.parametrize("T,H,ws,we,expect", [
    (1024, 64, 128, 4096, 0),    # config 5: 33 tiles per token, ~29 per segment
    (256, 64, 128, 4096, 0),     # ~21 per segment
    (64, 64, 128, 4096, 1),      # ~10 per segment (tokens split over CTAs)
    (128, 64, 128, 2048, 1),     # config 3 widths
    (256, 128, 128, 2048, 1),    # config 4: two 64-head groups
    (4096, 32, 128, 512, 0),     # 32 heads per group: the softmax warps stage Q
])
def test_plan_producer_q(lib, T, H, ws, we, expect):
    """The form whose producers stage Q is planned for 64 heads per group and
    fewer than 16 tiles per token segment (T tokens over C CTAs of a group:
    T + C segments)."""
    plan, _ = B.dsa_decode_plan(T, H, ws, we, 152)
    C, tpt = plan.ctas_per_group, plan.tiles_per_token
    rule = plan.heads_per_group == 64 and T * tpt < 16 * (T + C)
    assert plan.producer_q == int(rule) == expect
    p576, _ = B.dsa_decode_plan_qk(T, min(H, 64), ws, we, 152, 576)
    assert p576.producer_q == 0                      # V3.2 records: groups of at most 32


@pytest.mark.parametrize("T,H,ws,we,sms", [(1024, 64, 128, 4096, 152), (1, 64, 128, 4096, 152),
                                           (2, 64, 128, 9000, 1000), (4, 16, 128, 0, 152)])
def test_plan_merge_in_run_and_count_block(lib, T, H, ws, we, sms):
    """Split tokens are merged by the run kernel when tokens have few parts
    (C <= 4 T) and a token spans at most 64 CTAs; the per-token unit counts it uses ([head_groups][T] int32) sit
    between the status word and the selection records, inside the block each
    run zeroes."""
    plan, nbytes = B.dsa_decode_plan(T, H, ws, we, sms)
    span = min(plan.ctas_per_group, plan.tiles_per_token)
    expect = int(plan.split_tokens > 0 and span <= 64 and plan.ctas_per_group <= 4 * T)
    assert plan.merge_in_run == expect
    assert plan.ws_count_offset >= 4
    assert plan.ws_count_offset + 4 * plan.head_groups * T <= plan.ws_sel_offset
    assert plan.ws_sel_offset % 256 == 0 and plan.ws_sel_offset <= nbytes
