"""C-ABI checks of the V4.1 entry points (dsa_decode_run_v41 /
dsa_decode_combine_v41) that need no GPU: every call below breaks at least
one checked rule, so validation refuses it before any CUDA call."""
import ctypes

import pytest

from swa_paged_decode_gb300 import binding as B
from tests.test_abi import FAKE, Args, lib  # noqa: F401  (lib is a fixture)


def mx_desc(**over):
    d = dict(data=FAKE, scale=FAKE, data_stride_t=16 * 512, data_stride_g=4 * 512,
             scale_stride_t=64, scale_stride_g=16, scale_stride_w=1, group_size=4, reserved=0)
    d.update(over)
    return B.MxOutDesc(d["data"], d["scale"], d["data_stride_t"], d["data_stride_g"],
                       d["scale_stride_t"], d["scale_stride_g"], d["scale_stride_w"],
                       d["group_size"], d["reserved"])


def run_v41(lib, a, rope_style=B.DSA_ROPE_GPTJ, out=None, mx=None, **over):
    k = dict(a.kw)
    if mx is not None:   # an MXFP8 call needs the plan's larger workspace
        k["ws_bytes"] = a.plan.workspace_bytes_mx
    k.update(over)
    swa = over.get("swa_desc", a.swa)
    extra = over.get("extra_desc", a.extra)
    return lib.dsa_decode_run_v41(
        ctypes.byref(a.plan), k["ws"], k["ws_bytes"], k["q"], k["q_st"], k["q_sh"],
        ctypes.byref(swa), k["swa_idx"], k["swa_stride"], k["swa_lens"],
        ctypes.byref(extra) if extra is not None else None, k["extra_idx"], k["extra_stride"],
        k["extra_lens"], k["sink"], k["pos"], k["cs"], k["cs_rows"], rope_style, k["scale"],
        out, ctypes.byref(mx) if mx is not None else None, k["lse"], None)


FMT7 = B.CacheDesc(FAKE, 64, 64 * 528, 64, 7)   # unsupported format: -2, checked after the output


def test_exactly_one_output(lib):
    a = Args()
    assert run_v41(lib, a, out=None, mx=None, swa_desc=FMT7) == -1
    assert run_v41(lib, a, out=FAKE, mx=mx_desc(), swa_desc=FMT7) == -1
    assert run_v41(lib, a, out=FAKE, swa_desc=FMT7) == -2


def test_rope_style_must_be_known(lib):
    # the swa descriptor is misaligned too (-3, checked later): -1 shows that
    # the style was refused first
    a = Args()
    bad = B.CacheDesc(FAKE + 8, 64, 64 * 528, 64, 0)
    assert run_v41(lib, a, rope_style=2, out=FAKE, swa_desc=bad) == -1
    assert run_v41(lib, a, rope_style=-1, mx=mx_desc(), swa_desc=bad) == -1
    assert run_v41(lib, a, rope_style=1, out=FAKE, swa_desc=bad) == -3


@pytest.mark.parametrize("over,code", [
    (dict(group_size=0), -1), (dict(group_size=3), -1), (dict(group_size=32), -1),
    (dict(data=None), -1), (dict(scale=None), -1),
    (dict(data=FAKE + 2), -3), (dict(scale=FAKE + 2), -3),
    (dict(data_stride_t=16 * 512 + 2), -3), (dict(data_stride_g=4 * 512 + 1), -3),
])
def test_mx_descriptor_rules(lib, over, code):
    a = Args()   # H = 16; a broken cache descriptor (-2) is checked later
    assert run_v41(lib, a, mx=mx_desc(**over), swa_desc=FMT7) == code
    assert run_v41(lib, a, mx=mx_desc(), swa_desc=FMT7) == -2


def test_neox_inverse_rotation_is_not_offered(lib):
    a = Args()
    bad_page = B.CacheDesc(FAKE, 64, 64 * 528, 48, 0)        # -1, checked later
    assert run_v41(lib, a, rope_style=B.DSA_ROPE_NEOX, mx=mx_desc(), pos=FAKE, cs=FAKE,
                   cs_rows=16, swa_desc=bad_page) == -2
    # without RoPE there is nothing to undo: the descriptor passes and the call
    # is refused further on (a broken cache descriptor)
    bad = B.CacheDesc(FAKE, 64, 64 * 528, 48, 0)
    assert run_v41(lib, a, rope_style=B.DSA_ROPE_NEOX, mx=mx_desc(), swa_desc=bad) == -1


def test_ue8m0_record_format_is_accepted(lib):
    # swa list in the ue8m0 format, extra list misaligned: the refusal comes
    # from the extra list, so the ue8m0 descriptor passed.
    a = Args(we=256)
    ue = B.CacheDesc(FAKE, 64, 64 * 528, 64, 2)
    bad_extra = B.CacheDesc(FAKE + 8, 64, 64 * 288, 64, 1)
    assert run_v41(lib, a, out=FAKE, swa_desc=ue, extra_desc=bad_extra) == -3
    assert a.call(lib, swa_desc=ue, extra_desc=bad_extra) == -3
    assert a.call(lib, swa_desc=B.CacheDesc(FAKE, 64, 64 * 656, 64, 5)) == -2   # no format 5


def test_model1_record_format_is_accepted(lib):
    # MODEL1 (584-byte records): accepted in either list (the refusal comes
    # from the misaligned other list); its page stride is checked against 584
    a = Args(we=256)
    m1 = B.CacheDesc(FAKE, 64, 64 * 584, 64, 3)
    bad_extra = B.CacheDesc(FAKE + 8, 64, 64 * 288, 64, 1)
    assert a.call(lib, swa_desc=m1, extra_desc=bad_extra) == -3
    assert run_v41(lib, a, out=FAKE, swa_desc=m1, extra_desc=bad_extra) == -3
    bad_swa = B.CacheDesc(FAKE + 8, 64, 64 * 528, 64, 0)
    assert a.call(lib, swa_desc=bad_swa, extra_desc=B.CacheDesc(FAKE, 64, 64 * 584, 64, 3)) == -3
    assert a.call(lib, swa_desc=B.CacheDesc(FAKE, 64, 64 * 528, 64, 3)) == -1   # stride < 64 * 584


def test_combine_v41_validation(lib):
    a = Args(T=3, we=512)                      # 15 units over 4 CTAs: tokens are split
    assert a.plan.ctas_per_group > 1 and a.plan.split_tokens > 0
    p = ctypes.byref(a.plan)
    f = lib.dsa_decode_combine_v41
    nb, nm = a.nbytes, a.plan.workspace_bytes_mx
    assert f(p, FAKE, nb, None, None, None, 0, 1, None, None, FAKE, None) == -1
    m = mx_desc()
    assert f(p, FAKE, nm, None, None, None, 0, 1, FAKE, ctypes.byref(m), FAKE, None) == -1
    assert f(p, FAKE, nm, None, FAKE, FAKE, 16, 0, None, ctypes.byref(m), FAKE, None) == -2
    assert f(p, FAKE, nm, None, FAKE, None, 16, 1, None, ctypes.byref(m), FAKE, None) == -1
    assert f(p, None, 0, None, None, None, 0, 1, None, ctypes.byref(m), FAKE, None) == -4
    assert f(p, FAKE, nb, None, None, None, 0, 7, FAKE, None, FAKE, None) == -1
    bad = mx_desc(group_size=5)
    assert f(p, FAKE, nm, None, None, None, 0, 1, None, ctypes.byref(bad), FAKE, None) == -1


def test_mxfp8_workspace_size(lib):
    a = Args(T=4, H=16)
    p = a.plan
    assert p.ws_stage_offset >= p.workspace_bytes and p.ws_stage_offset % 256 == 0
    assert p.workspace_bytes_mx == p.ws_stage_offset + 4 * 4 * 16 * 512
    # the bf16 workspace is too small for an MXFP8 call (a later check would give -2)
    assert run_v41(lib, a, mx=mx_desc(), ws_bytes=a.nbytes, swa_desc=FMT7) == -4
    assert run_v41(lib, a, mx=mx_desc(), swa_desc=FMT7) == -2
    c = Args(T=64, we=512)
    f = lib.dsa_decode_combine_v41
    m = mx_desc()
    assert f(ctypes.byref(c.plan), FAKE, c.nbytes, None, None, None, 0, 1, None, ctypes.byref(m),
             FAKE, None) == -4
    # with bf16 output, a plan that splits nothing needs no combine; MXFP8 does
    d = Args(T=1, we=0)
    assert d.plan.ctas_per_group == 1
    g = lib.dsa_decode_combine_v41
    assert g(ctypes.byref(d.plan), None, 0, None, None, None, 0, 1, FAKE, None, FAKE, None) == 0
    assert g(ctypes.byref(d.plan), None, 0, None, None, None, 0, 1, None, ctypes.byref(m), FAKE,
             None) == -4


def test_zero_tokens_v41_is_a_no_op(lib):
    plan, _ = B.dsa_decode_plan(0, 16, 128, 0, 4)
    assert lib.dsa_decode_run_v41(ctypes.byref(plan), None, 0, None, 0, 0, None, None, 0, None,
                                  None, None, 0, None, None, None, None, 0, 1, 1.0, None, None,
                                  None, None) == 0
    assert lib.dsa_decode_combine_v41(ctypes.byref(plan), None, 0, None, None, None, 0, 1, None,
                                      None, None, None) == 0
