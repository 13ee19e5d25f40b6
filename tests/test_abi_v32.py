"""C-ABI checks of the V3.2 record (656 bytes, 576-dim keys) that need no
GPU: the d_qk plan and the rules a run checks before any CUDA call (every
run below breaks at least one of them)."""
import ctypes

import pytest

from swa_paged_decode_gb300 import binding as B
from tests.test_abi import FAKE, Args, lib  # noqa: F401  (lib is a fixture)
from tests.test_abi_v41 import run_v41

V32 = 4


def plan576(H=64, T=4, ws=128, we=256):
    return B.dsa_decode_plan_qk(T, H, ws, we, 4, 576)


def test_plan_caps_heads_per_group_at_32():
    for H, hpg in ((16, 16), (32, 32), (64, 32), (128, 32)):
        plan, _ = plan576(H=H, T=4096)            # a batch the small-batch split leaves alone
        assert plan.d_qk == 576 and plan.heads_per_group == hpg
        small, _ = plan576(H=H, T=4)
        assert small.heads_per_group <= hpg
        assert plan.head_groups * plan.heads_per_group == H and plan.kernel == 1
    plan, _ = B.dsa_decode_plan(4, 64, 128, 256, 4)
    assert plan.d_qk == 512
    plan2, _ = B.dsa_decode_plan_qk(4, 64, 128, 256, 4, 512)
    assert bytes(plan2) == bytes(plan)


def test_plan_rejects_other_dims_and_48_96_heads(lib):
    p, n = B.Plan(), ctypes.c_size_t(0)
    for d in (0, 511, 513, 575, 577, 1024):
        assert lib.dsa_decode_plan_qk(4, 64, 128, 0, 4, d, ctypes.byref(p), ctypes.byref(n)) == -1
    for H in (48, 96):
        assert lib.dsa_decode_plan_qk(4, H, 128, 0, 4, 576, ctypes.byref(p), ctypes.byref(n)) == -2
        assert lib.dsa_decode_plan_qk(4, H, 128, 0, 4, 512, ctypes.byref(p), ctypes.byref(n)) == 0


def v32_args(H=64):
    a = Args(H=H, we=256)
    a.plan, a.nbytes = plan576(H=H)
    a.kw["ws_bytes"] = a.nbytes
    a.kw["q_st"], a.kw["q_sh"] = H * 576, 576
    a.swa = B.CacheDesc(FAKE, 64, 64 * 656, 64, V32)
    a.extra = B.CacheDesc(FAKE, 64, 64 * 656, 64, V32)
    return a


def test_v32_descriptors_pass_the_list_checks(lib):
    a = v32_args()
    # the extra list's page stride is short of 64 records of 656 bytes
    assert a.call(lib, extra_desc=B.CacheDesc(FAKE, 64, 64 * 528, 64, V32)) == -1
    # misaligned extra list: the refusal comes after the sliding-window list passed
    assert a.call(lib, extra_desc=B.CacheDesc(FAKE + 8, 64, 64 * 656, 64, V32)) == -3


def test_q_rows_must_hold_576_dims(lib):
    a = v32_args()
    assert a.call(lib, q_sh=512, q_st=64 * 512) == -1


@pytest.mark.parametrize("case", ["fp8_list_576_plan", "v32_list_512_plan", "mixed", "rope"])
def test_v32_rules(lib, case):
    a = v32_args()
    if case == "fp8_list_576_plan":
        assert a.call(lib, swa_desc=B.CacheDesc(FAKE, 64, 64 * 528, 64, 0),
                      extra_desc=B.CacheDesc(FAKE, 64, 64 * 528, 64, 0)) == -2
    elif case == "v32_list_512_plan":
        b = Args(H=64, we=256)
        assert b.call(lib, swa_desc=a.swa, extra_desc=a.extra, q_sh=576, q_st=64 * 576) == -2
    elif case == "mixed":
        assert a.call(lib, extra_desc=B.CacheDesc(FAKE, 64, 64 * 288, 64, 1)) == -2
    else:   # q arrives rotated: a RoPE table is refused with these records
        assert a.call(lib, pos=FAKE, cs=FAKE, cs_rows=16) == -2


def test_v41_entry_refuses_v32(lib):
    a = v32_args()
    assert run_v41(lib, a, out=FAKE) == -2
