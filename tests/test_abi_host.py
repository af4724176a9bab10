"""Host-side checks of the C ABI (no GPU needed): symbols, argument validation, workspace queries."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import mixture_experts_routed_router_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "liger_moe.h")

OK, INVALID, MISALIGNED, CAPACITY, UNSUPPORTED = 0, -1, -2, -3, -4


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(liger_moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return moe.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("liger_moe_route_topk", "liger_moe_dispatch", "liger_moe_grouped_swiglu_fwd", "liger_moe_combine",
              "liger_moe_bwd_dx_dw", "liger_moe_grouped_swiglu_fwd_gather", "liger_moe_bwd_dx_dw_gather",
              "liger_moe_grouped_glu_fwd", "liger_moe_bwd_dx_dw_glu", "liger_moe_router_logits",
              "liger_moe_router_bwd"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in liger_moe.h but not exported"


def test_only_liger_symbols_are_exported():
    out = subprocess.run(["nm", "-D", "--defined-only", moe.library_path()], capture_output=True, text=True,
                         check=True).stdout
    syms = [l.split()[-1] for l in out.splitlines() if l.strip() and l.split()[-2] in ("T", "W", "D", "B")]
    assert syms and all(s.startswith("liger_moe_") or s.startswith("_") for s in syms), syms


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "liger_moe.h"\nint main(void){return liger_moe_abi_version() > 0 ? 0 : 1;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", "-I", os.path.dirname(HEADER), str(src), "-o",
                    str(tmp_path / "use.o")], check=True)


def test_status_strings(lib):
    assert lib.liger_moe_status_string(0) == b"LIGER_MOE_OK"
    assert lib.liger_moe_status_string(-3) == b"LIGER_MOE_ERR_CAPACITY"
    assert lib.liger_moe_abi_version() >= 100


D = ctypes.c_void_p(256)  # never dereferenced: every call below is rejected or is a size query


def test_route_argument_errors(lib):
    f = lib.liger_moe_route_topk
    assert f(D, -1, 8, 2, D, D, None) == INVALID
    assert f(D, 4, 8, 9, D, D, None) == INVALID      # k > E
    assert f(D, 4, 8, 0, D, D, None) == INVALID      # k < 1
    assert f(D, 4, 2048, 2, D, D, None) == CAPACITY  # E above the limit
    assert f(D, 4, 64, 33, D, D, None) == CAPACITY   # k above the limit
    assert f(None, 4, 8, 2, D, D, None) == INVALID
    assert f(D, 2 ** 30, 64, 8, D, D, None) == CAPACITY  # T*k beyond int32


def test_dispatch_validation_and_query(lib):
    n = ctypes.c_size_t(0)
    f = lib.liger_moe_dispatch
    assert f(D, None, None, 8192, 0, 256, 8, D, D, D, D, None, None, None, ctypes.byref(n), None) == OK
    assert n.value >= 256 * (8192 * 8 // 256) * 4
    assert f(D, None, D, 16, 100, 8, 2, D, D, D, D, None, D, None, ctypes.byref(n), None) == MISALIGNED
    assert f(D, None, None, 16, 0, 8, 2, D, D, D, D, D, None, None, ctypes.byref(n), None) == INVALID  # w_perm w/o w
    small = ctypes.c_size_t(8)
    assert f(D, None, None, 8192, 0, 256, 8, D, D, D, D, None, None, D, ctypes.byref(small), None) == CAPACITY


def test_grouped_validation_and_query(lib):
    n = ctypes.c_size_t(0)
    f = lib.liger_moe_grouped_swiglu_fwd
    assert f(D, D, D, D, D, 1024, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == OK
    assert n.value >= 4 * 9
    assert f(D, D, D, D, D, 1024, 256, 96, 8, D, None, D, None, ctypes.byref(n), None) == MISALIGNED
    assert f(D, D, D, D, D, 1024, 200, 128, 8, D, None, D, None, ctypes.byref(n), None) == MISALIGNED
    assert f(ctypes.c_void_p(258), D, D, D, D, 1024, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == MISALIGNED
    assert f(D, D, D, D, D, 1024, 256, 128, 0, D, None, D, None, ctypes.byref(n), None) == INVALID
    assert f(D, D, None, D, D, 1024, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == INVALID


def test_bwd_workspace_grows_when_recomputing(lib):
    a = moe.workspace_bytes("bwd_dx_dw", T=256, H=256, I=128, E=8, k=2, saved_gu=True)
    b = moe.workspace_bytes("bwd_dx_dw", T=256, H=256, I=128, E=8, k=2, saved_gu=False)
    R, H, I = 512, 256, 128
    # dy_perm [R,H] + dx_perm [R,H] + dgu hi/lo [2R,2I] + w*h hi/lo [2R,I] (bf16)
    assert a >= R * (4 * H + 12 * I)
    assert b >= a + R * 2 * I * 4
    # token-major entry point: dY rows are gathered inside the GEMMs, so no dy_perm
    g = moe.workspace_bytes("bwd_dx_dw", T=256, H=256, I=128, E=8, k=2, saved_gu=True, gather=True)
    assert g >= R * (2 * H + 12 * I) and a - g >= R * H * 2


def test_bwd_workspace_holds_the_fp16_copies_from_32768_rows(lib):
    """From R = 32768 routed rows the x_perm backward may take the fp16 weight-gradient pass: its
    workspace then holds fp16 copies of the x and dY rows; the gathered backward never does."""
    q = lambda T, gather=False: moe.workspace_bytes("bwd_dx_dw", T=T, H=256, I=128, E=8, k=2, gather=gather)
    small, big = q(16383), q(16384)  # R = 32766, 32768
    assert big - small >= 2 * 32768 * 256 * 2  # x16 and dy16 [R, H] fp16 on top
    assert q(16384, gather=True) - q(16383, gather=True) < 64 * 1024  # two more rows and alignment only


def test_dw_fp16_switch_validates(lib):
    assert lib.liger_moe_set_dw_fp16(2) == INVALID
    assert lib.liger_moe_set_dw_fp16(-1) == INVALID
    assert lib.liger_moe_set_dw_fp16(0) == OK
    assert lib.liger_moe_set_dw_fp16(1) == OK  # the default, restored


def test_gather_entry_points_validate_like_their_x_perm_twins(lib):
    n = ctypes.c_size_t(0)
    f = lib.liger_moe_grouped_swiglu_fwd_gather
    # (x, row_to_slot, T, k, m_indptr, w_gate_up, w_down, w_perm, H, I, E, h, gu, y, ws, ws_bytes, stream)
    assert f(D, D, 512, 2, D, D, D, D, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == OK
    q = n.value
    assert lib.liger_moe_grouped_swiglu_fwd(D, D, D, D, D, 1024, 256, 128, 8, D, None, D, None, ctypes.byref(n),
                                            None) == OK
    assert n.value == q
    assert f(None, D, 512, 2, D, D, D, D, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == INVALID
    assert f(D, None, 512, 2, D, D, D, D, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == INVALID
    assert f(D, D, 512, 0, D, D, D, D, 256, 128, 8, D, None, D, None, ctypes.byref(n), None) == INVALID
    assert f(D, D, 512, 2, D, D, D, D, 200, 128, 8, D, None, D, None, ctypes.byref(n), None) == MISALIGNED
    assert f(ctypes.c_void_p(258), D, 512, 2, D, D, D, D, 256, 128, 8, D, None, D, None, ctypes.byref(n),
             None) == MISALIGNED
    g = lib.liger_moe_bwd_dx_dw_gather
    args = [D, D, D, D, D, D, D, D, D, D, D, D, 256, 256, 128, 8, 2, D, D, D, D, None, ctypes.byref(n), None]
    assert g(*args) == OK
    assert n.value == moe.workspace_bytes("bwd_dx_dw", T=256, H=256, I=128, E=8, k=2, saved_gu=True, gather=True)
    bad = list(args)
    bad[1] = None  # x
    assert g(*bad) == INVALID
    bad = list(args)
    bad[16] = 9  # k > E
    assert g(*bad) == INVALID


def test_activation_ids_match_the_header():
    text = open(HEADER).read()
    for name, v in moe.ACTIVATIONS.items():
        assert re.search(rf"LIGER_MOE_ACT_{name.upper()}\s*=\s*{v}\b", text), name


def test_glu_entry_points_validate_the_activation(lib):
    n = ctypes.c_size_t(0)
    f = lib.liger_moe_grouped_glu_fwd
    F = ctypes.c_float

    def fwd(act, clamp):  # (x_perm, m_indptr, w_gu, w_d, w_perm, R, H, I, E, act, clamp, h, gu, y, ws, ws_bytes, s)
        return f(D, D, D, D, D, 1024, 256, 128, 8, act, F(clamp), D, None, D, None, ctypes.byref(n), None)

    assert fwd(0, 0.0) == OK
    q = n.value
    assert lib.liger_moe_grouped_swiglu_fwd(D, D, D, D, D, 1024, 256, 128, 8, D, None, D, None, ctypes.byref(n),
                                            None) == OK
    assert n.value == q  # same workspace for every activation
    for act, clamp in ((3, 0.0), (4, 0.0), (1, 7.0), (2, 7.0), (5, 0.0)):
        assert fwd(act, clamp) == OK
    # unknown ids; bounded variants need a finite positive clamp
    for act, clamp in ((-1, 0.0), (6, 0.0), (1, 0.0), (2, -1.0), (1, float("inf")), (2, float("nan"))):
        assert fwd(act, clamp) == INVALID, (act, clamp)
    g = lib.liger_moe_bwd_dx_dw_glu
    # (dy, x_perm, h, gu, ids, w, indptr, r2s, s2r, w_perm, w_gu, w_d, T, H, I, E, k, act, clamp, dx, dwgu, dwd,
    #  d_logits, ws, ws_bytes, stream)
    args = [D, D, D, D, D, D, D, D, D, D, D, D, 256, 256, 128, 8, 2, 3, F(0.0), D, D, D, D, None, ctypes.byref(n),
            None]
    assert g(*args) == OK
    assert n.value == moe.workspace_bytes("bwd_dx_dw", T=256, H=256, I=128, E=8, k=2, saved_gu=True)
    args[3] = None  # recompute the factors
    assert g(*args) == OK
    assert n.value == moe.workspace_bytes("bwd_dx_dw", T=256, H=256, I=128, E=8, k=2, saved_gu=False)
    args[17] = 7
    assert g(*args) == INVALID
    args[17], args[18] = 1, F(0.0)
    assert g(*args) == INVALID


def test_combine_argument_errors(lib):
    f = lib.liger_moe_combine
    assert f(D, D, 4, 100, 2, D, None) == MISALIGNED
    assert f(D, D, -1, 128, 2, D, None) == INVALID
    assert f(D, D, 4, 128, 33, D, None) == CAPACITY


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_calls_fail_loudly_without_a_device(lib):
    # valid arguments, no sm_103 device: the library refuses instead of computing anything
    assert lib.liger_moe_route_topk(D, 4, 8, 2, D, D, None) == UNSUPPORTED
    with pytest.raises(RuntimeError):  # LigerMoEError or torch's "no CUDA" error: never a silent result
        moe.device_error()


def test_router_entry_points_validate_before_launch(lib):
    f = lib.liger_moe_router_logits
    # (x, w_router, bias, T, H, E, logits, stream)
    assert f(D, D, None, -1, 256, 8, D, None) == INVALID
    assert f(D, D, None, 4, 256, 0, D, None) == INVALID
    assert f(D, D, None, 4, 256, 2048, D, None) == CAPACITY    # E above the limit
    assert f(D, D, None, 4, 200, 8, D, None) == MISALIGNED     # H not a multiple of 64
    assert f(None, D, None, 4, 256, 8, D, None) == INVALID
    assert f(D, None, None, 4, 256, 8, D, None) == INVALID
    assert f(D, D, None, 4, 256, 8, ctypes.c_void_p(260), None) == MISALIGNED
    g = lib.liger_moe_router_bwd
    # (d_logits, ids, m_indptr, row_to_slot, x, w_router, T, H, E, k, dx, dw_router, d_bias, stream)
    assert g(D, D, D, D, D, D, 4, 256, 8, 9, D, D, None, None) == INVALID       # k > E
    assert g(D, D, D, D, D, D, 4, 256, 8, 0, D, D, None, None) == INVALID       # k < 1
    assert g(D, D, D, D, D, D, 4, 256, 2048, 2, D, D, None, None) == CAPACITY
    assert g(D, D, D, D, D, D, 4, 192 + 8, 8, 2, D, D, None, None) == MISALIGNED
    assert g(D, D, None, D, D, D, 4, 256, 8, 2, D, D, None, None) == INVALID    # m_indptr
    assert g(D, D, D, D, D, D, 4, 256, 8, 2, None, D, None, None) == INVALID    # dx
    assert g(D, D, D, D, D, D, 4, 256, 8, 2, D, None, None, None) == INVALID    # dw_router
    assert g(D, D, D, D, ctypes.c_void_p(264), D, 4, 256, 8, 2, D, D, None, None) == MISALIGNED


def test_selftest_limit_is_validated(lib):
    for bad in (0, -5, 1000001):
        assert lib.liger_moe_selftest_wait_timeout(bad, None) == INVALID
