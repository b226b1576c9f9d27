"""The C-ABI library: builds, exports every declared symbol, validates on the host.

No test here launches a kernel: argument, alignment, precondition and workspace
errors are decided on the host before any CUDA call, and an otherwise valid call on
a machine without a GB300 stops at the device check.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "detgemm.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    from deterministic_detgemm_w8a8_gb300 import build as B
    B.build()
    import deterministic_detgemm_w8a8_gb300 as dg
    return dg.load()


def _declared():
    src = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"DETGEMM_API\s+[\w\s\*]*?\b(detgemm_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("detgemm_w8a8", "detgemm_ozaki_f32", "detgemm_quantize_pow2", "detgemm_slice_f32",
              "detgemm_w8a8_workspace_size", "detgemm_ozaki_workspace_size", "detgemm_get_device_status",
              "detgemm_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from deterministic_detgemm_w8a8_gb300 import LIB_PATH, SIGNATURES
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s+(detgemm_\w+)", out))
    declared = set(_declared())
    assert declared <= exported, declared - exported
    # the binding knows the signature of every declared call, and nothing else
    assert set(SIGNATURES) == declared
    for n in declared:
        assert hasattr(lib, n)


def test_status_strings(lib):
    import deterministic_detgemm_w8a8_gb300 as dg
    for code, name in [(0, "DETGEMM_OK"), (1, "DETGEMM_ERR_INVALID_ARG"), (2, "DETGEMM_ERR_ALIGNMENT"),
                       (3, "DETGEMM_ERR_PRECONDITION"), (4, "DETGEMM_ERR_WORKSPACE"),
                       (5, "DETGEMM_ERR_UNSUPPORTED_DEVICE"), (6, "DETGEMM_ERR_CUDA"),
                       (7, "DETGEMM_ERR_TIMEOUT"), (8, "DETGEMM_ERR_NONFINITE")]:
        assert dg.status_string(code) == name
    assert lib.detgemm_version() >= 100


# fake, never-dereferenced device addresses
P = 0x7f0000000000
P1 = P + 1


def _w8a8(lib, A=P, lda=512, W=P, ldw=512, ea=P, ew=P, C=P, ldc=256, M=64, N=256, K=512, split=1,
          ws=P, wsb=1 << 30):
    return lib.detgemm_w8a8(A, lda, W, ldw, ea, ew, C, ldc, M, N, K, split, ws, wsb, None)


def test_w8a8_argument_validation(lib):
    import deterministic_detgemm_w8a8_gb300 as dg
    assert _w8a8(lib, K=0) == dg.ERR_INVALID_ARG
    assert _w8a8(lib, M=-1) == dg.ERR_INVALID_ARG
    assert _w8a8(lib, K=131072, lda=131072, ldw=131072) == dg.ERR_PRECONDITION
    assert _w8a8(lib, split=0) == dg.ERR_INVALID_ARG
    assert _w8a8(lib, split=9) == dg.ERR_INVALID_ARG  # K=512 has 8 blocks of 64
    assert _w8a8(lib, A=None) == dg.ERR_INVALID_ARG
    assert _w8a8(lib, ea=None) == dg.ERR_INVALID_ARG
    assert _w8a8(lib, lda=500) == dg.ERR_INVALID_ARG  # lda < K
    assert _w8a8(lib, A=P1) == dg.ERR_ALIGNMENT
    assert _w8a8(lib, lda=520) == dg.ERR_ALIGNMENT
    assert _w8a8(lib, ldc=260) == dg.ERR_ALIGNMENT  # 520 bytes
    need = dg.w8a8_workspace_size(64, 256, 512, 2)
    assert need >= 64 * 256 * 4
    assert _w8a8(lib, split=2, ws=None, wsb=0) == dg.ERR_WORKSPACE
    assert _w8a8(lib, split=2, ws=P, wsb=need - 1) == dg.ERR_WORKSPACE
    # the decode-shaped path (M <= 64) needs scratch at any split; larger M only to split
    assert dg.w8a8_workspace_size(16, 256, 512, 1) >= 16 * 256 * 4
    assert _w8a8(lib, M=16, ws=None, wsb=0) == dg.ERR_WORKSPACE
    # empty problems succeed without touching the device
    assert _w8a8(lib, M=0, A=None, C=None) == dg.OK
    assert _w8a8(lib, N=0) == dg.OK


def test_bias_entry_points_validate(lib):
    import torch
    import deterministic_detgemm_w8a8_gb300 as dg
    wb = lib.detgemm_w8a8_bias

    def b(bias=P, M=64, split=1, ws=P, wsb=1 << 30, K=512):
        # A, lda, W, ldw, ea, ew, bias, C, ldc, M, N, K, split, ws, ws_bytes
        return wb(P, 512, P, 512, P, P, bias, P, 256, M, 256, K, split, ws, wsb, None)

    assert b(bias=None) == dg.ERR_INVALID_ARG
    assert b(bias=P1) == dg.ERR_ALIGNMENT
    assert b(K=0) == dg.ERR_INVALID_ARG
    assert b(K=1024) == dg.ERR_INVALID_ARG  # lda 512 < K
    assert b(K=131072) == dg.ERR_PRECONDITION
    assert b(split=2, ws=None, wsb=0) == dg.ERR_WORKSPACE
    assert b(M=0, bias=None) == dg.OK  # empty: nothing read
    lb = lib.detgemm_linear_w8a8_bias
    # X, dtype, ldx, mode, W, ldw, W16, ldw16, ew, bias, C, ldc, ea_out, M, N, K, split, ws, ws_bytes
    assert lb(P, 0, 64, 0, P, 64, None, 0, P, None, P, 64, None, 100, 64, 64, 1, P, 1 << 30, None) == \
        dg.ERR_INVALID_ARG
    assert lb(P, 0, 64, 0, P, 64, None, 0, P, P1, P, 64, None, 100, 64, 64, 1, P, 1 << 30, None) == \
        dg.ERR_ALIGNMENT
    assert lb(P, 2, 64, 0, P, 64, None, 0, P, P, P, 64, None, 4, 64, 64, 1, P, 1 << 30, None) == dg.ERR_INVALID_ARG
    assert lb(P, 0, 64, 0, P, 64, None, 0, P, P, P, 64, None, 0, 64, 64, 1, None, 0, None) == dg.OK
    if not torch.cuda.is_available():
        assert b() == dg.ERR_UNSUPPORTED_DEVICE
        assert lb(P, 0, 64, 0, P, 64, None, 0, P, P, P, 64, None, 100, 64, 64, 1, P, 1 << 30, None) == \
            dg.ERR_UNSUPPORTED_DEVICE


def test_w8a8_valid_call_stops_at_device_check_without_gpu(lib):
    import torch
    import deterministic_detgemm_w8a8_gb300 as dg
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _w8a8(lib) == dg.ERR_UNSUPPORTED_DEVICE


def test_other_entry_points_validate(lib):
    import deterministic_detgemm_w8a8_gb300 as dg
    q = lib.detgemm_quantize_pow2
    assert q(P, 2, 64, 4, 64, 0, P, 64, P, None) == dg.ERR_INVALID_ARG  # dtype
    assert q(P, 0, 64, 4, 64, 2, P, 64, P, None) == dg.ERR_INVALID_ARG  # mode
    assert q(P, 0, 60, 4, 60, 0, P, 64, P, None) == dg.ERR_ALIGNMENT  # 120-byte rows
    assert q(P, 0, 64, 0, 64, 0, None, 64, None, None) == dg.OK
    s = lib.detgemm_slice_f32
    assert s(P, 64, 4, 64, 0, 10, P, P, None) == dg.ERR_INVALID_ARG  # nslices
    assert s(P, 64, 4, 64, 2, 7, P, P, None) == dg.ERR_INVALID_ARG  # axis
    assert s(P1, 64, 4, 64, 0, 7, P, P, None) == dg.ERR_ALIGNMENT
    o = lib.detgemm_ozaki_f32
    assert o(P, 64, P, 64, P, 64, 64, 64, 64, 7, 19, 1, P, 1 << 30, None) == dg.ERR_INVALID_ARG
    # (max_diag - 1 pairs capped at nslices) * K * 127^2 must stay below 2^31
    assert o(P, 19024, P, 64, P, 64, 64, 64, 19024, 7, 8, 1, P, 1 << 40, None) == dg.ERR_PRECONDITION
    assert o(P, 64, P, 64, P, 64, 64, 64, 64, 7, 8, 1, P, 16, None) == dg.ERR_WORKSPACE
    assert dg.ozaki_workspace_size(64, 64, 64) > 7 * 64 * 64 * 2
    li = lib.detgemm_linear_w8a8
    # X, dtype, ldx, mode, W, ldw, W16, ldw16, ew, C, ldc, ea_out, M, N, K, split, ws, ws_bytes
    assert li(P, 2, 64, 0, P, 64, None, 0, P, P, 64, None, 4, 64, 64, 1, P, 1 << 30, None) == dg.ERR_INVALID_ARG
    assert li(P, 0, 64, 2, P, 64, None, 0, P, P, 64, None, 4, 64, 64, 1, P, 1 << 30, None) == dg.ERR_INVALID_ARG
    assert li(P, 0, 131072, 0, P, 131072, None, 0, P, P, 64, None, 4, 64, 131072, 1, P, 1 << 30,
              None) == dg.ERR_PRECONDITION
    assert li(P, 0, 60, 0, P, 64, None, 0, P, P, 64, None, 4, 64, 60, 1, P, 1 << 30, None) == dg.ERR_ALIGNMENT
    assert li(P, 0, 64, 0, P, 64, P1, 64, P, P, 64, None, 100, 64, 64, 1, P, 1 << 30, None) == dg.ERR_ALIGNMENT
    assert li(P, 0, 64, 0, P, 64, None, 0, P, P, 64, None, 100, 64, 64, 1, P, 16, None) == dg.ERR_WORKSPACE
    assert li(P, 0, 64, 0, P, 64, None, 0, P, P, 64, None, 0, 64, 64, 1, None, 0, None) == dg.OK
    assert lib.detgemm_linear_w8a8_workspace_size(100, 64, 64, 1, 0) > lib.detgemm_linear_w8a8_workspace_size(
        100, 64, 64, 1, 1)
    h = lib.detgemm_w8a8_host
    assert h(P, 64, P, 64, P, P, P, 64, 100, 64, 131072, P, 1 << 40, None) == dg.ERR_PRECONDITION
    assert h(P, 60, P, 64, P, P, P, 64, 100, 64, 64, P, 1 << 40, None) == dg.ERR_INVALID_ARG  # lda < K
    assert h(P, 64, P, 64, P, P, P, 64, 100, 64, 64, P, 16, None) == dg.ERR_WORKSPACE
    assert h(P, 64, P, 64, P, P, P, 64, 100, 64, 64, P + 16, 1 << 40, None) == dg.ERR_ALIGNMENT
    assert h(None, 64, None, 64, None, None, None, 64, 0, 64, 64, None, 0, None) == dg.OK
    assert lib.detgemm_w8a8_host_buffer_size(8192, 4096, 12288) > 4096 * 12288 * 3
    c = lib.detgemm_ozaki_combine
    assert c(P, 64, 1, P, P, P, 1, 64, 4, 64, None) == dg.ERR_INVALID_ARG  # max_diag < 2
    assert c(P, 64, 19, P, P, P, 1, 64, 4, 64, None) == dg.ERR_INVALID_ARG  # max_diag > 18
    assert c(P, 64, 8, P, P, P, 0, 64, 4, 64, None) == dg.ERR_INVALID_ARG  # bf16 output
    assert c(P, 60, 8, P, P, P, 1, 64, 4, 64, None) == dg.ERR_INVALID_ARG  # ldT < N
    assert c(P, 66, 8, P, P, P, 1, 64, 4, 64, None) == dg.ERR_ALIGNMENT  # 264-byte rows
    assert c(P, 64, 8, P, P, P, 2, 65, 4, 64, None) == dg.ERR_ALIGNMENT  # fp64 rows of 520 bytes
    assert c(P1, 64, 8, P, P, P, 1, 64, 4, 64, None) == dg.ERR_ALIGNMENT
    assert c(None, 64, 8, None, None, None, 1, 64, 0, 64, None) == dg.OK  # empty
    s64 = lib.detgemm_slice_f64
    assert s64(P, 64, 4, 64, 0, 13, P, P, None) == dg.ERR_INVALID_ARG  # nslices
    assert s64(P, 63, 4, 63, 0, 8, P, P, None) == dg.ERR_ALIGNMENT  # 504-byte rows
    o64 = lib.detgemm_ozaki_f64
    assert o64(P, 64, P, 64, P, 64, 64, 64, 64, 8, 17, 1, P, 1 << 30, None) == dg.ERR_INVALID_ARG
    assert o64(P, 64, P, 64, P, 64, 64, 64, 64, 13, 9, 1, P, 1 << 30, None) == dg.ERR_INVALID_ARG
    # 8 pairs * K * 127^2 must stay below 2^31: K = 16644 passes the bound, 16646 does not
    assert o64(P, 16646, P, 64, P, 64, 64, 64, 16646, 8, 9, 1, P, 1 << 40, None) == dg.ERR_PRECONDITION
    assert o64(P, 64, P, 64, P, 64, 64, 64, 64, 8, 9, 1, P, 16, None) == dg.ERR_WORKSPACE
    assert dg.ozaki_f64_workspace_size(64, 64, 64) > 8 * 64 * 64 * 2


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import deterministic_detgemm_w8a8_gb300 as dg
    A = torch.zeros((4, 16), dtype=torch.int8)
    with pytest.raises(ValueError):
        dg.w8a8(A, A, torch.zeros(4, dtype=torch.int32), torch.zeros(4, dtype=torch.int32))


def test_split_exact_entry_points_validate(lib):
    import torch
    import deterministic_detgemm_w8a8_gb300 as dg
    se = lib.detgemm_w8a8_split_exact
    parts = ctypes.c_int(-7)

    def w(M=300, K=512, split=2, ws=P, wsb=1 << 30, ea=P):
        # A, lda, W, ldw, ea, ew, C, ldc, M, N, K, split, ws, ws_bytes, parts_run, stream
        return se(P, 512, P, 512, ea, P, P, 256, M, 256, K, split, ws, wsb, ctypes.byref(parts), None)

    # the same host-side checks as detgemm_w8a8, and parts_run reads 0 after an error
    assert w(split=0) == dg.ERR_INVALID_ARG and parts.value == 0
    parts.value = -7
    assert w(split=9) == dg.ERR_INVALID_ARG and parts.value == 0
    assert w(K=131072) == dg.ERR_PRECONDITION
    assert w(ea=None) == dg.ERR_INVALID_ARG
    assert w(split=2, ws=None, wsb=0) == dg.ERR_WORKSPACE
    assert w(M=16, split=1, ws=None, wsb=0) == dg.ERR_WORKSPACE
    assert w(M=0) == dg.OK
    so = lib.detgemm_ozaki_f32_split_exact
    parts.value = -7
    assert so(P, 128, P, 64, P, 64, 64, 64, 128, 7, 8, 2, P, 16, ctypes.byref(parts), None) == dg.ERR_WORKSPACE
    assert parts.value == 0
    assert so(P, 64, P, 64, P, 64, 64, 64, 64, 7, 8, 0, P, 1 << 30, None, None) == dg.ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert w() == dg.ERR_UNSUPPORTED_DEVICE
        assert so(P, 64, P, 64, P, 64, 64, 64, 64, 7, 8, 1, P, 1 << 30, None, None) == dg.ERR_UNSUPPORTED_DEVICE


def test_noalloc_validates_in_w8a8_order(lib):
    import torch
    import deterministic_detgemm_w8a8_gb300 as dg
    na = lib.detgemm_w8a8_noalloc

    def n(A=P, ea=P, M=300, K=512, split=1):
        # A, lda, W, ldw, ea, ew, C, ldc, M, N, K, split, stream
        return na(A, 512, P, 512, ea, P, P, 256, M, 256, K, split, None)

    # a misaligned A with a null ea reports ALIGNMENT, as detgemm_w8a8 does
    assert n(A=P1, ea=None) == dg.ERR_ALIGNMENT
    assert n(ea=None) == dg.ERR_INVALID_ARG
    assert n(split=9) == dg.ERR_INVALID_ARG
    assert n(M=0) == dg.OK
    # the scratch-size rule: the decode kernels' scratch at M <= 64, the split accumulator above
    ss = lib.detgemm_w8a8_noalloc_scratch_size
    assert ss(300, 256, 512, 1) == 0
    assert ss(300, 256, 512, 2) >= 300 * 256 * 4
    assert ss(16, 256, 512, 1) >= 16 * 256 * 4 + 16 * 512 * 2
    assert ss(0, 256, 512, 1) == 0
    if not torch.cuda.is_available():
        # the device check comes before the size check
        assert na(P, 256, P, 256, P, P, P, 4096, 1024, 4096, 256, 2, None) == dg.ERR_UNSUPPORTED_DEVICE
        assert n() == dg.ERR_UNSUPPORTED_DEVICE
