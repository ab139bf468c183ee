"""Host-only checks of the C ABI (no GPU needed): the library loads, exports every entry
point include/awq.h declares, and rejects bad arguments on the host before touching a
device.  No call here reaches a kernel launch: the addresses are fake, so a call with
valid arguments (expected to return AWQ_ERR_UNSUPPORTED_DEVICE) runs only where no CUDA device is
present."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq.h")

INVALID, SHAPE, MISALIGNED, DEVICE = 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    # The calls below pass fake device addresses: where a CUDA device is present, a call
    # with valid arguments would launch a kernel on them, so these checks run only where
    # there is none (the GPU tests cover the same entry points with real buffers).
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only checks with fake device addresses; a CUDA device is present")
    from w4a16_weight_only_gb300 import build
    build.build()
    from w4a16_weight_only_gb300 import _binding
    return _binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(awq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("awq_gemm", "awq_dequant", "awq_runtime_available", "awq_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_header(lib):
    from w4a16_weight_only_gb300 import _binding
    assert set(_declared_functions()) == set(_binding.SIGNATURES)


def test_status_strings(lib):
    assert lib.awq_status_string(0) == b"AWQ_OK"
    assert lib.awq_status_string(6) == b"AWQ_ERR_TIMEOUT"


P = ctypes.c_void_p
A = P(0x100000)        # fake, 256-byte aligned "device" addresses: never dereferenced
B = P(0x200000)
ODD = P(0x100001)


def gemm(lib, M=1, K=256, N=256, G=128, x=A, qw=A, qz=A, sc=A, bias=None, y=B, path=0):
    return lib.awq_gemm_ex(x, qw, qz, sc, bias, M, K, N, G, y, path, None)


def test_gemm_shape_validation(lib):
    assert gemm(lib, K=0) == INVALID
    assert gemm(lib, K=-16) == INVALID
    assert gemm(lib, N=-8) == INVALID
    assert gemm(lib, M=-1) == INVALID
    assert gemm(lib, G=0) == INVALID
    assert gemm(lib, G=-2) == INVALID
    assert gemm(lib, N=12) == SHAPE            # not a multiple of 8
    assert gemm(lib, K=256, G=96) == SHAPE     # K % G != 0
    assert gemm(lib, K=1 << 31) == SHAPE       # size limit
    assert gemm(lib, path=7) == INVALID
    msg = lib.awq_last_error().decode()
    assert "path" in msg


def test_gemm_empty_is_ok_without_device(lib):
    # M == 0 or N == 0: nothing to compute, no launch, even with null pointers.
    assert lib.awq_gemm(None, None, None, None, None, 0, 256, 256, 128, None, None) == 0
    assert lib.awq_gemm(None, None, None, None, None, 4, 256, 0, 128, None, None) == 0
    assert lib.awq_last_error() == b""


def test_gemm_null_and_alignment(lib):
    assert gemm(lib, x=None) == INVALID
    assert gemm(lib, y=None) == INVALID
    assert gemm(lib, qz=None) == INVALID
    assert gemm(lib, x=ODD) == MISALIGNED
    assert gemm(lib, sc=ODD) == MISALIGNED
    assert gemm(lib, bias=ODD) == MISALIGNED
    assert gemm(lib, qw=P(0x100002)) == MISALIGNED


def test_dequant_validation(lib):
    d = lib.awq_dequant
    assert d(A, A, A, 0, 256, 128, B, 0, None) == INVALID
    assert d(A, A, A, 256, 20, 128, B, 0, None) == SHAPE
    assert d(A, A, A, 256, 256, 100, B, 0, None) == SHAPE
    assert d(A, A, A, 256, 256, 128, B, 5, None) == INVALID        # bad dtype
    assert d(A, A, A, 256, 256, 128, P(0x100002), 1, None) == MISALIGNED  # f32 out
    assert d(A, A, A, 256, 0, 128, B, 0, None) == 0                 # N == 0: no launch
    assert d(None, A, A, 256, 256, 128, B, 0, None) == INVALID


def test_path_selection_is_host_only(lib):
    sel = lib.awq_gemm_select_path
    # decode shapes
    assert sel(1, 4096, 4096, 128, A, A, A, A, None, B) == 1
    assert sel(32, 11008, 4096, 128, A, A, A, A, None, B) == 1
    # K not a multiple of 16 -> generic kernel
    assert sel(1, 200, 64, 8, A, A, A, A, None, B) == 3
    # group size not a multiple of 16 -> generic kernel
    assert sel(4, 256, 64, 8, A, A, A, A, None, B) == 3
    # invalid shape -> 0
    assert sel(1, 256, 12, 128, A, A, A, A, None, B) == 0


def test_valid_call_without_sm103_device_is_refused(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present; covered by the GPU tests")
    assert gemm(lib) == DEVICE
    assert lib.awq_runtime_available() == 0
    assert lib.awq_last_error() != b""


def test_selftest_argument_checks_are_host_side(lib):
    # out-of-range limits are refused before any device access
    assert lib.awq_selftest_wait_timeout(0, None) == 1
    assert lib.awq_selftest_wait_timeout(2_000_000_000, None) == 1
    # a valid limit without a CC 10.3 device is refused, nothing launched
    import torch
    if not torch.cuda.is_available():
        assert lib.awq_selftest_wait_timeout(1_000_000, None) == DEVICE


def test_binding_raises_loudly_without_library(tmp_path):
    from w4a16_weight_only_gb300 import _binding
    with pytest.raises(RuntimeError, match="missing"):
        _binding.load_library(str(tmp_path / "nope.so"))


def test_quantize_argument_checks_are_host_side(lib):
    q = lib.awq_quantize_rtn
    W = P(0x300000)  # 16-byte aligned fake device address
    assert q(W, 12, 64, 32, 0, A, A, B, None) == SHAPE       # N not a multiple of 8
    assert q(W, 8, 48, 12, 0, A, A, B, None) == SHAPE        # group size not a multiple of 8
    assert q(W, 8, 64, 24, 0, A, A, B, None) == SHAPE        # K % G != 0
    assert q(W, 8, 524288, 8, 0, A, A, B, None) == SHAPE     # more than 65535 groups
    assert q(W, 8, 64, 32, 2, A, A, B, None) == INVALID      # sym not 0/1
    assert q(W, 8, 0, 32, 0, A, A, B, None) == INVALID       # K == 0
    assert q(None, 8, 64, 32, 0, A, A, B, None) == INVALID
    assert q(P(0x300008), 8, 64, 32, 0, A, A, B, None) == MISALIGNED
    assert q(W, 0, 64, 32, 0, None, None, None, None) == 0   # N == 0: no launch
    import torch
    if not torch.cuda.is_available():
        assert q(W, 8, 64, 32, 1, A, A, B, None) == DEVICE


def test_grouped_argument_checks_are_host_side(lib):
    g = lib.awq_gemm_grouped
    # (x, qweight, qzeros, scales, bias, offsets, R, E, K, N, G, y, stream)
    assert g(A, A, A, A, None, A, 8, 0, 256, 256, 128, B, None) == INVALID       # E == 0
    assert g(A, A, A, A, None, A, 8, 5000, 256, 256, 128, B, None) == INVALID    # E too large
    assert g(A, A, A, A, None, A, 8, 2, 256, 12, 128, B, None) == SHAPE          # N % 8
    assert g(A, A, A, A, None, A, 600000, 2, 256, 256, 128, B, None) == SHAPE    # R / 8 + E > 65535
    assert g(A, A, A, A, None, None, 8, 2, 256, 256, 128, B, None) == INVALID    # null offsets
    assert g(A, A, A, A, None, ODD, 8, 2, 256, 256, 128, B, None) == MISALIGNED
    assert g(A, A, A, A, None, A, 8, 2, 96, 256, 32, B, None) == SHAPE           # outside the TMA contract
    assert g(None, None, None, None, None, None, 0, 2, 256, 256, 128, None, None) == 0  # R == 0



def test_w8_argument_checks_are_host_side(lib):
    import torch
    g = lib.awq_gemm_w8_ex
    # (x, qweight, qzeros, scales, bias, M, K, N, G, y, path, stream)
    assert g(A, A, A, A, None, 1, 256, 6, 128, B, 0, None) == SHAPE      # N % 4
    assert g(A, A, A, A, None, 1, 256, 12, 96, B, 0, None) == SHAPE     # K % G
    assert g(None, A, A, A, None, 1, 256, 12, 128, B, 0, None) == INVALID
    assert g(A, A, A, A, None, 1, 256, 12, 128, B, 9, None) == INVALID  # bad path
    assert g(A, A, A, A, None, 0, 256, 12, 128, B, 0, None) == 0        # M == 0: no launch
    d = lib.awq_dequant_w8
    assert d(A, A, A, 256, 6, 128, B, 0, None) == SHAPE
    assert d(A, A, A, 256, 12, 128, B, 5, None) == INVALID               # bad dtype
    assert d(A, A, A, 256, 0, 128, B, 0, None) == 0
    if not torch.cuda.is_available():
        assert g(A, A, A, A, None, 1, 256, 12, 128, B, 0, None) == DEVICE
        assert d(A, A, A, 256, 12, 128, B, 0, None) == DEVICE


def test_linear_layer_refuses_host_tensors_and_bad_widths(lib):
    import torch
    from w4a16_weight_only_gb300 import AwqLinear
    qw = torch.zeros((256, 32), dtype=torch.int32)
    qz = torch.zeros((2, 32), dtype=torch.int32)
    sc = torch.zeros((2, 256), dtype=torch.float16)
    with pytest.raises(ValueError):
        AwqLinear(qw, qz, sc, None, group_size=128)          # host tensors never reach a kernel
    with pytest.raises(ValueError):
        AwqLinear(qw, qz, sc, None, group_size=128, bits=5)


def test_select_path_ex_is_host_only(lib):
    sel = lib.awq_gemm_select_path_ex
    F16, BF16 = 0, 2
    assert sel(1, 4096, 4096, 128, A, A, A, A, None, B, F16, 4) == 1       # decode
    assert sel(1, 4096, 4096, 128, A, A, A, A, None, B, BF16, 4) == 1      # bf16 decode
    assert sel(1, 4096, 4096, 128, A, A, A, A, None, B, F16, 8) == 1       # 8-bit decode
    assert sel(1, 256, 40, 128, A, A, A, A, None, B, F16, 8) == 3          # N % 16 != 0: generic
    assert sel(1, 4096, 4096, 128, A, A, A, A, None, B, BF16, 8) == 0      # 8-bit bf16: invalid
    assert sel(1, 4096, 4096, 128, A, A, A, A, None, B, 1, 4) == 0         # f32 activations: invalid
    assert sel(1, 256, 12, 128, A, A, A, A, None, B, F16, 4) == 0          # N % 8 at 4 bits


def test_gemm_any_argument_checks_are_host_side(lib):
    import torch
    g = lib.awq_gemm_any
    F16, F32, BF16, AUTO = 0, 1, 2, 0
    # (x, qweight, qzeros, scales, bias, M, K, N, G, y, dtype, bits, path, flags, stream)
    assert g(A, A, A, A, None, 1, 256, 64, 128, B, F16, 4, AUTO, 2, None) == INVALID   # unknown flag
    assert g(A, A, A, A, None, 1, 256, 64, 128, B, F32, 4, AUTO, 0, None) == INVALID   # f32 activations
    assert g(A, A, A, A, None, 1, 256, 64, 128, B, F16, 6, AUTO, 0, None) == INVALID   # 6-bit codes
    assert g(A, A, A, A, None, 1, 256, 64, 128, B, BF16, 8, AUTO, 0, None) == INVALID  # 8-bit bf16
    assert g(A, A, A, A, None, 1, 256, 64, 128, B, F16, 4, 7, 1, None) == INVALID      # bad path
    assert g(A, A, A, A, None, 1, 256, 12, 128, B, F16, 4, AUTO, 1, None) == SHAPE     # N % 8 (4 bits)
    assert g(A, A, A, A, None, 0, 256, 64, 128, B, BF16, 4, AUTO, 1, None) == 0        # M == 0
    if not torch.cuda.is_available():
        assert g(A, A, A, A, None, 1, 256, 64, 128, B, F16, 4, AUTO, 1, None) == DEVICE
        assert g(A, A, A, A, None, 1, 256, 12, 128, B, F16, 8, AUTO, 1, None) == DEVICE    # N % 4 suffices at 8 bits


def test_packed_layout_argument_checks_are_host_side(lib):
    import ctypes
    import torch
    n = ctypes.c_size_t(0)
    assert lib.awq_repack_size(8192, 28672, 128, ctypes.byref(n)) == 0
    assert n.value == 224 * 128 * 4608
    assert lib.awq_repack_size(128, 136, -1, ctypes.byref(n)) == 0 and n.value == 2 * 2 * 4608
    assert lib.awq_repack_size(96, 64, 32, ctypes.byref(n)) == SHAPE     # K % 64
    assert lib.awq_repack_size(256, 64, 32, ctypes.byref(n)) == SHAPE    # G % 64
    assert lib.awq_repack_size(256, 12, 128, ctypes.byref(n)) == SHAPE   # N % 8
    assert lib.awq_repack_size(256, 64, 128, None) == INVALID
    r = lib.awq_repack
    # (qweight, qzeros, scales, K, N, G, packed, stream)
    assert r(A, A, A, 256, 64, 128, None, None) == INVALID
    assert r(A, A, A, 256, 64, 32, B, None) == SHAPE
    assert r(A, A, A, 256, 0, 128, B, None) == 0                         # N == 0: no launch
    assert r(A, A, A, 256, 64, 128, P(0x200008), None) == MISALIGNED            # packed 16-byte aligned
    g = lib.awq_gemm_packed
    # (x, packed, bias, M, K, N, G, y, stream)
    assert g(A, B, None, 4, 96, 64, 32, B, None) == SHAPE
    assert g(None, B, None, 4, 256, 64, 128, B, None) == INVALID
    assert g(P(0x100002), B, None, 4, 256, 64, 128, B, None) == MISALIGNED      # x 16-byte aligned
    assert g(A, B, None, 0, 256, 64, 128, B, None) == 0                  # M == 0: no launch
    assert g(A, B, None, -1, 256, 64, 128, B, None) == INVALID
    w = lib.awq_gemm_packed_ws
    # (x, packed, bias, M, K, N, G, y, workspace, workspace_bytes, stream)
    assert w(A, B, None, 4, 96, 64, 32, B, A, 1 << 20, None) == SHAPE
    assert w(A, B, None, 4, 256, 64, 128, B, P(0x100010), 1 << 20, None) == MISALIGNED  # 256-byte aligned
    assert w(A, B, None, 0, 256, 64, 128, B, A, 1 << 20, None) == 0         # M == 0: no launch
    assert w(None, B, None, 4, 256, 64, 128, B, A, 1 << 20, None) == INVALID
    assert lib.awq_gemm_packed_workspace_size(None) == INVALID
    # 8-bit tile-packed layout: 8704-byte blocks, N % 4
    assert lib.awq_repack_w8_size(8192, 28672, 128, ctypes.byref(n)) == 0 and n.value == 224 * 128 * 8704
    assert lib.awq_repack_w8_size(128, 260, -1, ctypes.byref(n)) == 0 and n.value == 3 * 2 * 8704
    assert lib.awq_repack_w8_size(256, 6, 128, ctypes.byref(n)) == SHAPE    # N % 4
    assert lib.awq_repack_w8_size(96, 64, 32, ctypes.byref(n)) == SHAPE     # K % 64
    r8 = lib.awq_repack_w8
    assert r8(A, A, A, 256, 64, 128, None, None) == INVALID
    assert r8(A, A, A, 256, 64, 128, P(0x200008), None) == MISALIGNED
    assert r8(A, A, A, 256, 0, 128, B, None) == 0
    g8 = lib.awq_gemm_packed_w8
    # (x, packed, bias, M, K, N, G, y, workspace, workspace_bytes, stream)
    assert g8(A, B, None, 4, 256, 6, 128, B, None, 0, None) == SHAPE
    assert g8(P(0x100002), B, None, 4, 256, 260, 128, B, None, 0, None) == MISALIGNED
    assert g8(A, B, None, 0, 256, 260, 128, B, None, 0, None) == 0
    e = lib.awq_gemm_packed_ex
    assert e(A, B, None, 4, 256, 64, 128, B, 1, None, 0, None) == INVALID   # fp32 activations
    gp = lib.awq_gemm_packed_grouped
    # (x, packed, bias, offsets, R, E, K, N, G, y, dtype, stream)
    assert gp(A, B, None, A, 8, 0, 256, 64, 128, B, 0, None) == INVALID          # E >= 1
    assert gp(A, B, None, A, 8, 257, 256, 64, 128, B, 0, None) == INVALID        # E <= 256
    assert gp(A, B, None, A, 8, 4, 96, 64, 32, B, 0, None) == SHAPE              # K % 64
    assert gp(A, B, None, A, 0, 4, 256, 64, 128, B, 0, None) == 0                # R == 0: no launch
    assert gp(A, B, None, A, 8, 4, 256, 64, 128, B, 1, None) == INVALID          # fp32
    z = lib.awq_gemm_packed_noalloc
    # (x, packed, bias, M, K, N, G, y, stream): the packed linear's checks, before any scratch use
    assert z(A, B, None, 4, 96, 64, 32, B, None) == SHAPE
    assert z(P(0x100002), B, None, 4, 256, 64, 128, B, None) == MISALIGNED
    assert z(A, B, None, 0, 256, 64, 128, B, None) == 0                   # M == 0: nothing to do
    if not torch.cuda.is_available():
        assert g(A, B, None, 4, 256, 64, 128, B, None) == DEVICE
        assert r(A, A, A, 256, 64, 128, B, None) == DEVICE
        assert w(A, B, None, 4, 256, 64, 128, B, A, 1 << 20, None) == DEVICE
        assert w(A, B, None, 4, 256, 64, 128, B, None, 0, None) == DEVICE    # no workspace: plain plan
        assert lib.awq_gemm_packed_workspace_size(ctypes.byref(n)) == DEVICE
        assert z(A, B, None, 4, 256, 64, 128, B, None) == DEVICE
        assert g8(A, B, None, 4, 256, 260, 128, B, None, 0, None) == DEVICE
        assert gp(A, B, None, A, 8, 4, 256, 64, 128, B, 2, None) == DEVICE
        assert r8(A, A, A, 256, 64, 128, B, None) == DEVICE
        assert e(A, B, None, 4, 256, 64, 128, B, 2, None, 0, None) == DEVICE
