"""ctypes binding over libawq_gb300.so (include/awq.h).  Argument marshalling only:
every step of the computation runs in the library's CUDA kernels.  There is no CPU or
PyTorch fallback: if the library is missing or the device is not sm_103a, calls raise."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libawq_gb300.so")

AWQ_OK = 0
STATUS_NAMES = {0: "AWQ_OK", 1: "AWQ_ERR_INVALID_ARGUMENT", 2: "AWQ_ERR_UNSUPPORTED_SHAPE",
                3: "AWQ_ERR_MISALIGNED", 4: "AWQ_ERR_UNSUPPORTED_DEVICE", 5: "AWQ_ERR_CUDA",
                6: "AWQ_ERR_TIMEOUT"}
PATHS = {"auto": 0, "decode": 1, "prefill": 2, "generic": 3}
PATH_NAMES = {v: k for k, v in PATHS.items()}
DTYPE_F16, DTYPE_F32, DTYPE_BF16 = 0, 1, 2

# Every entry point of include/awq.h: name -> (restype, argtypes)
_i64, _vp, _i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "awq_runtime_available": (_i32, []),
    "awq_last_error": (ctypes.c_char_p, []),
    "awq_status_string": (ctypes.c_char_p, [_i32]),
    "awq_dequant": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_gemm": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_gemm_select_path": (_i32, [_i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "awq_gemm_select_path_ex": (_i32, [_i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32]),
    "awq_device_status": (_i32, [_vp]),
    "awq_selftest_wait_timeout": (_i32, [ctypes.c_uint64, _vp]),
    "awq_quantize_rtn": (_i32, [_vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp]),
    "awq_gemm_bf16": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_bf16_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_dequant_bf16": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_gemm_grouped": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_w8": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_w8_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_dequant_w8": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_gemm_any": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _i32, _i32, _i32,
                            ctypes.c_uint32, _vp]),
    "awq_repack_size": (_i32, [_i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "awq_repack": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_packed": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_packed_workspace_size": (_i32, [ctypes.POINTER(ctypes.c_size_t)]),
    "awq_gemm_packed_ws": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, ctypes.c_size_t, _vp]),
    "awq_gemm_packed_noalloc": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_packed_ex": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _i32, _vp, ctypes.c_size_t, _vp]),
    "awq_repack_w8_size": (_i32, [_i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "awq_gemm_packed_grouped": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp, _i32, _vp]),
    "awq_repack_w8": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "awq_gemm_packed_w8": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, ctypes.c_size_t, _vp]),
}
GEMM_STATIC_WEIGHTS = 1

_lib = None
_lock = threading.Lock()


class AwqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libawq_gb300.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it first (python -m w4a16_weight_only_gb300.build or "
                "__graft_entry__.build()); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    return load_library().awq_last_error().decode()


def runtime_available() -> bool:
    return bool(load_library().awq_runtime_available())


def _check(status: int):
    if status != AWQ_OK:
        raise AwqError(status, last_error())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _cuda_index(t, name):
    d = t.get_device()
    if d < 0:
        raise ValueError(f"{name} must be a CUDA tensor")
    return d


def _need(t, name, dtype, shape, device):
    """Cheap per-call checks (this runs on every call): dtype, exact shape, row-major
    layout, and the same CUDA device as the first operand (a host tensor's address must
    never reach a kernel)."""
    if t.dtype is not dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.shape != shape:
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    if t.get_device() != device and t.numel():
        raise ValueError(f"{name} is on {t.device}, expected device {device}")


def _groups(K, group_size):
    G = K if group_size == -1 else group_size
    return K // G if (G > 0 and K % G == 0) else 1


def awq_gemm(x, qweight, qzeros, scales, bias=None, group_size=128, out=None, path="auto",
             stream=None, static_weights=False):
    """y = x @ dequant(qweight, qzeros, scales) (+ bias) via the library's awq_gemm_any
    (fp16 or bf16 activations, 4-bit codes).

    x fp16 or bf16 [M, K] (leading dims are flattened), qweight int32 [K, N/8], qzeros int32
    [K/G, N/8], scales [K/G, N] and bias [N] (or None) of x's dtype.  Returns [..., N] of
    x's dtype.  static_weights=True passes AWQ_GEMM_STATIC_WEIGHTS: the weights must then
    be complete before the kernel launched just before this call on the stream.
    """
    lib = load_library()
    lead = x.shape[:-1]
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    N = qweight.shape[1] * 8
    dev = _cuda_index(x, "x")
    dt = x.dtype if x.dtype in (torch.float16, torch.bfloat16) else torch.float16
    _need(x2, "x", dt, (M, K), dev)
    _need(qweight, "qweight", torch.int32, (K, N // 8), dev)
    ng = _groups(K, group_size)
    _need(qzeros, "qzeros", torch.int32, (ng, N // 8), dev)
    _need(scales, "scales", dt, (ng, N), dev)
    if bias is not None:
        _need(bias, "bias", dt, (N,), dev)
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=dev)
    else:
        _need(out, "out", dt, (M, N), dev)
    st = lib.awq_gemm_any(_ptr(x2), _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(bias),
                          M, K, N, group_size, _ptr(out),
                          DTYPE_BF16 if dt == torch.bfloat16 else DTYPE_F16, 4, PATHS[path],
                          GEMM_STATIC_WEIGHTS if static_weights else 0, _stream(stream))
    _check(st)
    return out.reshape(*lead, N)


# Rows from which a layer built with packed=True runs awq_gemm_packed (its tile-packed copy)
# rather than awq_gemm on the checkpoint layout: on GB300 the packed kernels were faster from
# 128 rows on every 7B / 70B linear (e.g. 25.0 against 34.4 us at 128 x 4096 x 11008, 80.5
# against 115 us at 128 x 8192 x 28672), mixed at 64 rows, slower at 32 and below.
PACKED_MIN_ROWS = 128


class AwqLinear:
    """An AWQ linear layer whose weights are validated once: ``layer(x)`` runs
    ``awq_gemm_any`` (fp16 or bf16 activations, 4- or 8-bit codes) with only x and out
    checked per call.

    packed=True (4-bit codes with fp16 or bf16, or 8-bit codes with fp16; K % 64 == 0, group
    size % 64 == 0) also keeps a tile-packed copy of the weights, written once by awq_repack at
    construction (a device allocation of awq_repack_size bytes, about the size of the packed
    weights), and runs calls of at least ``packed_min_rows`` rows through awq_gemm_packed_ex
    (8 bits: awq_gemm_packed_w8) with the stream's workspace; smaller calls keep the
    checkpoint layout.

    qweight int32 [K, N/8] (4 bits) or [K, N/4] (8 bits), qzeros int32 [K/G, N/8 or N/4],
    scales fp16 or bf16 [K/G, N] (it sets the activation dtype; 8 bits: fp16), bias [N] of
    the same dtype or None, all contiguous on one CUDA device.  The layer keeps references
    to the tensors and reads them in place on every call.

    static_weights=True (the default: weights loaded once, as at model load) passes
    AWQ_GEMM_STATIC_WEIGHTS, so a small-M call starts streaming the weights under the tail
    of the kernel launched just before it.  The weights must then be complete before that
    kernel is launched: a kernel that updates them in place must not be the one launched
    immediately before a call on the same stream (use static_weights=False for such
    layers)."""

    __slots__ = ("K", "N", "group_size", "bits", "dtype", "device", "_w", "_path",
                 "_tensors", "_dt", "_flags", "packed", "packed_min_rows")

    def __init__(self, qweight, qzeros, scales, bias=None, group_size=128, bits=4, path="auto",
                 static_weights=True, packed=False, packed_min_rows=PACKED_MIN_ROWS):
        lib = load_library()
        if bits not in (4, 8):
            raise ValueError("bits must be 4 or 8")
        if qweight.dim() != 2 or qweight.shape[0] == 0:
            raise ValueError("qweight must be a non-empty [K, N / (32 / bits)] int32 matrix")
        per = 32 // bits
        K, C = qweight.shape
        N = C * per
        dev = _cuda_index(qweight, "qweight")
        dt = scales.dtype
        if dt not in (torch.float16, torch.bfloat16) or (bits == 8 and dt is not torch.float16):
            raise TypeError("scales must be float16 (or bfloat16 with 4-bit codes)")
        _need(qweight, "qweight", torch.int32, (K, C), dev)
        ng = _groups(K, group_size)
        _need(qzeros, "qzeros", torch.int32, (ng, C), dev)
        _need(scales, "scales", dt, (ng, N), dev)
        if bias is not None:
            _need(bias, "bias", dt, (N,), dev)
        self.K, self.N, self.group_size, self.bits = K, N, group_size, bits
        self.dtype, self.device = dt, dev
        self._dt = DTYPE_BF16 if dt is torch.bfloat16 else DTYPE_F16
        self._flags = GEMM_STATIC_WEIGHTS if static_weights else 0
        self._w = (qweight.data_ptr(), qzeros.data_ptr(), scales.data_ptr(), _ptr(bias))
        self.packed = None
        self.packed_min_rows = int(packed_min_rows)
        if packed:
            self.packed = awq_repack(qweight, qzeros, scales, group_size, bits=bits)
        self._path = PATHS[path]
        self._tensors = (qweight, qzeros, scales, bias)

    def __call__(self, x, out=None, stream=None):
        """y [..., N] = x [..., K] @ W (+ bias) on ``stream`` (default: the current stream)."""
        K, N, dt = self.K, self.N, self.dtype
        if x.dtype is not dt:
            raise TypeError(f"x must be {dt}, got {x.dtype}")
        if x.get_device() != self.device:
            raise ValueError(f"x is on {x.device}, expected CUDA device {self.device}")
        shape = x.shape
        if shape[-1] != K or not x.is_contiguous():
            raise ValueError(f"x must be a contiguous [..., {K}] tensor, got {tuple(shape)}")
        M = x.numel() // K
        if out is None:
            out = torch.empty(shape[:-1] + (N,), dtype=dt, device=x.device)
        elif (out.dtype is not dt or out.get_device() != self.device or out.shape[-1] != N
              or out.numel() != M * N or not out.is_contiguous()):
            raise ValueError(f"out must be a contiguous {dt} [..., {N}] tensor of {M} rows "
                             f"on device {self.device}")
        w = self._w
        if self.packed is not None and M >= self.packed_min_rows:
            sh = ((stream if isinstance(stream, int) else stream.cuda_stream)
                  if stream is not None else torch.cuda.current_stream().cuda_stream)
            ws = packed_workspace(self.device, sh)
            if self.bits == 8:
                st = _lib.awq_gemm_packed_w8(x.data_ptr(), self.packed.data_ptr(), w[3], M, K, N,
                                             self.group_size, out.data_ptr(), ws.data_ptr(), ws.numel(), sh)
            else:
                st = _lib.awq_gemm_packed_ex(x.data_ptr(), self.packed.data_ptr(), w[3], M, K, N,
                                             self.group_size, out.data_ptr(), self._dt, ws.data_ptr(),
                                             ws.numel(), sh)
            if st != AWQ_OK:
                raise AwqError(st, last_error())
            return out
        st = _lib.awq_gemm_any(x.data_ptr(), w[0], w[1], w[2], w[3], M, K, N, self.group_size,
                               out.data_ptr(), self._dt, self.bits, self._path, self._flags,
                               (stream if isinstance(stream, int) else stream.cuda_stream)
                               if stream is not None else torch.cuda.current_stream().cuda_stream)
        if st != AWQ_OK:
            raise AwqError(st, last_error())
        return out


def awq_gemm_w8(x, qweight, qzeros, scales, bias=None, group_size=128, out=None, path="auto",
                stream=None, static_weights=False):
    """y = x @ dequant8(qweight, qzeros, scales) (+ bias) via awq_gemm_w8: 8-bit codes,
    qweight int32 [K, N/4], qzeros int32 [K/G, N/4], scales fp16 [K/G, N]; x fp16 [M, K]."""
    lib = load_library()
    lead = x.shape[:-1]
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    N = qweight.shape[1] * 4
    dev = _cuda_index(x, "x")
    _need(x2, "x", torch.float16, (M, K), dev)
    _need(qweight, "qweight", torch.int32, (K, N // 4), dev)
    ng = _groups(K, group_size)
    _need(qzeros, "qzeros", torch.int32, (ng, N // 4), dev)
    _need(scales, "scales", torch.float16, (ng, N), dev)
    if bias is not None:
        _need(bias, "bias", torch.float16, (N,), dev)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _need(out, "out", torch.float16, (M, N), dev)
    st = lib.awq_gemm_any(_ptr(x2), _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(bias),
                          M, K, N, group_size, _ptr(out), DTYPE_F16, 8, PATHS[path],
                          GEMM_STATIC_WEIGHTS if static_weights else 0, _stream(stream))
    _check(st)
    return out.reshape(*lead, N)


def awq_dequant_w8(qweight, qzeros, scales, group_size=128, out_dtype=torch.float16, stream=None):
    """Dense W [K, N] from 8-bit codes via awq_dequant_w8 (fp16 or fp32)."""
    lib = load_library()
    K, C = qweight.shape
    N = 4 * C
    dev = _cuda_index(qweight, "qweight")
    _need(qweight, "qweight", torch.int32, (K, C), dev)
    ng = _groups(K, group_size)
    _need(qzeros, "qzeros", torch.int32, (ng, C), dev)
    _need(scales, "scales", torch.float16, (ng, N), dev)
    if out_dtype not in (torch.float16, torch.float32):
        raise TypeError("out_dtype must be torch.float16 or torch.float32")
    out = torch.empty((K, N), dtype=out_dtype, device=dev)
    st = lib.awq_dequant_w8(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group_size, _ptr(out),
                            DTYPE_F32 if out_dtype == torch.float32 else DTYPE_F16, _stream(stream))
    _check(st)
    return out


def awq_gemm_grouped(x, qweight, qzeros, scales, offsets, bias=None, group_size=128, out=None,
                     stream=None):
    """Grouped (mixture-of-experts) linear via the library's awq_gemm_grouped: rows
    offsets[e]..offsets[e+1]-1 of x fp16 [R, K] through expert e (qweight int32 [E, K, N/8],
    qzeros int32 [E, K/G, N/8], scales fp16 [E, K/G, N], bias fp16 [E, N] or None);
    offsets int32 [E+1] on the device.  Returns fp16 [R, N]."""
    lib = load_library()
    R, K = x.shape
    E, _, C = qweight.shape
    N = 8 * C
    dev = _cuda_index(x, "x")
    _need(x, "x", torch.float16, (R, K), dev)
    _need(qweight, "qweight", torch.int32, (E, K, C), dev)
    ng = _groups(K, group_size)
    _need(qzeros, "qzeros", torch.int32, (E, ng, C), dev)
    _need(scales, "scales", torch.float16, (E, ng, N), dev)
    _need(offsets, "offsets", torch.int32, (E + 1,), dev)
    if bias is not None:
        _need(bias, "bias", torch.float16, (E, N), dev)
    if out is None:
        out = torch.empty((R, N), dtype=torch.float16, device=dev)
    else:
        _need(out, "out", torch.float16, (R, N), dev)
    st = lib.awq_gemm_grouped(_ptr(x), _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(bias),
                              _ptr(offsets), R, E, K, N, group_size, _ptr(out), _stream(stream))
    _check(st)
    return out


def awq_dequant(qweight, qzeros, scales, group_size=128, out_dtype=torch.float16, out=None,
                stream=None):
    """Dense W [K, N] = (code - zero) * scale via the library's awq_dequant (fp16 scales;
    out fp16 or fp32) or awq_dequant_bf16 (bf16 scales; out bf16 or fp32)."""
    lib = load_library()
    K, C = qweight.shape
    N = 8 * C
    dev = _cuda_index(qweight, "qweight")
    _need(qweight, "qweight", torch.int32, (K, C), dev)
    ng = _groups(K, group_size)
    _need(qzeros, "qzeros", torch.int32, (ng, C), dev)
    bf = scales.dtype == torch.bfloat16
    _need(scales, "scales", torch.bfloat16 if bf else torch.float16, (ng, N), dev)
    half = torch.bfloat16 if bf else torch.float16
    if out_dtype == torch.float16 and bf:
        out_dtype = torch.bfloat16
    if out_dtype not in (half, torch.float32):
        raise TypeError(f"out_dtype must be {half} or torch.float32")
    if out is None:
        out = torch.empty((K, N), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out_dtype, (K, N), dev)
    if bf:
        st = lib.awq_dequant_bf16(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group_size,
                                  _ptr(out), DTYPE_F32 if out_dtype == torch.float32 else DTYPE_BF16,
                                  _stream(stream))
    else:
        st = lib.awq_dequant(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group_size,
                             _ptr(out), DTYPE_F32 if out_dtype == torch.float32 else DTYPE_F16,
                             _stream(stream))
    _check(st)
    return out


def awq_quantize_rtn(w, group_size=128, sym=False, out=None, stream=None):
    """Round-to-nearest 4-bit group quantization of an fp16 linear weight w [N, K]
    (out_features x in_features) via the library's awq_quantize_rtn.  Returns
    (qweight int32 [K, N/8], qzeros int32 [K/G, N/8], scales fp16 [K/G, N]), written into
    `out` (a tuple of those three tensors) when given."""
    lib = load_library()
    N, K = w.shape
    dev = _cuda_index(w, "w")
    _need(w, "w", torch.float16, (N, K), dev)
    ng = _groups(K, group_size)
    if out is None:
        qweight = torch.empty((K, N // 8), dtype=torch.int32, device=dev)
        qzeros = torch.empty((ng, N // 8), dtype=torch.int32, device=dev)
        scales = torch.empty((ng, N), dtype=torch.float16, device=dev)
    else:
        qweight, qzeros, scales = out
        _need(qweight, "qweight", torch.int32, (K, N // 8), dev)
        _need(qzeros, "qzeros", torch.int32, (ng, N // 8), dev)
        _need(scales, "scales", torch.float16, (ng, N), dev)
    st = lib.awq_quantize_rtn(_ptr(w), N, K, group_size, 1 if sym else 0, _ptr(qweight),
                              _ptr(qzeros), _ptr(scales), _stream(stream))
    _check(st)
    return qweight, qzeros, scales


def select_path(x, qweight, qzeros, scales, bias=None, group_size=128, out=None, bits=4) -> str:
    """The kernel family awq_gemm (bits=4; bf16 when x is bfloat16) or awq_gemm_w8 (bits=8)
    would run for these tensors: "decode", "prefill", "generic", or "auto" if invalid."""
    lib = load_library()
    M, K = x.reshape(-1, x.shape[-1]).shape
    N = qweight.shape[1] * (32 // bits)
    dt = DTYPE_BF16 if x.dtype == torch.bfloat16 else DTYPE_F16
    r = lib.awq_gemm_select_path_ex(M, K, N, group_size, _ptr(x), _ptr(qweight), _ptr(qzeros),
                                    _ptr(scales), _ptr(bias), _ptr(out) if out is not None else _ptr(x),
                                    dt, bits)
    return PATH_NAMES.get(r, "auto")


def device_status(stream=None):
    _check(load_library().awq_device_status(_stream(stream)))


def selftest_wait_timeout(limit_ns=2_000_000, stream=None):
    """Launch the bounded-wait self test (awq.h); the next device_status() raises AwqError."""
    _check(load_library().awq_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def awq_repack_size(K, N, group_size=128, bits=4) -> int:
    """Bytes of the tile-packed layout of a [K, N] linear of 4- or 8-bit codes (host only)."""
    n = ctypes.c_size_t(0)
    lib = load_library()
    f = lib.awq_repack_w8_size if bits == 8 else lib.awq_repack_size
    _check(f(K, N, group_size, ctypes.byref(n)))
    return int(n.value)


def awq_repack(qweight, qzeros, scales, group_size=128, out=None, stream=None, bits=4):
    """One-off conversion of checkpoint-layout weights into the tile-packed layout via the
    library's awq_repack (bits=8: awq_repack_w8, fp16 scales).  Returns (or fills) an int32
    device tensor of awq_repack_size(K, N, group_size, bits) / 4 words."""
    lib = load_library()
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    K, C = qweight.shape
    N = (32 // bits) * C
    dev = _cuda_index(qweight, "qweight")
    _need(qweight, "qweight", torch.int32, (K, C), dev)
    ng = _groups(K, group_size)
    _need(qzeros, "qzeros", torch.int32, (ng, C), dev)
    if scales.dtype not in (torch.float16, torch.bfloat16) or (bits == 8 and scales.dtype is not torch.float16):
        raise TypeError("scales must be float16 or bfloat16 (their 16-bit words are copied; 8 bits: float16)")
    _need(scales, "scales", scales.dtype, (ng, N), dev)
    words = awq_repack_size(K, N, group_size, bits) // 4
    if out is None:
        out = torch.empty((words,), dtype=torch.int32, device=dev)
    else:
        _need(out, "out", torch.int32, (words,), dev)
    f = lib.awq_repack_w8 if bits == 8 else lib.awq_repack
    _check(f(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group_size, _ptr(out), _stream(stream)))
    return out


def awq_gemm_packed_workspace_size() -> int:
    """Bytes of workspace awq_gemm_packed_ws needs on the current device."""
    n = ctypes.c_size_t(0)
    _check(load_library().awq_gemm_packed_workspace_size(ctypes.byref(n)))
    return int(n.value)


_workspaces = {}


def packed_workspace(device, stream_handle):
    """The zero-filled uint8 workspace that packed calls on (device, stream) share (calls on
    one stream never overlap).  Allocated by PyTorch on first use: make the first packed call
    on a stream outside CUDA graph capture."""
    key = (int(device), int(stream_handle))
    ws = _workspaces.get(key)
    if ws is None:
        with torch.cuda.device(int(device)):
            ws = torch.zeros((awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device=int(device))
        _workspaces[key] = ws
    return ws


def awq_gemm_packed(x, packed, bias, K, N, group_size=128, out=None, stream=None, workspace=None, bits=4):
    """y = x @ W (+ bias) with W in the tile-packed layout (awq_repack's output) via the
    library's awq_gemm_packed; x fp16 [..., K] (leading dims flattened), bias fp16 [N] or
    None.  Returns [..., N] in x's dtype.  workspace: a zero-filled uint8 device tensor of at
    least awq_gemm_packed_workspace_size() bytes, or "auto" for the (device, stream) one: the
    call then goes through awq_gemm_packed_ws (stream-K on shapes that fill the SMs poorly).
    bfloat16 x (packed weights written from bfloat16 scales) goes through awq_gemm_packed_ex;
    bits=8 (packed weights from awq_repack(..., bits=8), float16 x) through awq_gemm_packed_w8."""
    lib = load_library()
    lead = x.shape[:-1]
    if x.shape[-1] != K:
        raise ValueError(f"x must be [..., {K}], got {tuple(x.shape)}")
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    dev = _cuda_index(x, "x")
    dt = x.dtype
    if dt not in (torch.float16, torch.bfloat16):
        raise TypeError("x must be float16 or bfloat16")
    _need(x2, "x", dt, (M, K), dev)
    if bits == 8 and dt is not torch.float16:
        raise TypeError("8-bit codes take float16 activations")
    _need(packed, "packed", torch.int32, (awq_repack_size(K, N, group_size, bits) // 4,), dev)
    if bias is not None:
        _need(bias, "bias", dt, (N,), dev)
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=dev)
    else:
        _need(out, "out", dt, (M, N), dev)
    sh = _stream(stream)
    if bits == 8:
        if isinstance(workspace, str) and workspace == "auto":
            workspace = packed_workspace(dev, sh.value or 0)
        ws, wsb = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel())
        _check(lib.awq_gemm_packed_w8(_ptr(x2), _ptr(packed), _ptr(bias), M, K, N, group_size, _ptr(out),
                                      ws, wsb, sh))
    elif dt is torch.bfloat16:  # awq_gemm_packed_ex (its workspace, if any, as below)
        if isinstance(workspace, str) and workspace == "auto":
            workspace = packed_workspace(dev, sh.value or 0)
        ws, wsb = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel())
        _check(lib.awq_gemm_packed_ex(_ptr(x2), _ptr(packed), _ptr(bias), M, K, N, group_size, _ptr(out),
                                      DTYPE_BF16, ws, wsb, sh))
    elif workspace is None:
        _check(lib.awq_gemm_packed(_ptr(x2), _ptr(packed), _ptr(bias), M, K, N, group_size, _ptr(out), sh))
    else:
        if isinstance(workspace, str) and workspace == "auto":
            workspace = packed_workspace(dev, sh.value or 0)
        if workspace.dtype is not torch.uint8 or workspace.get_device() != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 tensor on x's device")
        _check(lib.awq_gemm_packed_ws(_ptr(x2), _ptr(packed), _ptr(bias), M, K, N, group_size, _ptr(out),
                                      workspace.data_ptr(), workspace.numel(), sh))
    return out.reshape(*lead, N)


def awq_gemm_packed_noalloc(x, packed, bias, K, N, group_size=128, out=None, stream=None):
    """awq_gemm_packed through the library's awq_gemm_packed_noalloc: the stream-K workspace is
    the library's fixed device scratch, so the C call allocates nothing (pass ``out`` to keep
    this wrapper from allocating y).  Calls that overlap in time share that scratch and race."""
    lib = load_library()
    lead = x.shape[:-1]
    if x.shape[-1] != K:
        raise ValueError(f"x must be [..., {K}], got {tuple(x.shape)}")
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    dev = _cuda_index(x, "x")
    _need(x2, "x", torch.float16, (M, K), dev)
    _need(packed, "packed", torch.int32, (awq_repack_size(K, N, group_size) // 4,), dev)
    if bias is not None:
        _need(bias, "bias", torch.float16, (N,), dev)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=dev)
    else:
        _need(out, "out", torch.float16, (M, N), dev)
    _check(lib.awq_gemm_packed_noalloc(_ptr(x2), _ptr(packed), _ptr(bias), M, K, N, group_size, _ptr(out),
                                       _stream(stream)))
    return out.reshape(*lead, N)


def awq_repack_experts(qweight, qzeros, scales, group_size=128, stream=None):
    """E experts' 4-bit weights (qweight int32 [E, K, N/8], qzeros [E, K/G, N/8], fp16 or bf16
    scales [E, K/G, N]) into one int32 device tensor of E stacked tile-packed layouts, expert e's at
    word e * awq_repack_size(K, N, group_size) / 4 (one awq_repack launch per expert)."""
    E, K, C = qweight.shape
    N = 8 * C
    words = awq_repack_size(K, N, group_size) // 4
    out = torch.empty((E * words,), dtype=torch.int32, device=qweight.device)
    for e in range(E):
        awq_repack(qweight[e], qzeros[e], scales[e], group_size, out=out[e * words:(e + 1) * words],
                   stream=stream)
    return out


def awq_gemm_packed_grouped(x, packed, offsets, K, N, bias=None, group_size=128, out=None, stream=None):
    """Grouped (mixture-of-experts) linear on stacked tile-packed experts (awq_repack_experts)
    via the library's awq_gemm_packed_grouped: rows offsets[e]..offsets[e+1]-1 of x [R, K]
    through expert e; offsets int32 [E+1] on the device, bias [E, N] or None; x, bias and the
    result fp16, or bf16 (experts repacked from bf16 scales).  Returns [R, N] in x's dtype."""
    lib = load_library()
    R = x.shape[0]
    dev = _cuda_index(x, "x")
    dt = x.dtype
    if dt not in (torch.float16, torch.bfloat16):
        raise TypeError("x must be float16 or bfloat16")
    _need(x, "x", dt, (R, K), dev)
    words = awq_repack_size(K, N, group_size) // 4
    if packed.numel() % words != 0:
        raise ValueError("packed must hold whole experts' tile-packed layouts")
    E = packed.numel() // words
    _need(packed, "packed", torch.int32, (E * words,), dev)
    _need(offsets, "offsets", torch.int32, (E + 1,), dev)
    if bias is not None:
        _need(bias, "bias", dt, (E, N), dev)
    if out is None:
        out = torch.empty((R, N), dtype=dt, device=dev)
    else:
        _need(out, "out", dt, (R, N), dev)
    _check(lib.awq_gemm_packed_grouped(_ptr(x), _ptr(packed), _ptr(bias), _ptr(offsets), R, E, K, N,
                                       group_size, _ptr(out), DTYPE_BF16 if dt is torch.bfloat16 else DTYPE_F16,
                                       _stream(stream)))
    return out
