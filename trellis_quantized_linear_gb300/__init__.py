"""Python binding of libexl3.so, the sm_103a trellis-quantized linear layer.

The functions here carry the C ABI's names (include/exl3.h) and only marshal
arguments: tensors become device pointers, the stream defaults to torch's
current stream, and a non-zero status raises ``Exl3Error``. Every step of
the computation runs in the library's CUDA kernels; there is no fallback. If
``libexl3.so`` has not been built, loading it raises immediately.

With ``EXL3_BOUNDS_CHECKED=1`` in the environment the package builds and
loads ``libexl3_bounds.so`` instead: the same kernels with every access
checked against its launch's extents (a failed check records
EXL3_ERR_OUT_OF_BOUNDS in the device error word).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "Exl3Error", "build", "load", "EXL3_F16", "EXL3_F32", "EXL3_LAYOUT_KN", "EXL3_LAYOUT_NK",
    "EXL3_RECONSTRUCT_CHUNK_COLS", "EXL3_NOALLOC_SCRATCH_BYTES", "exl3_init", "exl3_status_string", "exl3_supported_bits",
    "exl3_aligned_logits_width", "exl3_decode_plan", "exl3_prefill_path", "exl3_linear_workspace_bytes_for",
    "exl3_linear_workspace_bytes", "exl3_workspace_init", "exl3_hadamard128", "exl3_reconstruct",
    "exl3_linear", "exl3_logits_masked", "exl3_get_device_status", "exl3_selftest_wait_timeout",
    "exl3_linear_decode_noalloc", "exl3_silu_mul", "exl3_reconstruct_rotated",
    "exl3_weight_rotated_workspace_bytes", "exl3_linear_weight_rotated", "exl3_bounds_checked",
    "exl3_selftest_bounds", "HEADER_SYMBOLS", "BOUNDS_CHECKED",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
BOUNDS_CHECKED = os.environ.get("EXL3_BOUNDS_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_PKG, "libexl3_bounds.so" if BOUNDS_CHECKED else "libexl3.so")

EXL3_F16 = 0
EXL3_F32 = 1
EXL3_LAYOUT_KN = 0
EXL3_LAYOUT_NK = 1
EXL3_RECONSTRUCT_CHUNK_COLS = 32768
EXL3_NOALLOC_SCRATCH_BYTES = 24 << 20

STATUS_NAMES = {
    0: "EXL3_OK", 1: "EXL3_ERR_INVALID_ARG", 2: "EXL3_ERR_ALIGNMENT", 3: "EXL3_ERR_UNSUPPORTED_BITS",
    4: "EXL3_ERR_WORKSPACE_TOO_SMALL", 5: "EXL3_ERR_NOT_INITIALIZED", 6: "EXL3_ERR_CUDA",
    7: "EXL3_ERR_DEVICE_TIMEOUT", 8: "EXL3_ERR_NOALLOC_TOO_LARGE", 9: "EXL3_ERR_OUT_OF_BOUNDS",
}

# Every function include/exl3.h declares.
HEADER_SYMBOLS = (
    "exl3_init", "exl3_status_string", "exl3_supported_bits", "exl3_aligned_logits_width",
    "exl3_decode_plan", "exl3_prefill_path", "exl3_linear_workspace_bytes_for", "exl3_linear_workspace_bytes",
    "exl3_workspace_init", "exl3_hadamard128", "exl3_reconstruct", "exl3_linear",
    "exl3_logits_masked", "exl3_get_device_status", "exl3_selftest_wait_timeout",
    "exl3_linear_decode_noalloc", "exl3_silu_mul", "exl3_reconstruct_rotated",
    "exl3_weight_rotated_workspace_bytes", "exl3_linear_weight_rotated", "exl3_bounds_checked",
    "exl3_selftest_bounds",
)


class Exl3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.name = STATUS_NAMES.get(self.status, f"status {status}")
        super().__init__(f"{where}: {self.name} ({_status_text(self.status)})")


_lib = None
_lock = threading.Lock()
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the library this process loads (libexl3.so, or libexl3_bounds.so
    under EXL3_BOUNDS_CHECKED=1) for sm_103a with nvcc (in-tree)."""
    from . import _build
    return _build.build(force=force, verbose=verbose, bounds_checked=BOUNDS_CHECKED)


def load():
    """Loads the library (LIB_PATH); raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with trellis_quantized_linear_gb300.build()")
        lib = ctypes.CDLL(LIB_PATH)
        sig = {
            "exl3_init": (ctypes.c_int, [ctypes.c_int]),
            "exl3_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "exl3_supported_bits": (ctypes.c_int, [ctypes.c_int]),
            "exl3_aligned_logits_width": (_i64, [_i64, _i64]),
            "exl3_decode_plan": (ctypes.c_int, [_i64, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                                ctypes.POINTER(ctypes.c_int)]),
            "exl3_prefill_path": (ctypes.c_int, [_i64, _i64, ctypes.c_int]),
            "exl3_linear_workspace_bytes_for": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.c_int, _i64, ctypes.c_int]),
            "exl3_linear_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.c_int, _i64]),
            "exl3_workspace_init": (ctypes.c_int, [_vp, ctypes.c_size_t, _vp]),
            "exl3_hadamard128": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _vp]),
            "exl3_reconstruct": (ctypes.c_int, [_vp, ctypes.c_int, _i64, _i64, _i64, _i64, _vp, ctypes.c_int, _vp]),
            "exl3_linear": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _i64, _i64, _vp, _vp, _vp,
                                           ctypes.c_int, _i64, _vp, ctypes.c_size_t, _vp]),
            "exl3_logits_masked": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp,
                                                  _vp, _vp, _i64, _vp, ctypes.c_size_t, _vp]),
            "exl3_get_device_status": (ctypes.c_int, [_vp]),
            "exl3_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, _vp]),
            "exl3_silu_mul": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp]),
            "exl3_linear_decode_noalloc": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _i64, _i64, _vp, _vp,
                                                          _vp, ctypes.c_int, _vp]),
            "exl3_reconstruct_rotated": (ctypes.c_int, [_vp, ctypes.c_int, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                                                        ctypes.c_int, _vp]),
            "exl3_weight_rotated_workspace_bytes": (ctypes.c_size_t, [_i64, _i64]),
            "exl3_linear_weight_rotated": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _i64, _i64, _vp, _vp,
                                                          _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]),
            "exl3_bounds_checked": (ctypes.c_int, []),
            "exl3_selftest_bounds": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), _vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _status_text(status: int) -> str:
    try:
        return load().exl3_status_string(int(status)).decode()
    except Exception:  # the library may be the thing that failed to load
        return STATUS_NAMES.get(int(status), "unknown")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise Exl3Error(status, where)


def _ptr(t):
    """Device pointer of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def exl3_init(device: int = 0) -> None:
    _check(load().exl3_init(int(device)), "exl3_init")


def exl3_status_string(status: int) -> str:
    return load().exl3_status_string(int(status)).decode()


def exl3_supported_bits(bits: int) -> bool:
    return bool(load().exl3_supported_bits(int(bits)))


def exl3_aligned_logits_width(n_decodable: int, n_stored: int) -> int:
    return int(load().exl3_aligned_logits_width(int(n_decodable), int(n_stored)))


def exl3_decode_plan(K: int, n_gemm: int, num_sms: int):
    s, g = ctypes.c_int(), ctypes.c_int()
    rc = load().exl3_decode_plan(int(K), int(n_gemm), int(num_sms), ctypes.byref(s), ctypes.byref(g))
    if rc != 0:
        raise ValueError("exl3_decode_plan: invalid geometry")
    return s.value, g.value


def exl3_prefill_path(M: int, n_gemm: int, num_sms: int) -> int:
    """1: a prefill-shaped call of M rows on an n_gemm-wide layer takes the
    fused prefill kernel; 0: reconstruct + GEMM; -1: invalid input."""
    return int(load().exl3_prefill_path(int(M), int(n_gemm), int(num_sms)))


def exl3_linear_workspace_bytes_for(M_max, K, n_gemm, bits, m_threshold, num_sms) -> int:
    return int(load().exl3_linear_workspace_bytes_for(int(M_max), int(K), int(n_gemm), int(bits),
                                                      int(m_threshold), int(num_sms)))


def exl3_linear_workspace_bytes(M_max, K, n_gemm, bits, m_threshold) -> int:
    return int(load().exl3_linear_workspace_bytes(int(M_max), int(K), int(n_gemm), int(bits), int(m_threshold)))


def exl3_workspace_init(workspace, workspace_bytes: int | None = None, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check(load().exl3_workspace_init(_ptr(workspace), int(nbytes), _stream(stream)), "exl3_workspace_init")


def exl3_hadamard128(x, y, pre_scale=None, rows: int | None = None, cols: int | None = None, stream=None) -> None:
    rows = x.shape[0] if rows is None else rows
    cols = x.shape[1] if cols is None else cols
    _check(load().exl3_hadamard128(_ptr(x), _ptr(y), _ptr(pre_scale), int(rows), int(cols), _stream(stream)),
           "exl3_hadamard128")


def exl3_reconstruct(trellis, bits: int, K: int, n_stored: int, n0: int, n_cols: int, w,
                     layout: int = EXL3_LAYOUT_KN, stream=None) -> None:
    _check(load().exl3_reconstruct(_ptr(trellis), int(bits), int(K), int(n_stored), int(n0), int(n_cols),
                                   _ptr(w), int(layout), _stream(stream)), "exl3_reconstruct")


def exl3_reconstruct_rotated(trellis, bits: int, K: int, n_stored: int, n0: int, n_cols: int, su, sv, w,
                             layout: int = EXL3_LAYOUT_KN, stream=None) -> None:
    _check(load().exl3_reconstruct_rotated(_ptr(trellis), int(bits), int(K), int(n_stored), int(n0), int(n_cols),
                                           _ptr(su), _ptr(sv), _ptr(w), int(layout), _stream(stream)),
           "exl3_reconstruct_rotated")


def exl3_weight_rotated_workspace_bytes(K: int, n_gemm: int) -> int:
    return int(load().exl3_weight_rotated_workspace_bytes(int(K), int(n_gemm)))


def exl3_linear_weight_rotated(x, M: int, K: int, trellis, bits: int, n_stored: int, n_gemm: int, su, sv, y,
                               y_dtype: int, workspace, workspace_bytes: int | None = None, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check(load().exl3_linear_weight_rotated(_ptr(x), int(M), int(K), _ptr(trellis), int(bits), int(n_stored),
                                             int(n_gemm), _ptr(su), _ptr(sv), _ptr(y), int(y_dtype),
                                             _ptr(workspace), int(nbytes), _stream(stream)),
           "exl3_linear_weight_rotated")


def exl3_linear(x, M: int, K: int, trellis, bits: int, n_stored: int, n_gemm: int, su, sv, y, y_dtype: int,
                m_threshold: int, workspace, workspace_bytes: int | None = None, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check(load().exl3_linear(_ptr(x), int(M), int(K), _ptr(trellis), int(bits), int(n_stored), int(n_gemm),
                              _ptr(su), _ptr(sv), _ptr(y), int(y_dtype), int(m_threshold), _ptr(workspace),
                              int(nbytes), _stream(stream)), "exl3_linear")


def exl3_logits_masked(x, M: int, K: int, trellis, bits: int, n_stored: int, n_gemm: int, n_decodable: int,
                       su, sv, logits, argmax, m_threshold: int, workspace, workspace_bytes: int | None = None,
                       stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check(load().exl3_logits_masked(_ptr(x), int(M), int(K), _ptr(trellis), int(bits), int(n_stored),
                                     int(n_gemm), int(n_decodable), _ptr(su), _ptr(sv), _ptr(logits),
                                     _ptr(argmax), int(m_threshold), _ptr(workspace), int(nbytes),
                                     _stream(stream)), "exl3_logits_masked")


def exl3_get_device_status(stream=None) -> int:
    """Synchronises the stream, reads and clears the device error word."""
    return int(load().exl3_get_device_status(_stream(stream)))


def exl3_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launches the bounded-wait self-test kernel (see include/exl3.h)."""
    _check(load().exl3_selftest_wait_timeout(int(limit_us), _stream(stream)), "exl3_selftest_wait_timeout")


def exl3_bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return load().exl3_bounds_checked() == 1


def exl3_selftest_bounds(stream=None) -> tuple[int, int]:
    """Runs the bounds-check reporting self-test (see include/exl3.h); returns
    (units that reported, units probed): (6, 6) in the bounds-checked build,
    (0, 0) in libexl3.so."""
    rep, tot = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().exl3_selftest_bounds(ctypes.byref(rep), ctypes.byref(tot), _stream(stream)), "exl3_selftest_bounds")
    return rep.value, tot.value


def exl3_linear_decode_noalloc(x, M: int, K: int, trellis, bits: int, n_stored: int, n_gemm: int, su, sv, y,
                               y_dtype: int, stream=None) -> None:
    """Decode-shaped linear layer that allocates nothing: its scratch is a
    fixed buffer of EXL3_NOALLOC_SCRATCH_BYTES (24 MiB) inside the library.
    Rows run in groups of 16 through the 16-row decode kernel."""
    _check(load().exl3_linear_decode_noalloc(_ptr(x), int(M), int(K), _ptr(trellis), int(bits), int(n_stored),
                                             int(n_gemm), _ptr(su), _ptr(sv), _ptr(y), int(y_dtype),
                                             _stream(stream)), "exl3_linear_decode_noalloc")


def exl3_silu_mul(gate, up, out, n: int | None = None, stream=None) -> None:
    """out = fp16(silu(gate) * up), the dense-MLP glue between projections."""
    n = gate.numel() if n is None else n
    _check(load().exl3_silu_mul(_ptr(gate), _ptr(up), _ptr(out), int(n), _stream(stream)), "exl3_silu_mul")
