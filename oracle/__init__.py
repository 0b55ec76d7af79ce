"""CPU oracle for the trellis-quantized linear layer (test infrastructure).

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package. The CUDA library never does: it shares no code
with ``oracle.c`` and must fail loudly when its own extension is missing.

The C source is compiled with gcc on first use (or by ``build()``) into
``oracle/liboracle.so``; these wrappers only marshal numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_float_to_half_rne.argtypes = [ctypes.c_float]
        lib.oracle_float_to_half_rne.restype = ctypes.c_uint16
        for name in ("oracle_lcg_raw", "oracle_lcg_masked"):
            getattr(lib, name).argtypes = [ctypes.c_uint32]
            getattr(lib, name).restype = ctypes.c_uint32
        lib.oracle_decode_state.argtypes = [ctypes.c_uint32]
        lib.oracle_decode_state.restype = ctypes.c_uint16
        for name in ("oracle_tile_states_walk", "oracle_tile_states_window", "oracle_decode_tile"):
            getattr(lib, name).argtypes = [_u16p, ctypes.c_int, _u16p]
            getattr(lib, name).restype = None
        lib.oracle_reconstruct.argtypes = [_u16p, ctypes.c_int, _i64, _i64, _i64, _i64, _u16p]
        lib.oracle_reconstruct.restype = None
        lib.oracle_reconstruct_rotated.argtypes = [_u16p, ctypes.c_int, _i64, _i64, _u16p, _u16p, _i64, _i64,
                                                   ctypes.c_int, _u16p]
        lib.oracle_reconstruct_rotated.restype = ctypes.c_int
        lib.oracle_hadamard128_f64.argtypes = [_f64p, _f64p, _i64]
        lib.oracle_hadamard128_f64.restype = None
        lib.oracle_hadamard128_f32.argtypes = [_f32p, _f32p, _i64]
        lib.oracle_hadamard128_f32.restype = None
        lib.oracle_input_rotation.argtypes = [_u16p, ctypes.c_void_p, _i64, _i64, _u16p]
        lib.oracle_input_rotation.restype = None
        lib.oracle_linear.argtypes = [_u16p, _i64, _i64, _u16p, ctypes.c_int, _i64, _u16p, _u16p,
                                      _i64, _i64, _f64p]
        lib.oracle_linear.restype = ctypes.c_int
        lib.oracle_mask_argmax.argtypes = [_f64p, _i64, _i64, _i64, _i32p, ctypes.c_int]
        lib.oracle_mask_argmax.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _bits16(a) -> np.ndarray:
    """View fp16 (or uint16) data as contiguous uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16/uint16, got {a.dtype}")
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def half_to_float(h: int) -> float:
    return float(_load().oracle_half_to_float(int(h)))


def float_to_half_rne(f: float) -> int:
    return int(_load().oracle_float_to_half_rne(float(f)))


def lcg_raw(state: int) -> int:
    return int(_load().oracle_lcg_raw(int(state)))


def lcg_masked(state: int) -> int:
    return int(_load().oracle_lcg_masked(int(state)))


def decode_state(state: int) -> int:
    """fp16 bits of the weight a 16-bit state decodes to."""
    return int(_load().oracle_decode_state(int(state)))


def decode_table() -> np.ndarray:
    """fp16 bits for all 65536 states (uint16[65536])."""
    lib = _load()
    return np.array([lib.oracle_decode_state(s) for s in range(65536)], dtype=np.uint16)


def tile_states_walk(words, bits: int) -> np.ndarray:
    out = np.zeros(256, np.uint16)
    _load().oracle_tile_states_walk(_bits16(words), int(bits), out)
    return out


def tile_states_window(words, bits: int) -> np.ndarray:
    out = np.zeros(256, np.uint16)
    _load().oracle_tile_states_window(_bits16(words), int(bits), out)
    return out


def decode_tile(words, bits: int) -> np.ndarray:
    """256 fp16 weights of one tile, row-major 16x16 (returned as float16)."""
    out = np.zeros(256, np.uint16)
    _load().oracle_decode_tile(_bits16(words), int(bits), out)
    return out.view(np.float16).reshape(16, 16)


def reconstruct(trellis, bits: int, K: int, n_stored: int, n0: int = 0, ncols: int | None = None) -> np.ndarray:
    """W[:, n0:n0+ncols] as float16 (K x ncols, row-major)."""
    if ncols is None:
        ncols = n_stored - n0
    out = np.zeros((K, ncols), np.uint16)
    _load().oracle_reconstruct(_bits16(trellis), int(bits), K, n_stored, n0, ncols, out)
    return out.view(np.float16)


def reconstruct_rotated(trellis, bits: int, K: int, n_stored: int, su, sv, n0: int = 0,
                        ncols: int | None = None, layout: int = 0) -> np.ndarray:
    """Columns [n0, n0+ncols) of the weight-side rotated weight
    W' = diag(su) . had_r_128(K) . W . had_r_128(N) . diag(sv) as float16,
    K x ncols (layout 0) or ncols x K (layout 1)."""
    if ncols is None:
        ncols = n_stored - n0
    shape = (K, ncols) if layout == 0 else (ncols, K)
    out = np.zeros(shape, np.uint16)
    rc = _load().oracle_reconstruct_rotated(_bits16(trellis), int(bits), K, n_stored, _bits16(su), _bits16(sv),
                                            n0, ncols, int(layout), out)
    if rc != 0:
        raise ValueError(f"oracle_reconstruct_rotated rejected its arguments (rc={rc})")
    return out.view(np.float16)


def matmul_f64(x, w) -> np.ndarray:
    """x . w in fp64 for fp16 x (M x K) and fp16 w (K x n): the weight-side
    variant's layer output from its rotated weight."""
    return np.asarray(x, np.float16).astype(np.float64) @ np.asarray(w, np.float16).astype(np.float64)


def hadamard128_f64(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty_like(v)
    _load().oracle_hadamard128_f64(v.reshape(-1), out.reshape(-1), v.size)
    return out


def hadamard128_f32(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty_like(v)
    _load().oracle_hadamard128_f32(v.reshape(-1), out.reshape(-1), v.size)
    return out


def input_rotation(x, su=None) -> np.ndarray:
    """RNE_fp16(had_r_128(x * su)) per 128-block of each row (float16)."""
    xb = _bits16(x)
    rows, cols = xb.shape
    out = np.zeros((rows, cols), np.uint16)
    su_b = _bits16(su) if su is not None else None
    _load().oracle_input_rotation(xb, su_b.ctypes.data if su_b is not None else None, rows, cols, out)
    return out.view(np.float16)


def linear(x, trellis, bits: int, K: int, n_stored: int, su, sv, c0: int = 0,
           ncols: int | None = None) -> np.ndarray:
    """Output columns [c0, c0+ncols) of the layer, fp64 (M x ncols)."""
    xb = _bits16(x)
    M = xb.shape[0]
    if ncols is None:
        ncols = n_stored - c0
    y = np.zeros((M, ncols), np.float64)
    rc = _load().oracle_linear(xb, M, K, _bits16(trellis), int(bits), n_stored, _bits16(su),
                               _bits16(sv), c0, ncols, y)
    if rc != 0:
        raise ValueError(f"oracle_linear rejected its arguments (rc={rc})")
    return y


def mask_argmax(logits, n_decodable: int, skip_mask: bool = False):
    """Masks [n_decodable, n_gemm) to -inf in place and returns int32 argmax per row."""
    if logits.dtype != np.float64 or not logits.flags.c_contiguous:
        raise TypeError("logits must be a C-contiguous float64 array")
    M, n_gemm = logits.shape
    am = np.zeros(M, np.int32)
    _load().oracle_mask_argmax(logits, M, n_gemm, int(n_decodable), am, int(bool(skip_mask)))
    return am


def logits_masked(x, trellis, bits: int, K: int, n_stored: int, n_gemm: int, n_decodable: int,
                  su, sv, skip_mask: bool = False):
    """Full masked logits (M x n_gemm, fp64) and their greedy argmax."""
    y = linear(x, trellis, bits, K, n_stored, su, sv, 0, n_gemm)
    am = mask_argmax(y, n_decodable, skip_mask)
    return y, am
