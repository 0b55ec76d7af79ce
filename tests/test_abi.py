"""Host-side checks of the C ABI that need no GPU.

The library must load and export every function include/exl3.h declares,
reject invalid arguments before touching the device, and carry the pages'
host-side arithmetic (logits width alignment, scratch bound).
"""
import ctypes
import os
import re

import pytest

import trellis_quantized_linear_gb300 as tql

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    tql.build()
    return tql.load()


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_header_declarations_are_exported(lib):
    with open(os.path.join(ROOT, "include", "exl3.h")) as f:
        text = f.read()
    declared = set(re.findall(r"^\s*(?:exl3_status|int|int64_t|size_t|const char \*)\s*\**\s*(exl3_\w+)\s*\(",
                              text, flags=re.M))
    assert declared == set(tql.HEADER_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(10):
        assert tql.exl3_status_string(s)
    assert tql.exl3_status_string(99) == "unknown status"


def test_bounds_checked_build_exports_the_same_abi(lib):
    # The bounds-checked build compiles the same sources with EXL3_DEBUG_BOUNDS=1
    # into its own library; it must export every declared entry point and say
    # which build it is. No GPU call: the self-test stops at its host checks.
    from trellis_quantized_linear_gb300 import _build
    path = _build.build(bounds_checked=True)
    assert os.path.basename(path) == "libexl3_bounds.so"
    blib = ctypes.CDLL(path)
    for name in tql.HEADER_SYMBOLS:
        assert hasattr(blib, name), name
    assert blib.exl3_bounds_checked() == 1
    assert lib.exl3_bounds_checked() == 0
    rep, tot = ctypes.c_int(-1), ctypes.c_int(-1)
    blib.exl3_selftest_bounds.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert blib.exl3_selftest_bounds(None, ctypes.byref(tot), None) == 1  # EXL3_ERR_INVALID_ARG
    blib.exl3_status_string.restype = ctypes.c_char_p
    assert b"bounds" in blib.exl3_status_string(9)


def test_supported_bits(lib):
    assert [b for b in range(0, 10) if tql.exl3_supported_bits(b)] == [1, 2, 3, 4, 5, 6, 7, 8]


def test_logits_width_matches_page_example(lib):
    g = _golden("logits_width.txt")
    n = tql.exl3_aligned_logits_width(g["n_decodable"], g["n_stored"])
    assert n == g["n_gemm"]
    assert n % g["align"] == 0
    assert n - g["n_decodable"] == g["n_pad"]
    # the clamp: the aligned width never exceeds the stored rows
    assert tql.exl3_aligned_logits_width(300, 320) == 320
    assert tql.exl3_aligned_logits_width(0, 10) == -1
    assert tql.exl3_aligned_logits_width(11, 10) == -1


def test_workspace_holds_one_reconstruct_chunk_within_page_bound(lib):
    g = _golden("scratch_bound.txt")
    K, chunk = g["K"], g["chunk_cols"]
    assert chunk == tql.EXL3_RECONSTRUCT_CHUNK_COLS
    chunk_bytes = K * chunk * g["bytes_per_weight"]
    assert chunk_bytes <= g["bound_mb"] * 1_000_000
    # a prefill-capable workspace for a logits-width geometry holds exactly one
    # chunk more than a decode-shaped-only one (both hold the rotated rows; its
    # decode-shaped split-K slots already exceed the prefill GEMM's tail slots)
    n_gemm, M = 248192, 2048
    with_prefill = tql.exl3_linear_workspace_bytes_for(M, K, n_gemm, 6, 128, 152)
    decode_only = tql.exl3_linear_workspace_bytes_for(M, K, n_gemm, 6, 0, 152)
    assert with_prefill - decode_only == chunk_bytes
    # narrower than one chunk: the scratch shrinks with n_gemm (rounded to 256
    # rows), plus at most the prefill GEMM's tail slots (3 x SMs fp32 128x256 tiles)
    small = tql.exl3_linear_workspace_bytes_for(M, K, 17408, 4, 128, 152) - \
        tql.exl3_linear_workspace_bytes_for(M, K, 17408, 4, 0, 152)
    assert 17408 * K * 2 <= small <= 17408 * K * 2 + 3 * 152 * 128 * 256 * 4
    # a pure 16-row decode workspace holds neither rotated rows nor a chunk
    d16 = tql.exl3_linear_workspace_bytes_for(16, K, 17408, 4, 0, 152)
    assert d16 < 32 << 20


def _owner(z, P, TS):
    return ((z + 1) * P - 1) // TS


@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120), (5120, 248192), (512, 512), (128, 128)])
@pytest.mark.parametrize("sms", [148, 152, 160])
def test_decode_plan_invariants(lib, K, N, sms):
    """Stream-K split: 12 warps per CTA, one CTA per SM, every warp at least
    one slab; slots = the most warps sharing one 128-column n-block."""
    W = 12
    slots, ctas = tql.exl3_decode_plan(K, N, sms)
    KT, NB = K // 16, N // 128
    TS = NB * KT
    P = min(W * sms, TS)
    assert ctas == -(-P // W) and ctas <= sms
    want = max(_owner((nb + 1) * KT - 1, P, TS) - _owner(nb * KT, P, TS) + 1 for nb in range(NB))
    assert slots == want
    # each warp owns a non-empty, contiguous range and the ranges tile the slab space
    z = [p * TS // P for p in range(P + 1)]
    assert z[0] == 0 and z[-1] == TS and all(b > a for a, b in zip(z, z[1:]))


@pytest.mark.parametrize("M,N,sms,want", [
    (512, 17408, 152, 1), (513, 17408, 152, 0), (1, 17408, 152, 1),   # gate: up to one 512-row block
    (512, 5120, 152, 0),                                               # down: 20 column blocks
    (300, 248192, 152, 1),                                             # odd-vocab logits
    (256, 11776, 152, 1), (256, 11520, 152, 0),                        # 46 / 45 column blocks of 256
    (256, 11520, 148, 1),                                              # the rule scales with the SM count
    (0, 512, 152, -1), (512, 100, 152, -1), (512, 512, 0, -1),         # invalid
])
def test_prefill_path_rule(lib, M, N, sms, want):
    """The prefill-shaped side takes the fused prefill kernel for at most 512
    rows on layers with at least 0.3 x SMs column blocks of 256 (where it was
    measured faster), else reconstruct + GEMM."""
    assert tql.exl3_prefill_path(M, N, sms) == want


def test_decode_plan_gate_geometry_fills_every_sm(lib):
    slots, ctas = tql.exl3_decode_plan(5120, 17408, 152)
    assert ctas == 152 and slots == 15


@pytest.mark.parametrize("sms", [132, 148, 152, 160])
def test_noalloc_limit_covers_mlp_geometries(lib, sms):
    lim = tql.EXL3_NOALLOC_SCRATCH_BYTES
    with open(os.path.join(ROOT, "include", "exl3.h")) as f:
        assert "#define EXL3_NOALLOC_SCRATCH_BYTES ((size_t)24 << 20)" in f.read()
    for K, N, bits in ((5120, 17408, 4), (17408, 5120, 4), (5120, 17408, 3)):
        assert tql.exl3_linear_workspace_bytes_for(16, K, N, bits, 0, sms) <= lim
    assert tql.exl3_linear_workspace_bytes_for(16, 5120, 248192, 6, 0, sms) > lim


def test_weight_rotated_workspace_is_one_slice(lib):
    # one 32768-column slice of W'^T (n rows rounded to 256, K fp16 each)
    assert tql.exl3_weight_rotated_workspace_bytes(5120, 17408) == 17408 * 5120 * 2
    assert tql.exl3_weight_rotated_workspace_bytes(5120, 248192) == 32768 * 5120 * 2
    assert tql.exl3_weight_rotated_workspace_bytes(512, 384) == 512 * 512 * 2
    assert tql.exl3_weight_rotated_workspace_bytes(100, 384) == 0
    assert tql.exl3_weight_rotated_workspace_bytes(512, 100) == 0


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    good = 1 << 20  # a 16-byte aligned fake address; never dereferenced
    L = lib
    # K not a multiple of 128
    assert L.exl3_linear(good, 4, 100, good, 4, 256, 256, good, good, good, 1, 0, good, 1 << 30, None) == 1
    # n_gemm > n_stored; n_stored above 2^24 columns
    assert L.exl3_linear(good, 4, 128, good, 4, 256, 384, good, good, good, 1, 0, good, 1 << 30, None) == 1
    big = (1 << 24) + 128
    assert L.exl3_linear(good, 4, 128, good, 4, big, 256, good, good, good, 1, 0, good, 1 << 62, None) == 1
    # bad dtype, negative threshold, negative M
    assert L.exl3_linear(good, 4, 128, good, 4, 256, 256, good, good, good, 7, 0, good, 1 << 30, None) == 1
    assert L.exl3_linear(good, 4, 128, good, 4, 256, 256, good, good, good, 1, -1, good, 1 << 30, None) == 1
    assert L.exl3_linear(good, -1, 128, good, 4, 256, 256, good, good, good, 1, 0, good, 1 << 30, None) == 1
    # unsupported bits
    assert L.exl3_linear(good, 4, 128, good, 9, 256, 256, good, good, good, 1, 0, good, 1 << 30, None) == 3
    assert L.exl3_linear(good, 4, 128, good, 0, 256, 256, good, good, good, 1, 0, good, 1 << 30, None) == 3
    # misaligned / null pointers
    assert L.exl3_linear(good + 2, 4, 128, good, 4, 256, 256, good, good, good, 1, 0, good, 1 << 30, None) == 2
    assert L.exl3_linear(good, 4, 128, None, 4, 256, 256, good, good, good, 1, 0, good, 1 << 30, None) == 2
    # logits: n_decodable out of range
    assert L.exl3_logits_masked(good, 1, 128, good, 6, 256, 256, 0, good, good, good, good, 0, good,
                                1 << 30, None) == 1
    assert L.exl3_logits_masked(good, 1, 128, good, 6, 256, 256, 257, good, good, good, good, 0, good,
                                1 << 30, None) == 1
    # reconstruct: slice not 128-aligned, bad layout
    assert L.exl3_reconstruct(good, 4, 128, 256, 64, 128, good, 0, None) == 1
    assert L.exl3_reconstruct(good, 4, 128, 256, 0, 128, good, 2, None) == 1
    assert L.exl3_reconstruct(good, 4, 128, 256, 128, 256, good, 0, None) == 1
    # weight-side rotation variant: K not a multiple of 128, slice out of range, workspace too small
    assert L.exl3_reconstruct_rotated(good, 4, 64, 256, 0, 128, good, good, good, 0, None) == 1
    assert L.exl3_reconstruct_rotated(good, 4, 128, 256, 128, 256, good, good, good, 0, None) == 1
    assert L.exl3_reconstruct_rotated(good, 9, 128, 256, 0, 128, good, good, good, 0, None) == 3
    assert L.exl3_reconstruct_rotated(good, 4, 128, 256, 0, 128, good + 8, good, good, 0, None) == 2
    assert L.exl3_linear_weight_rotated(good, 4, 100, good, 4, 256, 256, good, good, good, 1, good, 1 << 30,
                                        None) == 1
    # hadamard: cols not a multiple of 128
    assert L.exl3_hadamard128(good, good, None, 2, 100, None) == 1
    assert L.exl3_hadamard128(good, good + 8, None, 2, 128, None) == 2
    # self-test limit out of range
    assert L.exl3_selftest_wait_timeout(0, None) == 1
    # the no-alloc entry point applies the same shape, row and bit rules
    assert L.exl3_linear_decode_noalloc(good, 4, 100, good, 4, 256, 256, good, good, good, 1, None) == 1
    assert L.exl3_linear_decode_noalloc(good, 4, 128, good, 4, big, 256, good, good, good, 1, None) == 1
    assert L.exl3_linear_decode_noalloc(good, 4, 128, good, 4, 256, 384, good, good, good, 1, None) == 1
    assert L.exl3_linear_decode_noalloc(good, -1, 128, good, 4, 256, 256, good, good, good, 1, None) == 1
    assert L.exl3_linear_decode_noalloc(good, (1 << 31) + 1, 128, good, 4, 256, 256, good, good, good, 1,
                                        None) == 1
    assert L.exl3_linear_decode_noalloc(good, 4, 128, good, 4, 256, 256, good, good, good, 5, None) == 1
    assert L.exl3_linear_decode_noalloc(good, 4, 128, good, 9, 256, 256, good, good, good, 1, None) == 3
    assert L.exl3_linear_decode_noalloc(good + 4, 4, 128, good, 4, 256, 256, good, good, good, 1, None) == 2


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib
    mod = importlib.reload(tql)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "libexl3.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(ImportError):
        mod.load()
    importlib.reload(tql)
