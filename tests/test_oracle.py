"""Pins for the CPU oracle, checked against things other than itself.

Every pin here is independent of the oracle's own code path: library routines
(numpy's IEEE binary16 conversions, scipy's Sylvester Hadamard matrix),
closed forms derived by hand from the storage-format definition, invariants
of the mathematics, a second decoder, and dense brute force. None of these
tests needs a GPU.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg

import synthetic

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------
# binary16 conversions versus numpy (a library implementation of IEEE 754)
# --------------------------------------------------------------------------

def test_half_to_float_matches_numpy_for_every_bit_pattern(oracle):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    lib = oracle._load()
    got = np.array([lib.oracle_half_to_float(int(p)) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _rne_cases():
    g = np.random.default_rng(123)
    # random fp32 bit patterns over the whole exponent range
    rnd = g.integers(0, 2**32, 200_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    # exact midpoints between adjacent fp16 values (ties), normal and subnormal
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    special = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e-8, 2.0**-25,
                        2.0**-25 * 1.0000001, 2.0**-24, 2.0**-14, np.inf, -np.inf, 3.0e38],
                       np.float32)
    return np.concatenate([rnd, mids, -mids, special])


def test_float_to_half_rne_matches_numpy(oracle):
    vals = _rne_cases()
    ref = vals.astype(np.float16).view(np.uint16)
    lib = oracle._load()
    got = np.array([lib.oracle_float_to_half_rne(float(v)) for v in vals], np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


# --------------------------------------------------------------------------
# Trellis state -> weight
# --------------------------------------------------------------------------

def test_lcg_is_affine_mod_2_32(oracle):
    # u(s) = a*s + c (mod 2^32): second differences vanish, first differences are constant
    us = np.array([oracle.lcg_raw(s) for s in range(0, 65536, 257)], dtype=np.uint64)
    d1 = (us[1:] - us[:-1]) % 2**32
    assert len(set(d1.tolist())) == 1
    step = int(d1[0])
    a = (step * pow(257, -1, 2**32)) % 2**32
    assert a == 89226354
    assert oracle.lcg_raw(0) == 64248484


def test_masked_word_fixes_exponent_bits(oracle):
    # After (u & 0x8FFF8FFF) ^ 0x3B603B60 each half's exponent field is 0b011xx,
    # i.e. both halves lie in +-[2^-3, 2^1).
    ms = np.array([oracle.lcg_masked(s) for s in range(65536)], dtype=np.uint32)
    fixed = ~np.uint32(0x8FFF8FFF)
    assert np.all((ms & fixed) == (np.uint32(0x3B603B60) & fixed))
    for half in (ms & 0xFFFF, ms >> 16):
        exp = (half >> 10) & 0x1F
        assert exp.min() >= 12 and exp.max() <= 15


def test_decode_is_rne_of_exact_half_sum(oracle):
    table = oracle.decode_table()
    ms = np.array([oracle.lcg_masked(s) for s in range(65536)], dtype=np.uint32)
    lo = (ms & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    hi = (ms >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    exact = lo + hi
    # the fp32 sum is exact: the halves share a 2^-13 grid and |sum| < 4
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    ref = exact.astype(np.float16).view(np.uint16)  # numpy's RNE
    assert np.array_equal(table, ref)
    vals = table.view(np.float16).astype(np.float64)
    assert np.all(np.abs(vals) < 4.0)
    # RNE matters: a sizeable share of the sums sit exactly halfway between two fp16 values
    r16 = exact.astype(np.float16)
    other = np.nextafter(r16, np.where(exact > r16, np.float16(np.inf), np.float16(-np.inf)))
    inexact = r16.astype(np.float64) != exact
    ties = inexact & (np.abs(exact - r16) == np.abs(other.astype(np.float64) - exact))
    assert ties.sum() > 1000


# --------------------------------------------------------------------------
# Windowing and bit order: closed forms derived from the format definition
# --------------------------------------------------------------------------

def _single_bit_stream(bits, p):
    w = np.zeros(16 * bits, np.uint16)
    w[p // 16] = 1 << (15 - p % 16)
    return w


def _closed_form_state(bits, p, i):
    """Weight i's state for a stream whose only set bit is p."""
    L = 256 * bits
    e = (i + 1) * bits - 1
    d = (e - p) % L
    return (1 << d) if d <= 15 else 0


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_single_bit_streams_match_closed_form(oracle, bits):
    L = 256 * bits
    for p in sorted({0, 1, 7, 15, 16, L // 2 + 3, L - 16, L - 2, L - 1}):
        w = _single_bit_stream(bits, p)
        want = np.array([_closed_form_state(bits, p, i) for i in range(256)], np.uint16)
        assert np.array_equal(oracle.tile_states_walk(w, bits), want), (bits, p)


def test_documented_bit_order_example(oracle):
    # bits=4, only stream bit 0 (MSB of word 0) set: weights 0..3 see it at
    # state bits 3, 7, 11, 15; every later weight's window excludes it.
    w = _single_bit_stream(4, 0)
    st = oracle.tile_states_walk(w, 4)
    assert st[:4].tolist() == [8, 128, 2048, 32768]
    assert not st[4:].any()
    # the wrap: only the last stream bit set -> weight 0 sees it at state bit `bits`
    st = oracle.tile_states_walk(_single_bit_stream(4, 1023), 4)
    assert st[0] == 16 and st[255] == 1


@pytest.mark.parametrize("bits", [3, 4, 6])
def test_constant_streams(oracle, bits):
    zeros = np.zeros(16 * bits, np.uint16)
    ones = np.full(16 * bits, 0xFFFF, np.uint16)
    assert not oracle.tile_states_walk(zeros, bits).any()
    assert np.all(oracle.tile_states_walk(ones, bits) == 0xFFFF)
    d0 = oracle.decode_tile(zeros, bits).view(np.uint16)
    assert np.all(d0 == oracle.decode_state(0))


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_walk_and_window_decoders_agree(oracle, bits):
    g = np.random.default_rng(bits)
    for _ in range(20):
        w = g.integers(0, 65536, 16 * bits, dtype=np.uint16)
        assert np.array_equal(oracle.tile_states_walk(w, bits), oracle.tile_states_window(w, bits))


def test_reconstruct_places_tiles_row_major(oracle):
    # Tile (tk, tn) holds W[16tk:16tk+16, 16tn:16tn+16], tiles row-major over (k/16, n/16).
    bits, K, N = 3, 48, 64
    m = synthetic.make_matrix(K, N, bits, seed=7)
    W = oracle.reconstruct(m.trellis, bits, K, N)
    wpt = 16 * bits
    for tk in range(K // 16):
        for tn in range(N // 16):
            t = tk * (N // 16) + tn
            tile = oracle.decode_tile(m.trellis[t * wpt:(t + 1) * wpt], bits)
            assert np.array_equal(W[16 * tk:16 * tk + 16, 16 * tn:16 * tn + 16].view(np.uint16),
                                  tile.view(np.uint16))
    # a column slice is the same columns of the full matrix
    Ws = oracle.reconstruct(m.trellis, bits, K, N, 16, 32)
    assert np.array_equal(Ws.view(np.uint16), W[:, 16:48].view(np.uint16))


# --------------------------------------------------------------------------
# Hadamard
# --------------------------------------------------------------------------

def test_hadamard_matches_sylvester_matrix(oracle):
    H = scipy.linalg.hadamard(128).astype(np.float64) / math.sqrt(128.0)
    rows = oracle.hadamard128_f64(np.eye(128))
    assert np.allclose(rows, H, atol=1e-15, rtol=0)
    # closed form of the basis-vector response: (-1)^popcount(i & j) / sqrt(128)
    i = np.arange(128)[:, None]
    j = np.arange(128)[None, :]
    sign = np.where(np.vectorize(lambda v: bin(v).count("1") % 2)(i & j) == 1, -1.0, 1.0)
    assert np.allclose(rows, sign / math.sqrt(128.0), atol=1e-15, rtol=0)


def test_hadamard_orthonormal_involutive_parseval(oracle):
    Hm = oracle.hadamard128_f64(np.eye(128))
    assert np.abs(Hm @ Hm.T - np.eye(128)).max() < 1e-12
    assert np.abs(Hm - Hm.T).max() == 0.0
    v = np.random.default_rng(0).standard_normal(128 * 5)
    hv = oracle.hadamard128_f64(v)
    for b in range(5):
        s = slice(128 * b, 128 * b + 128)
        assert abs(np.linalg.norm(hv[s]) - np.linalg.norm(v[s])) < 1e-12
    assert np.abs(oracle.hadamard128_f64(hv) - v).max() < 1e-13


def test_hadamard_f32_basis_is_exact(oracle):
    # had of a basis vector involves no rounding before the final scale
    rows = oracle.hadamard128_f32(np.eye(128, dtype=np.float32))
    c = np.float32(1.0 / math.sqrt(128.0))
    assert np.all(np.abs(rows) == c)
    assert np.float16(c).view(np.uint16) == 0x2DA8


def test_input_rotation_against_dense_fp64(oracle):
    g = np.random.default_rng(5)
    M, K = 7, 384
    x = g.standard_normal((M, K)).astype(np.float16)
    su = np.where(g.integers(0, 2, K) == 1, 1.0, -1.0).astype(np.float16)
    H = scipy.linalg.hadamard(128) / math.sqrt(128.0)
    dense = np.zeros((M, K))
    xs = x.astype(np.float64) * su.astype(np.float64)
    for b in range(K // 128):
        dense[:, 128 * b:128 * b + 128] = xs[:, 128 * b:128 * b + 128] @ H
    got = oracle.input_rotation(x, su).astype(np.float64)
    ref = dense.astype(np.float16).astype(np.float64)
    # fp32 butterflies vs exact: identical after fp16 rounding except rare 1-ulp flips
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= ulp)
    assert np.mean(got == ref) > 0.99
    # basis input -> the +-fp16(1/sqrt(128)) pattern
    e = np.zeros((1, 128), np.float16)
    e[0, 5] = 1
    r = oracle.input_rotation(e, np.ones(128, np.float16)).view(np.uint16)
    assert set((r & 0x7FFF).ravel().tolist()) == {0x2DA8}


# --------------------------------------------------------------------------
# Linear: dense brute force
# --------------------------------------------------------------------------

@pytest.mark.parametrize("K,N,M,bits", [(128, 128, 3, 4), (256, 384, 5, 3), (384, 256, 2, 6)])
def test_linear_against_dense_brute_force(oracle, K, N, M, bits):
    m = synthetic.make_matrix(K, N, bits, seed=11)
    x = synthetic.make_activations(M, K, seed=11)
    y = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    W = oracle.reconstruct(m.trellis, bits, K, N).astype(np.float64)
    H = scipy.linalg.hadamard(128) / math.sqrt(128.0)
    BH_K = np.kron(np.eye(K // 128), H)
    BH_N = np.kron(np.eye(N // 128), H)
    xr = (x.astype(np.float64) @ np.diag(m.su.astype(np.float64)) @ BH_K).astype(np.float16)
    ref = (xr.astype(np.float64) @ W @ BH_N) * m.sv.astype(np.float64)[None, :]
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.abs(y - ref).max() / rms < 2e-3
    # with the oracle's own (pinned) rotated input the composition agrees to fp64 rounding
    xo = oracle.input_rotation(x, m.su).astype(np.float64)
    ref2 = (xo @ W @ BH_N) * m.sv.astype(np.float64)[None, :]
    assert np.abs(y - ref2).max() / rms < 1e-12


def test_linear_column_slices_agree(oracle):
    K, N, bits = 256, 512, 4
    m = synthetic.make_matrix(K, N, bits, seed=3)
    x = synthetic.make_activations(4, K, seed=3)
    full = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    part = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv, 256, 128)
    assert np.array_equal(full[:, 256:384], part)


# --------------------------------------------------------------------------
# Weight-side rotation variant
# --------------------------------------------------------------------------

def _dense_rotated_weight(oracle, m, K, N, bits):
    """diag(su) . H_K . W . H_N . diag(sv) in fp64 with scipy's Sylvester H."""
    W = oracle.reconstruct(m.trellis, bits, K, N).astype(np.float64)
    H = scipy.linalg.hadamard(128) / math.sqrt(128.0)
    BH_K = np.kron(np.eye(K // 128), H)
    BH_N = np.kron(np.eye(N // 128), H)
    return np.diag(m.su.astype(np.float64)) @ BH_K @ W @ BH_N @ np.diag(m.sv.astype(np.float64)), W, BH_K, BH_N


@pytest.mark.parametrize("K,N,bits", [(128, 128, 4), (256, 384, 3), (384, 256, 6)])
def test_reconstruct_rotated_against_dense_fp64(oracle, K, N, bits):
    m = synthetic.make_matrix(K, N, bits, seed=31 + bits)
    wr = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv).astype(np.float64)
    ref, _, _, _ = _dense_rotated_weight(oracle, m, K, N, bits)
    # fp32 transforms then one fp16 rounding: within one fp16 spacing of the
    # exact value everywhere, and its round-to-nearest almost everywhere
    spacing = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    assert (np.abs(wr - ref) <= spacing).all()
    assert np.mean(wr == ref.astype(np.float16).astype(np.float64)) > 0.99
    # su and sv on the wrong sides (a plausible slip) is far outside that bound
    W = oracle.reconstruct(m.trellis, bits, K, N).astype(np.float64)
    H = scipy.linalg.hadamard(128) / math.sqrt(128.0)
    wrong = np.kron(np.eye(K // 128), H) @ (W * m.sv.astype(np.float64)[None, :]) @ np.kron(np.eye(N // 128), H)
    assert np.abs(wrong - ref).max() > 100 * spacing.max()


def test_reconstruct_rotated_layouts_and_slices(oracle):
    K, N, bits = 256, 512, 4
    m = synthetic.make_matrix(K, N, bits, seed=37)
    kn = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv, layout=0)
    nk = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv, layout=1)
    assert np.array_equal(kn.T.view(np.uint16), nk.view(np.uint16))
    part = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv, n0=256, ncols=128)
    assert np.array_equal(kn[:, 256:384].view(np.uint16), part.view(np.uint16))


@pytest.mark.parametrize("K,N,M,bits", [(256, 384, 6, 4), (384, 256, 3, 3)])
def test_weight_side_variant_is_the_same_layer(oracle, K, N, M, bits):
    m = synthetic.make_matrix(K, N, bits, seed=41 + K)
    x = synthetic.make_activations(M, K, seed=41)
    ref_w, W, BH_K, BH_N = _dense_rotated_weight(oracle, m, K, N, bits)
    x64 = x.astype(np.float64)
    # exact arithmetic: moving both rotations onto the weight changes nothing
    y_weight_side = x64 @ ref_w
    y_layer_exact = ((x64 * m.su.astype(np.float64)[None, :]) @ BH_K @ W @ BH_N) * m.sv.astype(np.float64)[None, :]
    rms = np.sqrt(np.mean(y_layer_exact ** 2))
    assert np.abs(y_weight_side - y_layer_exact).max() / rms < 1e-12
    # with the fp16-rounded rotated weight, against the layer oracle (which
    # rounds x' instead): two independent fp16 roundings, each ~2.8e-4 rms of
    # y per element, so the derived bound for this comparison is 3e-3
    y_ws = oracle.matmul_f64(x, oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv))
    y_layer = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert np.abs(y_ws - y_layer).max() / np.sqrt(np.mean(y_layer ** 2)) < 3e-3


def test_linear_rejects_bad_shapes(oracle):
    m = synthetic.make_matrix(128, 128, 4, seed=0)
    x = synthetic.make_activations(1, 128, seed=0)
    with pytest.raises(ValueError):
        oracle.linear(x, m.trellis, 4, 128, 128, m.su, m.sv, 64, 64)


# --------------------------------------------------------------------------
# Logits mask + greedy selection, with a planted-mistake check
# --------------------------------------------------------------------------

def pad_invariant_violations(logits, argmax, n_decodable):
    """Names every way the pad-column invariant is broken (empty list = holds)."""
    out = []
    pad = logits[:, n_decodable:]
    if pad.size and not np.all(np.isneginf(pad)):
        out.append("pad column is not -inf")
    if not np.all(np.isfinite(logits[:, :n_decodable])):
        out.append("decodable column is not finite")
    if np.any(argmax >= n_decodable):
        out.append(f"pad id {int(argmax.max())} survived selection")
    return out


def test_logits_mask_invariant_and_mutation(oracle):
    K, n_stored, n_gemm, bits = 256, 640, 512, 6
    m = synthetic.make_matrix(K, n_stored, bits, seed=4)
    x = synthetic.make_activations(6, K, seed=4)
    raw = oracle.linear(x, m.trellis, bits, K, n_stored, m.su, m.sv, 0, n_gemm)
    # choose the decodable width so that row 0's unmasked maximum sits in the pad
    n_decodable = int(np.argmax(raw[0]))
    assert 0 < n_decodable < n_gemm
    y, am = oracle.logits_masked(x, m.trellis, bits, K, n_stored, n_gemm, n_decodable, m.su, m.sv)
    assert pad_invariant_violations(y, am, n_decodable) == []
    ref = np.argmax(np.where(np.arange(n_gemm) < n_decodable, raw, -np.inf), axis=1)
    assert np.array_equal(am, ref)
    # planted mistake: skipping the mask must be caught by the invariant check
    y2, am2 = oracle.logits_masked(x, m.trellis, bits, K, n_stored, n_gemm, n_decodable,
                                   m.su, m.sv, skip_mask=True)
    v = pad_invariant_violations(y2, am2, n_decodable)
    assert "pad column is not -inf" in v and any("survived selection" in s for s in v)


def test_argmax_first_index_on_ties(oracle):
    lg = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 9.0]])
    am = oracle.mask_argmax(lg, 3)
    assert am.tolist() == [1, 0]


def test_decode_table_matches_committed_fixture():
    """Regression guard on the whole decode table: the oracle reproduces the
    SHA-256 of the fp16 weights of all 65536 states, the sample states, the
    exact-tie count (states whose half-sum lies exactly between two fp16
    values, where only round-to-nearest-even picks the stored value) and
    the summary statistics written to tests/golden/decode_table.txt by
    make_decode_table.py."""
    import importlib.util
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_decode_table", os.path.join(here, "make_decode_table.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    want = {}
    samples = {}
    for line in open(os.path.join(here, "decode_table.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        if k == "state":
            samples[int(v[0], 16)] = int(v[1], 16)
        else:
            want[k] = v[0]
    got = mk.table_facts()
    assert got["sha256"] == want["sha256"]
    assert got["samples"] == samples
    assert got["ties"] == int(want["ties"])
    assert got["sum"] == float(want["sum"]) and got["min"] == float(want["min"]) and got["max"] == float(want["max"])
