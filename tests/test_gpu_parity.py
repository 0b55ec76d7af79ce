"""GPU parity: every entry point of libexl3 against the CPU oracle.

Bars: bit-exact for the reconstructed weights, the input rotation and the
pad mask / argmax; max|y - y_ref| / rms(y_ref) <= 2e-3 for the fp32 layer
output (fp32 accumulation against the oracle's fp64); the fp16 output is the
round-to-nearest-even of the same call's fp32 output, bit for bit.
"""
import numpy as np
import pytest

import synthetic
import trellis_quantized_linear_gb300 as tql
from gpu_util import TOL, Layer, argmax_agrees, rel_err, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tql.build()
    torch.cuda.set_device(0)
    tql.exl3_init(0)
    yield
    assert tql.exl3_get_device_status() == 0


# ---------------------------------------------------------------------------
# input rotation
# ---------------------------------------------------------------------------

# (2048, 5120) is the prefill-shaped gate input; (700, 3840) a ragged large one.
@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 640), (256, 5120), (2048, 5120), (700, 3840)])
@pytest.mark.parametrize("with_scale", [True, False])
def test_hadamard128_bit_exact(oracle, rows, cols, with_scale):
    torch = torch_mod()
    x = synthetic.make_activations(rows, cols, seed=rows + cols)
    su = synthetic.make_matrix(cols, 128, 4, seed=rows).su if with_scale else None
    xd = to_dev(x)
    yd = torch.empty_like(xd)
    tql.exl3_hadamard128(xd, yd, to_dev(su) if su is not None else None)
    torch.cuda.synchronize()
    ref = oracle.input_rotation(x, su).view(np.uint16)
    got = yd.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("rows,cols", [(9, 384), (700, 3840)])
def test_hadamard128_in_place(oracle, rows, cols):
    torch = torch_mod()
    x = synthetic.make_activations(rows, cols, seed=3)
    xd = to_dev(x)
    tql.exl3_hadamard128(xd, xd, None)
    torch.cuda.synchronize()
    assert np.array_equal(xd.cpu().numpy().view(np.uint16), oracle.input_rotation(x).view(np.uint16))
    assert tql.exl3_get_device_status() == 0


# ---------------------------------------------------------------------------
# reconstruct
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("layout", [tql.EXL3_LAYOUT_KN, tql.EXL3_LAYOUT_NK])
@pytest.mark.parametrize("n0,n_cols", [(0, 640), (256, 256)])
def test_reconstruct_bit_exact(oracle, bits, layout, n0, n_cols):
    torch = torch_mod()
    K, N = 272, 640
    m = synthetic.make_matrix(K, N, bits, seed=bits)
    tr = to_dev(m.trellis)
    shape = (K, n_cols) if layout == tql.EXL3_LAYOUT_KN else (n_cols, K)
    w = torch.full(shape, 7.0, dtype=torch.float16, device="cuda")
    tql.exl3_reconstruct(tr, bits, K, N, n0, n_cols, w, layout)
    torch.cuda.synchronize()
    ref = oracle.reconstruct(m.trellis, bits, K, N, n0, n_cols).view(np.uint16)
    got = w.cpu().numpy().view(np.uint16)
    if layout == tql.EXL3_LAYOUT_NK:
        got = got.T
    assert np.array_equal(got, ref)


def test_reconstruct_full_gate_geometry(oracle):
    """The whole 5120 x 17408 gate_proj weight, both layouts, bit for bit."""
    torch = torch_mod()
    K, N, bits = 5120, 17408, 4
    m = synthetic.make_matrix(K, N, bits, seed=1)
    tr = to_dev(m.trellis)
    w = torch.empty((K, N), dtype=torch.float16, device="cuda")
    tql.exl3_reconstruct(tr, bits, K, N, 0, N, w, tql.EXL3_LAYOUT_KN)
    wt = torch.empty((N, K), dtype=torch.float16, device="cuda")
    tql.exl3_reconstruct(tr, bits, K, N, 0, N, wt, tql.EXL3_LAYOUT_NK)
    torch.cuda.synchronize()
    assert torch.equal(w.t().contiguous(), wt)
    ref = oracle.reconstruct(m.trellis, bits, K, N).view(np.uint16)
    assert np.array_equal(w.cpu().numpy().view(np.uint16), ref)


# ---------------------------------------------------------------------------
# linear: both paths
# ---------------------------------------------------------------------------

DECODE, PREFILL = 0, 1  # m_threshold values that force each path


@pytest.mark.parametrize("K,N,bits", [(512, 512, 4), (128, 256, 3), (640, 384, 6), (256, 768, 2),
                                      (384, 256, 5), (256, 256, 8), (256, 384, 1), (384, 384, 7)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16, 37])
def test_linear_decode_path(oracle, K, N, bits, M):
    m = synthetic.make_matrix(K, N, bits, seed=K + N + bits)
    x = synthetic.make_activations(M, K, seed=M)
    L = Layer(m)
    y = L.linear(to_dev(x), DECODE).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("M", [1, 4])
def test_decode_small_rows_long_k(oracle, M):
    """A long-K, wide decode-shaped layer (K=17408, N=20480): each warp's
    slab range (about 95 slabs) streams many more chunks than its ring holds,
    and every n-block (1088 slabs) is split over 12-13 warps' partial slots;
    every output column against the oracle."""
    K, N, bits = 17408, 20480, 4
    m = synthetic.make_matrix(K, N, bits, seed=M + 40)
    x = synthetic.make_activations(M, K, seed=M + 41)
    y = Layer(m).linear(to_dev(x), DECODE).cpu().numpy()
    assert rel_err(y, oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)) <= TOL


@pytest.mark.parametrize("K,N,bits", [(512, 512, 4), (256, 384, 3), (640, 640, 6), (128, 256, 1), (384, 256, 7),
                                      (1024, 256, 2), (256, 384, 5), (384, 256, 8)])
@pytest.mark.parametrize("M", [17, 50, 100, 128, 129, 200, 256, 300])
def test_linear_fused_decode_path(oracle, K, N, bits, M):
    """Decode-shaped calls above 16 rows run the fused tensor-core kernel
    (256 rows per launch, stream-K over n-blocks and 64-row k steps). The M
    values cover MMA widths 32..256 and x' rings of 8, 4, 3 and 2 stages;
    M = 300 is a 256-row launch plus a 44-row one."""
    m = synthetic.make_matrix(K, N, bits, seed=K + 7 * N + bits)
    x = synthetic.make_activations(M, K, seed=M + 3)
    L = Layer(m)
    y = L.linear(to_dev(x), DECODE).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("M", [24, 64, 256])
def test_fused_decode_full_gate_geometry(oracle, M):
    """The tensor-core decode-shaped kernel on the whole gate_proj geometry
    (K=5120, N=17408): every output column against the oracle. Its stream-K
    plan puts a different k-step boundary in every n-block, so no block is
    left unchecked."""
    K, N, bits = 5120, 17408, 4
    m = synthetic.make_matrix(K, N, bits, seed=2)
    x = synthetic.make_activations(M, K, seed=2)
    y = Layer(m).linear(to_dev(x), DECODE).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("K,N,bits", [(512, 512, 4), (256, 384, 3), (640, 640, 6), (256, 256, 1), (384, 256, 7)])
@pytest.mark.parametrize("M", [1, 32, 130, 256])
def test_linear_prefill_path(oracle, K, N, bits, M):
    m = synthetic.make_matrix(K, N, bits, seed=K * 3 + N + bits)
    x = synthetic.make_activations(M, K, seed=M + 1)
    L = Layer(m)
    y = L.linear(to_dev(x), PREFILL).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("K,N,n_dec,M", [(2048, 384, 300, 6), (1024, 640, 640, 130), (4096, 256, 256, 1),
                                         (512, 33152, 33000, 520)])
def test_prefill_stream_k_tail(oracle, K, N, n_dec, M):
    """Prefill-shaped calls whose tiles do not fill a wave: the tail tiles'
    k blocks are spread over all CTAs and reduced from fp32 partial slots,
    including a masked split tile, a last tile of only 128 columns and two
    reconstruct chunks."""
    bits = 4
    m = synthetic.make_matrix(K, N, bits, seed=K + N + M)
    x = synthetic.make_activations(M, K, seed=M + 5)
    L = Layer(m)
    lg, am = L.logits(to_dev(x), n_dec, 1)
    lg = lg.cpu().numpy()
    assert np.all(np.isneginf(lg[:, n_dec:]))
    ref, _ = oracle.logits_masked(x, m.trellis, bits, K, N, N, n_dec, m.su, m.sv)
    fin = np.isfinite(ref)
    assert rel_err(lg[fin], ref[fin]) <= TOL
    assert np.array_equal(am.cpu().numpy(), np.argmax(lg, axis=1))


@pytest.mark.parametrize("M,bits,N", [(300, 4, 5120), (1100, 2, 5120), (512, 5, 5120), (1100, 3, 5248)])
def test_prefill_pair_tiles(oracle, M, bits, N):
    """Prefill-shaped calls that run as CTA-pair tiles (256 x 256, two SMs per
    tile): an odd number of 128-row tiles (M = 300, 1100), whose last pair
    has no second row tile, and an even one; no split tail; N = 5248 ends in
    a tile column only 128 wide. Every output checked."""
    K = 512
    m = synthetic.make_matrix(K, N, bits, seed=M + bits)
    x = synthetic.make_activations(M, K, seed=M)
    y = Layer(m).linear(to_dev(x), PREFILL).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y, ref) <= TOL


# The fused prefill kernel (CTA pairs, 512-row x 256-column tiles, the
# trellis decoded into the MMA operand) serves prefill-shaped calls of at most
# 512 rows on layers with at least 46 column blocks of 256 (152 SMs).
@pytest.mark.parametrize("bits,M,N", [(b, 300, 12288) for b in range(1, 9)] +
                         [(4, 1, 12288), (4, 200, 12288), (4, 512, 12288), (3, 300, 12416), (5, 512, 12416)])
def test_fused_prefill_path(oracle, bits, M, N):
    """Every bit width; one and two 256-row sub-blocks (M <= 256, > 256),
    a partial second sub-block (M = 300), a full tile (M = 512); N = 12416
    ends in a 128-wide column block, whose odd CTA decodes a block it never
    stores. Every output against the oracle, fp32 and fp16 (RNE of fp32)."""
    K = 512
    m = synthetic.make_matrix(K, N, bits, seed=N + bits + M)
    x = synthetic.make_activations(M, K, seed=M + bits)
    L = Layer(m)
    xd = to_dev(x)
    y32 = L.linear(xd, PREFILL, tql.EXL3_F32).cpu().numpy()
    y16 = L.linear(xd, PREFILL, tql.EXL3_F16).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y32, ref) <= TOL
    assert np.array_equal(y16.view(np.uint16), y32.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("M", [300, 512])
def test_fused_prefill_full_gate_geometry(oracle, M):
    """The fused prefill on the whole gate_proj geometry (K=5120, N=17408):
    68 column blocks on 76 CTA pairs, every output column of every row."""
    K, N, bits = 5120, 17408, 4
    m = synthetic.make_matrix(K, N, bits, seed=synthetic.PREFILL_SEED)
    x = synthetic.make_activations(M, K, seed=synthetic.PREFILL_SEED)
    y = Layer(m).linear(to_dev(x), 128).cpu().numpy()
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y, ref) <= TOL


def test_tiny_workload_both_paths_and_fp16_rounding(oracle):
    t = synthetic.TINY
    m = synthetic.make_matrix(t["K"], t["N"], t["bits"], seed=t["seed"])
    x = synthetic.make_activations(t["M"], t["K"], seed=t["seed"], x_scale=t["x_scale"])
    L = Layer(m)
    xd = to_dev(x)
    ref = oracle.linear(x, m.trellis, t["bits"], t["K"], t["N"], m.su, m.sv)
    for thr in (DECODE, PREFILL):
        y32 = L.linear(xd, thr, tql.EXL3_F32).cpu().numpy()
        y16 = L.linear(xd, thr, tql.EXL3_F16).cpu().numpy()
        assert rel_err(y32, ref) <= TOL
        assert np.array_equal(y16.view(np.uint16), y32.astype(np.float16).view(np.uint16))


def test_prefill_chunks_past_32768_columns(oracle):
    # n_gemm = 32768 + 384: two reconstruct chunks, the second narrower than a
    # GEMM tile (M > 512, so the prefill side is reconstruct + GEMM)
    K, N, bits, M = 128, 33152, 4, 520
    m = synthetic.make_matrix(K, N, bits, seed=9)
    x = synthetic.make_activations(M, K, seed=9)
    L = Layer(m)
    xd = to_dev(x)
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    for thr in (PREFILL, DECODE):
        y = L.linear(xd, thr).cpu().numpy()
        assert rel_err(y, ref) <= TOL


def test_empty_inputs_are_no_ops():
    # M = 0 rows (and zero rows / columns for the building blocks) is a valid
    # call on every entry point: EXL3_OK, nothing written, no device error.
    torch = torch_mod()
    K, N, bits = 256, 384, 4
    m = synthetic.make_matrix(K, N, bits, seed=21)
    L = Layer(m)
    x = torch.ones((1, K), dtype=torch.float16, device="cuda")  # valid pointer; no row is read
    for thr in (DECODE, PREFILL, 1000):
        ws = L.workspace(1, thr)
        y = torch.full((1, N), 7.0, dtype=torch.float32, device="cuda")
        am = torch.full((4,), -5, dtype=torch.int32, device="cuda")
        tql.exl3_linear(x, 0, K, L.trellis, bits, N, N, L.su, L.sv, y, tql.EXL3_F32, thr, ws)
        tql.exl3_logits_masked(x, 0, K, L.trellis, bits, N, N, N - 3, L.su, L.sv, y, am, thr, ws)
        torch.cuda.synchronize()
        assert bool(torch.all(y == 7.0)) and bool(torch.all(am == -5))
    y16 = torch.full((1, N), 3.0, dtype=torch.float16, device="cuda")
    tql.exl3_linear_decode_noalloc(x, 0, K, L.trellis, bits, N, N, L.su, L.sv, y16, tql.EXL3_F16)
    xr = torch.full((1, K), 3.0, dtype=torch.float16, device="cuda")
    tql.exl3_hadamard128(x, xr, L.su, rows=0, cols=K)
    w = torch.full((K, 128), 3.0, dtype=torch.float16, device="cuda")
    tql.exl3_reconstruct(L.trellis, bits, K, N, 128, 0, w, tql.EXL3_LAYOUT_KN)
    tql.exl3_reconstruct_rotated(L.trellis, bits, K, N, 128, 0, L.su, L.sv, w, tql.EXL3_LAYOUT_KN)
    torch.cuda.synchronize()
    assert bool(torch.all(y16 == 3.0)) and bool(torch.all(xr == 3.0)) and bool(torch.all(w == 3.0))
    assert tql.exl3_get_device_status() == 0


# The smallest shapes the ABI accepts: one 128-row k block and one 128-column
# n block (8 k slabs for the decode path, a half-width tile on the prefill
# path), on every path.
@pytest.mark.parametrize("bits", [1, 4, 8])
@pytest.mark.parametrize("M,thr", [(1, DECODE), (16, DECODE), (17, DECODE), (200, PREFILL)])
def test_smallest_shapes(oracle, bits, M, thr):
    K, N = 128, 128
    m = synthetic.make_matrix(K, N, bits, seed=41 + bits)
    x = synthetic.make_activations(M, K, seed=41 + M)
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    y = Layer(m).linear(to_dev(x), thr).cpu().numpy()
    assert rel_err(y, ref) <= TOL


# The largest K the ABI accepts (131072 = 2^17): 8192 k slabs per n-block on
# the decode path, 2048 k steps on the tensor-core decode path, a 2048-block
# K loop (stream-K tail split) on the prefill path.
@pytest.mark.parametrize("M,thr", [(1, DECODE), (16, DECODE), (40, DECODE), (200, PREFILL)])
def test_maximum_k(oracle, M, thr):
    K, N, bits = 131072, 256, 2
    m = synthetic.make_matrix(K, N, bits, seed=31)
    x = synthetic.make_activations(M, K, seed=31)
    ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
    y = Layer(m).linear(to_dev(x), thr).cpu().numpy()
    assert rel_err(y, ref) <= TOL


def test_runtime_dispatch_uses_threshold(oracle):
    K, N, bits = 256, 256, 4
    m = synthetic.make_matrix(K, N, bits, seed=5)
    L = Layer(m)
    for M in (7, 8, 9):
        x = synthetic.make_activations(M, K, seed=M)
        ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
        y = L.linear(to_dev(x), 8).cpu().numpy()
        assert rel_err(y, ref) <= TOL


def test_gemm_width_narrower_than_stored(oracle):
    K, n_stored, n_gemm, bits, M = 256, 640, 384, 4, 20
    m = synthetic.make_matrix(K, n_stored, bits, seed=12)
    x = synthetic.make_activations(M, K, seed=12)
    L = Layer(m, n_gemm=n_gemm)
    ref = oracle.linear(x, m.trellis, bits, K, n_stored, m.su, m.sv, 0, n_gemm)
    for thr in (DECODE, PREFILL):
        assert rel_err(L.linear(to_dev(x), thr).cpu().numpy(), ref) <= TOL


def test_workspace_too_small_is_rejected():
    torch = torch_mod()
    m = synthetic.make_matrix(256, 256, 4, seed=1)
    L = Layer(m)
    x = to_dev(synthetic.make_activations(64, 256, seed=1))
    need = tql.exl3_linear_workspace_bytes(64, 256, 256, 4, 1)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y = torch.empty((64, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(tql.Exl3Error) as e:
        tql.exl3_linear(x, 64, 256, L.trellis, 4, 256, 256, L.su, L.sv, y, tql.EXL3_F32, 1, ws, need - 256)
    assert e.value.status == 4


# ---------------------------------------------------------------------------
# logits: mask + greedy selection
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("thr", [DECODE, PREFILL])
@pytest.mark.parametrize("M", [6, 40])  # decode-shaped: the 16-row kernel / the tensor-core kernel
def test_logits_mask_and_argmax_small(oracle, thr, M):
    K, n_stored, n_gemm, bits = 256, 640, 512, 6
    m = synthetic.make_matrix(K, n_stored, bits, seed=4)
    x = synthetic.make_activations(M, K, seed=4)
    raw = oracle.linear(x, m.trellis, bits, K, n_stored, m.su, m.sv, 0, n_gemm)
    n_decodable = int(np.argmax(raw[0]))  # row 0's unmasked maximum lands in the pad
    L = Layer(m, n_gemm=n_gemm)
    lg, am = L.logits(to_dev(x), n_decodable, thr)
    lg = lg.cpu().numpy()
    am = am.cpu().numpy()
    assert np.all(np.isneginf(lg[:, n_decodable:]))
    assert np.all(np.isfinite(lg[:, :n_decodable]))
    assert np.array_equal(am, np.argmax(lg, axis=1))  # the CPU argmax of the GPU's own buffer
    ref, ref_am = oracle.logits_masked(x, m.trellis, bits, K, n_stored, n_gemm, n_decodable, m.su, m.sv)
    fin = np.isfinite(ref)
    assert rel_err(lg[fin], ref[fin]) <= TOL
    rms = float(np.sqrt(np.mean(ref[fin] ** 2)))
    argmax_agrees(am, ref, 2 * TOL * rms)


# ---------------------------------------------------------------------------
# full-size workloads, checked on sampled 128-column blocks
# ---------------------------------------------------------------------------

def test_decode_gate_full_size(oracle):
    """The decode-shaped headline workload (gate_proj K=5120 N=17408 bits=4,
    M = 1, 4, 8, 16): every output column of every call against the oracle.
    The stream-K decode splits each of the 136 n-blocks at a different k
    slab, so every n-block exercises its own slot boundary."""
    g = synthetic.GATE_DECODE
    K, N, bits = g["K"], g["N"], g["bits"]
    m = synthetic.make_matrix(K, N, bits, seed=g["seed"])
    L = Layer(m)
    for M in g["Ms"]:
        x = synthetic.make_activations(M, K, seed=g["seed"], x_scale=g["x_scale"])
        y = L.linear(to_dev(x), DECODE).cpu().numpy()
        ref = oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)
        assert rel_err(y, ref) <= TOL, M


@pytest.mark.parametrize("geom", [0, 1])
def test_prefill_full_size_sampled_rows(oracle, geom):
    """Prefill-shaped calls at full size (gate 5120->17408 at M=2048, down
    17408->5120 at M=1024): 128 evenly spaced rows, every output column."""
    gm = synthetic.PREFILL_GEOMS[geom]
    K, N, bits = gm["K"], gm["N"], 4
    M = 2048 if geom == 0 else 1024
    m = synthetic.make_matrix(K, N, bits, seed=synthetic.PREFILL_SEED)
    x = synthetic.make_activations(M, K, seed=synthetic.PREFILL_SEED)
    y = Layer(m).linear(to_dev(x), 128)
    rows = np.arange(0, M, M // 128)
    got = y[rows].cpu().numpy()
    ref = oracle.linear(x[rows], m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(got, ref) <= TOL


@pytest.mark.parametrize("M,thr,n_rows", [(1, 128, 1), (16, 128, 16), (64, 128, 16), (300, 1, 16), (2048, 128, 64)])
def test_logits_full_vocab(oracle, M, thr, n_rows):
    """Odd-vocab logits (K=5120, n_stored=248320, n_gemm=248192,
    n_decodable=248077, bits=6) at M = 1, 16 (the 16-row decode kernel), 64
    (the tensor-core decode kernel) and 2048 (prefill-shaped): the pad is
    -inf, the rest finite, the GPU argmax equals the CPU argmax of the GPU's
    own buffer on every row, and on n_rows evenly spaced rows every logit
    and the greedy pick are checked against the oracle over the whole vocab."""
    c = synthetic.LOGITS
    K, n_stored, n_gemm, n_dec, bits = c["K"], c["n_stored"], c["n_gemm"], c["n_decodable"], c["bits"]
    assert tql.exl3_aligned_logits_width(n_dec, n_stored) == n_gemm
    m = synthetic.make_matrix(K, n_stored, bits, seed=c["seed"])
    x = synthetic.make_activations(M, K, seed=c["seed"])
    L = Layer(m, n_gemm=n_gemm)
    lg, am = L.logits(to_dev(x), n_dec, thr)
    torch = torch_mod()
    assert bool(torch.isneginf(lg[:, n_dec:]).all())
    assert bool(torch.isfinite(lg[:, :n_dec]).all())
    assert torch.equal(am.long(), torch.argmax(lg, dim=1))
    rows = np.arange(0, M, M // n_rows)
    ref, ref_am = oracle.logits_masked(x[rows], m.trellis, bits, K, n_stored, n_gemm, n_dec, m.su, m.sv)
    got = lg[torch.from_numpy(rows).cuda()].cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got))
    assert rel_err(got[fin], ref[fin]) <= TOL
    rms = float(np.sqrt(np.mean(ref[fin] ** 2)))
    argmax_agrees(am.cpu().numpy()[rows], ref, 2 * TOL * rms)


# Each kernel path that writes logits applies the pad mask itself. A case per
# path: the pad covers columns that path writes, and the decodable width is
# chosen below row 0's unmasked maximum, so a path that dropped the mask would
# leave a finite pad column and let the pad win row 0's argmax. The planted
# mistake lives in the oracle (skip_mask): with it, row 0's pick lands in the
# pad, which is what the checks below would then catch.
MASK_PATHS = {
    # 16-row stream-K decode kernel, n-blocks shared by several warps (slot reduction)
    "decode_slot_reduction": dict(K=256, n_stored=640, n_gemm=512, bits=6, M=6, thr=0),
    # the same kernel on a wide, shallow layer: warps that own whole n-blocks finish them in place
    "decode_whole_block": dict(K=128, n_stored=248320, n_gemm=248192, bits=6, M=3, thr=0),
    # tensor-core decode kernel (16 < M), its slot reduction
    "fused_decode": dict(K=256, n_stored=640, n_gemm=512, bits=6, M=40, thr=0),
    # prefill GEMM: whole-tile epilogue over two reconstruct chunks (M > 512)
    "prefill_epilogue": dict(K=256, n_stored=33408, n_gemm=33152, bits=4, M=520, thr=1),
    # fused prefill (one 512-row block, many column blocks): its TMEM epilogue
    "fused_prefill": dict(K=256, n_stored=33408, n_gemm=33152, bits=4, M=300, thr=1),
    # prefill GEMM: last partial wave split along K, reduced by its finalize kernel
    "prefill_split_tail": dict(K=2048, n_stored=512, n_gemm=384, bits=4, M=6, thr=1),
}


@pytest.mark.parametrize("path", sorted(MASK_PATHS))
def test_pad_mask_on_every_logits_path(oracle, path):
    c = MASK_PATHS[path]
    K, ns, ng, bits, M, thr = c["K"], c["n_stored"], c["n_gemm"], c["bits"], c["M"], c["thr"]
    m = synthetic.make_matrix(K, ns, bits, seed=K + ns + M)
    x = synthetic.make_activations(M, K, seed=M + 7)
    raw = oracle.linear(x, m.trellis, bits, K, ns, m.su, m.sv, 0, ng)
    # pad starts below row 0's unmasked maximum (and within the first 300 columns,
    # so that it spans every n-block, tile and chunk after it)
    n_dec = max(1, min(int(np.argmax(raw[0])), 300))
    ref, ref_am = oracle.logits_masked(x, m.trellis, bits, K, ns, ng, n_dec, m.su, m.sv)
    _, bad_am = oracle.logits_masked(x, m.trellis, bits, K, ns, ng, n_dec, m.su, m.sv, skip_mask=True)
    assert bad_am[0] >= n_dec  # the planted mistake is visible to these checks
    lg, am = Layer(m, n_gemm=ng).logits(to_dev(x), n_dec, thr)
    lg = lg.cpu().numpy()
    am = am.cpu().numpy()
    assert np.all(np.isneginf(lg[:, n_dec:]))
    assert np.all(np.isfinite(lg[:, :n_dec]))
    assert np.all(am < n_dec)
    assert np.array_equal(am, np.argmax(lg, axis=1))
    fin = np.isfinite(ref)
    assert rel_err(lg[fin], ref[fin]) <= TOL
    rms = float(np.sqrt(np.mean(ref[fin] ** 2)))
    argmax_agrees(am, ref, 2 * TOL * rms)


def test_silu_mul_glue():
    torch = torch_mod()
    g = synthetic.make_activations(7, 384, seed=31)
    u = synthetic.make_activations(7, 384, seed=32)
    out = torch.empty((7, 384), dtype=torch.float16, device="cuda")
    tql.exl3_silu_mul(to_dev(g), to_dev(u), out)
    torch.cuda.synchronize()
    a = g.astype(np.float64)
    ref = (a / (1.0 + np.exp(-a)) * u.astype(np.float64)).astype(np.float16).astype(np.float64)
    got = out.cpu().numpy().astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= ulp)


@pytest.mark.parametrize("layer", [0, 31, 63])
@pytest.mark.parametrize("bits", [3, 4])
def test_mlp_stack_layers_sampled(oracle, layer, bits):
    """Dense MLP stack geometry: each layer's gate, up and down projections on
    fresh N(0,1) input at M=2048 (prefill path), 128 sampled rows x 2 column
    blocks checked against the oracle."""
    st = synthetic.MLP_STACK
    d, f, M = st["d_model"], st["d_ff"], st["M"]
    rows = np.arange(0, M, M // 128)
    for j, (K, N) in enumerate(((d, f), (d, f), (f, d))):
        m = synthetic.make_matrix(K, N, bits, seed=st["seed_base"] + layer, matrix_index=j)
        x = synthetic.make_activations(M, K, seed=st["seed_base"])
        y = Layer(m).linear(to_dev(x), 128).cpu().numpy()
        for b in (0, N // 128 - 1):
            ref = oracle.linear(x[rows], m.trellis, bits, K, N, m.su, m.sv, 128 * b, 128)
            assert rel_err(y[rows, 128 * b:128 * b + 128], ref) <= TOL, (j, b)


# ---------------------------------------------------------------------------
# graph capture: the dispatch lives inside the call
# ---------------------------------------------------------------------------

def test_graph_capture_keeps_each_path(oracle):
    torch = torch_mod()
    K, N, bits, thr = 256, 512, 4, 64
    m = synthetic.make_matrix(K, N, bits, seed=21)
    L = Layer(m)
    ws = L.workspace(256, thr)
    need_decode = tql.exl3_linear_workspace_bytes(8, K, N, bits, thr)  # decode-only prefix of the workspace
    x_small = to_dev(synthetic.make_activations(8, K, seed=22))
    x_big = to_dev(synthetic.make_activations(256, K, seed=23))
    y_small = torch.empty((8, N), dtype=torch.float32, device="cuda")
    y_big = torch.empty((256, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(s):
        for xd, yd in ((x_small, y_small), (x_big, y_big)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                tql.exl3_linear(xd, xd.shape[0], K, L.trellis, bits, N, N, L.su, L.sv, yd, tql.EXL3_F32, thr, ws)
            graphs.append(g)
    torch.cuda.synchronize()
    scratch = ws[need_decode:]
    scratch.fill_(0x5A)
    torch.cuda.synchronize()
    graphs[0].replay()
    torch.cuda.synchronize()
    assert bool((scratch == 0x5A).all()), "the decode-shaped graph touched the prefill scratch"
    graphs[1].replay()
    torch.cuda.synchronize()
    assert not bool((scratch == 0x5A).all()), "the prefill-shaped graph did not use its scratch"
    ref_s = oracle.linear(x_small.cpu().numpy(), m.trellis, bits, K, N, m.su, m.sv)
    ref_b = oracle.linear(x_big.cpu().numpy(), m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(y_small.cpu().numpy(), ref_s) <= TOL
    assert rel_err(y_big.cpu().numpy(), ref_b) <= TOL


# ---------------------------------------------------------------------------
# weight-side rotation variant
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [1, 3, 4, 6, 8])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("n0,n_cols", [(0, 384), (256, 128)])
def test_reconstruct_rotated_bit_exact(oracle, bits, layout, n0, n_cols):
    torch = torch_mod()
    K, N = 256, 384
    m = synthetic.make_matrix(K, N, bits, seed=50 + bits)
    L = Layer(m)
    shape = (K, n_cols) if layout == 0 else (n_cols, K)
    w = torch.empty(shape, dtype=torch.float16, device="cuda")
    tql.exl3_reconstruct_rotated(L.trellis, bits, K, N, n0, n_cols, L.su, L.sv, w, layout)
    torch.cuda.synchronize()
    ref = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv, n0, n_cols, layout)
    assert np.array_equal(w.cpu().numpy().view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("K,N,bits", [(256, 384, 4), (384, 256, 3), (640, 512, 6)])
@pytest.mark.parametrize("M", [5, 130])
def test_linear_weight_rotated(oracle, K, N, bits, M):
    torch = torch_mod()
    m = synthetic.make_matrix(K, N, bits, seed=60 + K + bits)
    x = synthetic.make_activations(M, K, seed=M + 61)
    L = Layer(m)
    ws = torch.empty(tql.exl3_weight_rotated_workspace_bytes(K, N), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tql.exl3_linear_weight_rotated(to_dev(x), M, K, L.trellis, bits, N, N, L.su, L.sv, y, tql.EXL3_F32, ws)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    wr = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv)
    assert rel_err(got, oracle.matmul_f64(x, wr)) <= TOL
    # the same layer as exl3_linear, within the budget derived for moving the
    # fp16 rounding from x' to W'
    assert rel_err(got, oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)) <= 3e-3


def test_weight_rotated_full_gate_geometry_sampled(oracle):
    torch = torch_mod()
    K, N, bits, M = 5120, 17408, 4, 256
    m = synthetic.make_matrix(K, N, bits, seed=2)
    x = synthetic.make_activations(M, K, seed=2)
    L = Layer(m)
    ws = torch.empty(tql.exl3_weight_rotated_workspace_bytes(K, N), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tql.exl3_linear_weight_rotated(to_dev(x), M, K, L.trellis, bits, N, N, L.su, L.sv, y, tql.EXL3_F32, ws)
    w = torch.empty((128, K), dtype=torch.float16, device="cuda")
    for b in (0, 77, N // 128 - 1):
        tql.exl3_reconstruct_rotated(L.trellis, bits, K, N, 128 * b, 128, L.su, L.sv, w, tql.EXL3_LAYOUT_NK)
        torch.cuda.synchronize()
        ref_w = oracle.reconstruct_rotated(m.trellis, bits, K, N, m.su, m.sv, 128 * b, 128, 1)
        assert np.array_equal(w.cpu().numpy().view(np.uint16), ref_w.view(np.uint16)), b
        ref = oracle.matmul_f64(x, ref_w.T)
        assert rel_err(y[:, 128 * b:128 * b + 128].cpu().numpy(), ref) <= TOL, b


@pytest.mark.parametrize("M", [1, 16, 40])
def test_decode_stack_graph_matches_eager(oracle, M):
    """A whole decode step of a small MLP stack (3 layers of gate, up,
    SiLU*up, down) captured as one CUDA graph gives the eager result bit for
    bit (same kernels, deterministic reductions), and its first gate output
    matches the oracle."""
    torch = torch_mod()
    d, f, bits, nl = 256, 384, 4, 3
    layers = []
    for l in range(nl):
        mats = [synthetic.make_matrix(K, N, bits, seed=100 + 3 * l + j) for j, (K, N) in
                enumerate(((d, f), (d, f), (f, d)))]
        layers.append([Layer(m) for m in mats])
    ws = torch.zeros(max(tql.exl3_linear_workspace_bytes(M, d, f, bits, 0),
                         tql.exl3_linear_workspace_bytes(M, f, d, bits, 0)), dtype=torch.uint8, device="cuda")
    tql.exl3_workspace_init(ws)
    x = synthetic.make_activations(M, d, seed=77, x_scale=0.5)
    x0 = to_dev(x)
    g = torch.empty((M, f), dtype=torch.float16, device="cuda")
    u, h = torch.empty_like(g), torch.empty_like(g)
    xa = torch.empty((M, d), dtype=torch.float16, device="cuda")
    g1 = torch.empty((M, f), dtype=torch.float32, device="cuda")

    def step():
        xin = x0
        for li, (lg, lu, ld) in enumerate(layers):
            if li == 0:
                tql.exl3_linear(xin, M, d, lg.trellis, bits, f, f, lg.su, lg.sv, g1, tql.EXL3_F32, 0, ws)
            tql.exl3_linear(xin, M, d, lg.trellis, bits, f, f, lg.su, lg.sv, g, tql.EXL3_F16, 0, ws)
            tql.exl3_linear(xin, M, d, lu.trellis, bits, f, f, lu.su, lu.sv, u, tql.EXL3_F16, 0, ws)
            tql.exl3_silu_mul(g, u, h)
            tql.exl3_linear(h, M, f, ld.trellis, bits, d, d, ld.su, ld.sv, xa, tql.EXL3_F16, 0, ws)
            xin = xa

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager_out, eager_g1 = xa.clone(), g1.clone()
    xa.fill_(0)
    g1.fill_(0)
    with torch.cuda.stream(s):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            step()
    xa.fill_(0)
    torch.cuda.synchronize()
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(xa.view(torch.int16), eager_out.view(torch.int16))
    assert torch.equal(g1.view(torch.int32), eager_g1.view(torch.int32))
    m0 = layers[0][0].m
    ref = oracle.linear(x, m0.trellis, bits, d, f, m0.su, m0.sv)
    assert rel_err(g1.cpu().numpy(), ref) <= TOL


# ---------------------------------------------------------------------------
# failure detection without a fault: a bounded wait that runs out
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_context_survives(oracle):
    torch = torch_mod()
    assert tql.exl3_get_device_status() == 0
    tql.exl3_selftest_wait_timeout(2000)  # 2 ms
    assert tql.exl3_get_device_status() == 7
    assert tql.exl3_get_device_status() == 0  # read-and-clear
    # the context still works
    m = synthetic.make_matrix(128, 128, 4, seed=2)
    x = synthetic.make_activations(3, 128, seed=2)
    y = Layer(m).linear(to_dev(x), DECODE).cpu().numpy()
    assert rel_err(y, oracle.linear(x, m.trellis, 4, 128, 128, m.su, m.sv)) <= TOL
    torch.cuda.synchronize()
