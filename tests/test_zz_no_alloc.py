"""The decode-shaped entry point that allocates nothing.

Some callers cannot allocate device memory: a plugin inside a host program
that owns every device buffer, or code that must not call cudaMalloc at run
time because it synchronises the whole device. exl3_linear_decode_noalloc
serves them with the library's own fixed 24 MiB scratch buffer. These tests
call it through the C ABI twice in a row and compare each result with the
ordinary exl3_linear (decode-shaped, caller-provided workspace) and with the
CPU oracle, within the tolerance the parity tests use. This file is
collected last on purpose.
"""
import numpy as np
import pytest

import synthetic
import trellis_quantized_linear_gb300 as tql
from gpu_util import TOL, Layer, rel_err, to_dev, torch_mod

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


def _noalloc(L, xd, y_dtype):
    torch = torch_mod()
    M = xd.shape[0]
    dt = torch.float32 if y_dtype == tql.EXL3_F32 else torch.float16
    y = torch.full((M, L.n_gemm), float("nan"), dtype=dt, device="cuda")
    tql.exl3_linear_decode_noalloc(xd, M, L.K, L.trellis, L.bits, L.n_stored, L.n_gemm, L.su, L.sv, y, y_dtype)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("K,N,bits,Ms", [(5120, 17408, 4, (1, 16)), (512, 512, 4, (37, 5)), (640, 384, 6, (9, 2))])
def test_noalloc_matches_linear_on_two_calls(oracle, K, N, bits, Ms):
    m = synthetic.make_matrix(K, N, bits, seed=K + N)
    L = Layer(m)
    for call, M in enumerate(Ms):  # two calls in a row, different inputs
        x = synthetic.make_activations(M, K, seed=100 + call, x_scale=0.05)
        xd = to_dev(x)
        ref = L.linear(xd, 0, tql.EXL3_F32).cpu().numpy().astype(np.float64)
        got = _noalloc(L, xd, tql.EXL3_F32).cpu().numpy()
        assert rel_err(got, ref) <= TOL, (M, call)
        # and against the oracle directly (M = 37 runs row groups of 16, 16 and 5)
        assert rel_err(got, oracle.linear(x, m.trellis, bits, K, N, m.su, m.sv)) <= TOL, (M, call)
        got16 = _noalloc(L, xd, tql.EXL3_F16).cpu().numpy()
        assert np.array_equal(got16.view(np.uint16), got.astype(np.float16).view(np.uint16))
    assert tql.exl3_get_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_buffer():
    torch = torch_mod()
    lim = tql.EXL3_NOALLOC_SCRATCH_BYTES
    # on this device's SM count: the MLP projections fit the buffer, the logits layer does not
    for K, N, bits in ((5120, 17408, 4), (17408, 5120, 4), (5120, 17408, 3)):
        assert tql.exl3_linear_workspace_bytes(16, K, N, bits, 0) <= lim
    c = synthetic.LOGITS
    K, ns, ng = c["K"], c["n_stored"], c["n_gemm"]
    assert tql.exl3_linear_workspace_bytes(16, K, ng, c["bits"], 0) > lim
    x = torch.zeros((1, K), dtype=torch.float16, device="cuda")
    tr = torch.zeros((16,), dtype=torch.int16, device="cuda")
    su = torch.zeros((K,), dtype=torch.float16, device="cuda")
    sv = torch.zeros((ns,), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(tql.Exl3Error) as e:
        tql.exl3_linear_decode_noalloc(x, 1, K, tr, c["bits"], ns, ng, su, sv, y, tql.EXL3_F32)
    assert e.value.status == 8
