"""Helpers for the GPU parity tests: move seeded inputs to the device and call
the library through its C ABI (via the thin Python binding)."""
import numpy as np

import trellis_quantized_linear_gb300 as tql

TOL = 2e-3  # max|y - y_ref| / rms(y_ref) for floating-point outputs


def torch_mod():
    import torch
    return torch


def to_dev(a):
    torch = torch_mod()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def rel_err(y, ref):
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    return float(np.abs(y.astype(np.float64) - ref).max()) / rms


class Layer:
    """A trellis matrix resident on the GPU."""

    def __init__(self, mat, n_gemm=None):
        self.m = mat
        self.K, self.n_stored, self.bits = mat.K, mat.n_stored, mat.bits
        self.n_gemm = n_gemm if n_gemm is not None else mat.n_stored
        self.trellis = to_dev(mat.trellis)
        self.su = to_dev(mat.su)
        self.sv = to_dev(mat.sv)

    def workspace(self, M_max, m_threshold):
        torch = torch_mod()
        nbytes = tql.exl3_linear_workspace_bytes(M_max, self.K, self.n_gemm, self.bits, m_threshold)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        tql.exl3_workspace_init(ws)
        return ws

    def linear(self, x_dev, m_threshold, y_dtype=tql.EXL3_F32, ws=None):
        torch = torch_mod()
        M = x_dev.shape[0]
        if ws is None:
            ws = self.workspace(M, m_threshold)
        dt = torch.float32 if y_dtype == tql.EXL3_F32 else torch.float16
        y = torch.empty((M, self.n_gemm), dtype=dt, device="cuda")
        tql.exl3_linear(x_dev, M, self.K, self.trellis, self.bits, self.n_stored, self.n_gemm, self.su,
                        self.sv, y, y_dtype, m_threshold, ws)
        torch.cuda.synchronize()
        return y

    def logits(self, x_dev, n_decodable, m_threshold, ws=None):
        torch = torch_mod()
        M = x_dev.shape[0]
        if ws is None:
            ws = self.workspace(M, m_threshold)
        lg = torch.empty((M, self.n_gemm), dtype=torch.float32, device="cuda")
        am = torch.empty((max(M, 4),), dtype=torch.int32, device="cuda")
        tql.exl3_logits_masked(x_dev, M, self.K, self.trellis, self.bits, self.n_stored, self.n_gemm, n_decodable,
                               self.su, self.sv, lg, am, m_threshold, ws)
        torch.cuda.synchronize()
        return lg, am[:M]


def argmax_agrees(gpu_am, ref_logits, margin):
    """Exact agreement where the oracle's top-2 gap exceeds `margin`;
    elsewhere the GPU's pick must lie within `margin` of the oracle maximum.
    Returns the number of near-tie rows."""
    near = 0
    for r in range(ref_logits.shape[0]):
        row = ref_logits[r]
        top = np.argmax(row)
        srt = np.sort(row[np.isfinite(row)])
        gap = srt[-1] - srt[-2] if srt.size > 1 else np.inf
        if gap > margin:
            assert int(gpu_am[r]) == int(top), (r, int(gpu_am[r]), int(top))
        else:
            near += 1
            assert row[int(gpu_am[r])] >= row[top] - margin
    return near
