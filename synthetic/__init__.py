"""Seeded synthetic inputs for the trellis-quantized linear layer.

This module only draws random numbers and lays them out in the storage
formats the layer consumes. It holds none of the layer's arithmetic (no
trellis decode, no Hadamard, no matmul), so both the CPU oracle and the CUDA
path can take their inputs from here without sharing any of the method.

Recipe (one numpy Generator per (seed, stream)):
  * stream 0 draws the activations x: fp16 of ``x_scale * N(0, 1)``.
  * matrix ``j`` (gate 0, up 1, down 2; 0 for single-matrix workloads) draws
    from stream ``1 + j``, in this order: the K input signs su (+-1), the
    N_stored output signs, the N_stored output magnitudes U(0.005, 0.02)
    (sv = sign * magnitude, computed in fp64 and rounded to fp16), then the
    trellis words as uniform uint16.
  * Trellis words: tiles of 16x16 weights, ordered row-major over
    (k/16, n/16); each tile owns ``16 * bits`` little-endian uint16 words.
"""
from __future__ import annotations

import dataclasses

import numpy as np


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def trellis_words_per_tile(bits: int) -> int:
    """Each 16x16 tile owns a 256*bits-bit stream, i.e. 16*bits uint16 words."""
    return 16 * bits


def trellis_num_words(K: int, n_stored: int, bits: int) -> int:
    return (K // 16) * (n_stored // 16) * trellis_words_per_tile(bits)


def make_activations(M: int, K: int, seed: int, x_scale: float = 1.0) -> np.ndarray:
    """fp16 activations x of shape (M, K), x_scale * N(0,1), stream 0."""
    g = _rng(seed, 0)
    return (x_scale * g.standard_normal((M, K))).astype(np.float16)


@dataclasses.dataclass
class TrellisMatrix:
    K: int
    n_stored: int
    bits: int
    su: np.ndarray       # (K,) fp16, +-1
    sv: np.ndarray       # (n_stored,) fp16
    trellis: np.ndarray  # (tiles * 16 * bits,) uint16

    @property
    def nbytes(self) -> int:
        return int(self.trellis.nbytes)


def make_matrix(K: int, n_stored: int, bits: int, seed: int, matrix_index: int = 0) -> TrellisMatrix:
    """Random signs, output scales and uniform random tile bitstreams."""
    if K % 16 or n_stored % 16:
        raise ValueError("K and n_stored must be multiples of 16")
    g = _rng(seed, 1 + matrix_index)
    su = np.where(g.integers(0, 2, K) == 1, 1.0, -1.0).astype(np.float16)
    sv_sign = np.where(g.integers(0, 2, n_stored) == 1, 1.0, -1.0)
    sv_mag = g.uniform(0.005, 0.02, n_stored)
    sv = (sv_sign * sv_mag).astype(np.float16)
    words = g.integers(0, 65536, trellis_num_words(K, n_stored, bits), dtype=np.uint16)
    return TrellisMatrix(K=K, n_stored=n_stored, bits=bits, su=su, sv=sv, trellis=words)


# Workload shapes used by the tests and the benchmark, named for what they are.
TINY = dict(name="tiny K=512 N=512 bits=4 M=32", K=512, N=512, bits=4, M=32, seed=0, x_scale=1.0)
GATE_DECODE = dict(name="decode-shaped gate_proj K=5120 N=17408 bits=4 M in {1,4,8,16}",
                   K=5120, N=17408, bits=4, Ms=(1, 4, 8, 16), seed=1, x_scale=0.05)
PREFILL_GEOMS = (dict(name="gate/up K=5120 N=17408", K=5120, N=17408),
                 dict(name="down K=17408 N=5120", K=17408, N=5120))
PREFILL_MS = (64, 128, 256, 1024, 2048, 4096)
PREFILL_SEED = 2
MLP_STACK = dict(layers=64, d_model=5120, d_ff=17408, M=2048, bits=(3, 4), seed_base=3)
LOGITS = dict(name="odd-vocab logits K=5120 n_stored=248320 n_gemm=248192 n_decodable=248077 bits=6",
              K=5120, n_stored=248320, n_gemm=248192, n_decodable=248077, bits=6,
              Ms=(1, 16, 2048), seed=4, chunk=32768)


def make_matrix_device(K: int, n_stored: int, bits: int, seed: int, matrix_index: int = 0, device="cuda"):
    """Timing-only stand-in for make_matrix drawn on the device with torch's
    seeded generator (same shapes and distributions, different stream): used
    where host generation of many gigabytes would dominate a benchmark.
    Returns (trellis int16, su fp16, sv fp16) device tensors."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(matrix_index))
    n_words = trellis_num_words(K, n_stored, bits)
    trellis = torch.randint(-32768, 32768, (n_words,), generator=g, device=device, dtype=torch.int32).to(torch.int16)
    su = torch.where(torch.randint(0, 2, (K,), generator=g, device=device) == 1, 1.0, -1.0).to(torch.float16)
    sign = torch.where(torch.randint(0, 2, (n_stored,), generator=g, device=device) == 1, 1.0, -1.0)
    mag = torch.rand((n_stored,), generator=g, device=device, dtype=torch.float64) * 0.015 + 0.005
    sv = (sign.double() * mag).to(torch.float16)
    return trellis, su, sv
