"""Seeded synthetic inputs for the W4A8 block-64 prefill linear.

This module only draws random numbers and encodes them in the input formats
(fp32 activations, u4 weight codes packed two per byte, fp16 scales and zeros).
It holds none of the method's arithmetic, so both the CUDA path and the CPU
oracle can be fed from it.

Workloads stand in for the 512-token prefill ("pp512") runs of Qwen3-class
models in "MNN LLM inference on the SpacemiT K3", section 1 (results table):
no model weights or prompts are used.

Distributions (one recipe for every workload):
  x     fp32 N(0,1), with 4 channels (chosen by the seed, fixed per matrix) scaled
        by an outlier factor (x20; x50 for the 1.7B-class down-projection input)
  q     u4 uniform on 0..15, packed two per byte, even k in the low nibble
  s_w   fp16 (round-to-nearest-even) of U[0.005, 0.02], one per 64 weights along K
  z_w   fp16 (round-to-nearest-even) of U[6, 9], one per 64 weights along K
  bias  fp32 N(0, 0.1^2) where a workload has one
The bit generator is Philox (counter-based), keyed by (seed, matrix index).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BLOCK = 64


@dataclass(frozen=True)
class LinearSpec:
    name: str
    M: int
    K: int
    N: int
    bias: bool = False
    outlier: float = 20.0
    seed: int = 0
    index: int = 0

    @property
    def ops(self) -> int:
        """Effective operations 2*M*N*K (one multiply and one add per MAC)."""
        return 2 * self.M * self.N * self.K


def _cfg(name, rows):
    return name, tuple(LinearSpec(*r) for r in rows)


# Five synthetic prefill workloads.  Sizes: tokens M, input features K, outputs N.
WORKLOADS: dict[str, tuple[str, tuple[LinearSpec, ...]]] = {
    "c0": _cfg("tiny single linear M128 K1024 N1024", [
        ("linear", 128, 1024, 1024, False, 20.0, 0, 0)]),
    "c1": _cfg("pp512 single linear M512 K1024 N3072 +bias (0.6B-class MLP up-projection)", [
        ("up", 512, 1024, 3072, True, 20.0, 0, 0)]),
    "c2": _cfg("pp512 1.7B-class pair M512: K2048->N6144 and K6144->N2048 (x50 outliers)", [
        ("up", 512, 2048, 6144, False, 20.0, 0, 0),
        ("down", 512, 6144, 2048, False, 50.0, 0, 1)]),
    "c3": _cfg("pp512 decoder-layer linear set M512 hidden 2048 (q,k,v,o,gate,up,down)", [
        ("q", 512, 2048, 2048, False, 20.0, 1000, 0),
        ("k", 512, 2048, 1024, False, 20.0, 1001, 0),
        ("v", 512, 2048, 1024, False, 20.0, 1002, 0),
        ("o", 512, 2048, 2048, False, 20.0, 1003, 0),
        ("gate", 512, 2048, 6144, False, 20.0, 1004, 0),
        ("up", 512, 2048, 6144, False, 20.0, 1005, 0),
        ("down", 512, 6144, 2048, False, 20.0, 1006, 0)]),
    "c4": _cfg("7B-class prefill M8192: K4096->N14336 then K14336->N4096", [
        ("up", 8192, 4096, 14336, False, 20.0, 0, 0),
        ("down", 8192, 14336, 4096, False, 20.0, 0, 1)]),
    # One-token decode steps through the same projections (the few-token form).
    "d1": _cfg("decode 1 token, M1 K1024 N3072 +bias (0.6B-class MLP up-projection)", [
        ("up", 1, 1024, 3072, True, 20.0, 0, 0)]),
    "d3": _cfg("decode 1 token through the decoder-layer linear set, hidden 2048 (q,k,v,o,gate,up,down)", [
        ("q", 1, 2048, 2048, False, 20.0, 1000, 0),
        ("k", 1, 2048, 1024, False, 20.0, 1001, 0),
        ("v", 1, 2048, 1024, False, 20.0, 1002, 0),
        ("o", 1, 2048, 2048, False, 20.0, 1003, 0),
        ("gate", 1, 2048, 6144, False, 20.0, 1004, 0),
        ("up", 1, 2048, 6144, False, 20.0, 1005, 0),
        ("down", 1, 6144, 2048, False, 20.0, 1006, 0)]),
    "d4": _cfg("decode 1 token, 7B-class: K4096->N14336 then K14336->N4096", [
        ("up", 1, 4096, 14336, False, 20.0, 0, 0),
        ("down", 1, 14336, 4096, False, 20.0, 0, 1)]),
}

DECODE_MAX_M = 8  # token counts the library runs in its weight-streaming (decode) form


def weight_bytes(spec: LinearSpec) -> int:
    """Bytes of one linear's weights as streamed: packed u4 codes + fp16 s_w and z_w."""
    return spec.N * spec.K // 2 + 2 * 2 * spec.N * (spec.K // BLOCK)


def workload(key: str) -> tuple[str, tuple[LinearSpec, ...]]:
    return WORKLOADS[key]


def _rng(seed: int, index: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, index, stream])))


def pack_u4(q: np.ndarray) -> np.ndarray:
    """Pack u4 codes q[N, K] into bytes [N, K/2]: even k low nibble, odd k high nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] & 0x0F) | ((q[:, 1::2] & 0x0F) << 4)


def make_activations(spec: LinearSpec, rows: int | None = None) -> np.ndarray:
    """fp32 activations x[M, K] (or the first ``rows`` rows, same values)."""
    rng = _rng(spec.seed, spec.index, 1)
    chans = rng.choice(spec.K, size=4, replace=False)
    m = spec.M if rows is None else rows
    x = _rng(spec.seed, spec.index, 2).standard_normal((m, spec.K), dtype=np.float32)
    x[:, chans] *= np.float32(spec.outlier)
    return x


def make_weights(spec: LinearSpec):
    """Returns (q u8 [N,K] codes, wq u8 [N,K/2] packed, s_w fp16 [N,K/64], z_w fp16 [N,K/64], bias fp32 [N] or None)."""
    nb = spec.K // BLOCK
    rng = _rng(spec.seed, spec.index, 3)
    q = rng.integers(0, 16, size=(spec.N, spec.K), dtype=np.uint8)
    s_w = rng.uniform(0.005, 0.02, size=(spec.N, nb)).astype(np.float16)
    z_w = rng.uniform(6.0, 9.0, size=(spec.N, nb)).astype(np.float16)
    bias = None
    if spec.bias:
        bias = (rng.standard_normal(spec.N) * 0.1).astype(np.float32)
    return q, pack_u4(q), s_w, z_w, bias


def make_linear(spec: LinearSpec):
    """All inputs of one linear: dict with x, q, wq, s_w, z_w, bias."""
    q, wq, s_w, z_w, bias = make_weights(spec)
    return {"x": make_activations(spec), "q": q, "wq": wq, "s_w": s_w, "z_w": z_w, "bias": bias}


def random_small(M: int, K: int, N: int, seed: int, bias: bool = True, outlier: float = 20.0):
    """Small random case with the same recipe, for parity sweeps over odd shapes."""
    spec = LinearSpec("small", M, K, N, bias, outlier, seed, 7)
    return make_linear(spec)
