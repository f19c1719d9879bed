"""Seeded synthetic inputs for one MoE-layer forward.

This module only draws random numbers; it holds none of the layer's arithmetic.
The CUDA-path tests, the bench and the oracle tests all take their inputs from
here, so both sides of every parity check see the same bits.

Generator (counter based, so any element can be drawn on any device):
  * key      = mix64(seed * 1000003 + tensor_id)             (Python ints, mod 2**64)
  * word(c)  = mix64(key + (c + 1) * 0x9E3779B97F4A7C15)     (SplitMix64 finaliser)
  * element i of a tensor uses words 2i and 2i+1:
        u1 = ((word(2i)   >> 11) + 1) * 2**-53   in (0, 1]
        u2 =  (word(2i+1) >> 11)      * 2**-53   in [0, 1)
        n  = sqrt(-2 ln u1) * cos(2 pi u2)       (Box-Muller, cosine branch, float64)
  * value    = bf16(fp32(n * sigma))  (round-to-nearest-even at both steps)

Tensor ids: x=1, router weight=2, W1=3, W3=4, W2=5, bias permutation=6, free
rows for combine-only tests=7.

The Zipf logit bias draws E uniforms from tensor id 6, ranks them into a
permutation pi of 1..E and sets b[e] = fp32(-s * ln pi(e)), so expert e's
routing weight is multiplied by pi(e)**-s.

The uint64 SplitMix64 arithmetic runs on torch int64 tensors: multiplication
wraps modulo 2**64 and right shifts are made logical with a mask, so the low
64 bits equal the unsigned result on CPU and on CUDA alike.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

TID_X, TID_WR, TID_W1, TID_W3, TID_W2, TID_BIAS, TID_ROWS = 1, 2, 3, 4, 5, 6, 7


def _s64(v: int) -> int:
    """Unsigned 64-bit constant as the signed int64 with the same bits."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference for the tensor version)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def tensor_key(seed: int, tensor_id: int) -> int:
    return mix64_int(seed * 1000003 + tensor_id)


def words(key: int, start: int, count: int, device) -> torch.Tensor:
    """word(c) for c in [start, start+count) as int64 (bit pattern of the uint64)."""
    c = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = c * _s64(_GAMMA) + _s64(key)
    return _mix64(z)


def normals(key: int, start: int, count: int, device) -> torch.Tensor:
    """Standard normals for elements [start, start+count) of the tensor keyed by key (float64)."""
    w = words(key, 2 * start, 2 * count, device).view(count, 2)
    a = _lsr(w[:, 0], 11).to(torch.float64)
    b = _lsr(w[:, 1], 11).to(torch.float64)
    u1 = (a + 1.0) * (2.0 ** -53)
    u2 = b * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def uniforms(key: int, count: int, device="cpu") -> torch.Tensor:
    w = words(key, 0, count, device)
    return _lsr(w, 11).to(torch.float64) * (2.0 ** -53)


def gaussian_bf16(shape, sigma: float, seed: int, tensor_id: int, device="cpu",
                  chunk: int = 1 << 25) -> torch.Tensor:
    """bf16 tensor of N(0, sigma^2) draws, generated in chunks on `device`."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    key = tensor_key(seed, tensor_id)
    for s0 in range(0, n, chunk):
        c = min(chunk, n - s0)
        v = normals(key, s0, c, device) * sigma
        out[s0:s0 + c] = v.to(torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """fp32 logit offsets b[e] = -s * ln(pi(e)), pi a seeded permutation of 1..E."""
    u = uniforms(tensor_key(seed, TID_BIAS), E).numpy()
    order = np.argsort(u, kind="stable")
    pi = np.empty(E, dtype=np.int64)
    pi[order] = np.arange(1, E + 1)
    return (-s * np.log(pi.astype(np.float64))).astype(np.float32)


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    S: int = 1          # owner-aligned output segments (simulated source ranks)
    zipf_s: float = 0.0  # 0 = balanced routing, no bias
    note: str = ""

    @property
    def R(self) -> int:
        return self.T * self.k

    def gemm_flops(self) -> float:
        return 6.0 * self.T * self.k * self.d * self.F

    def router_flops(self) -> float:
        return 2.0 * self.T * self.d * self.E

    def flops(self) -> float:
        return self.gemm_flops() + self.router_flops()

    def minimal_bytes(self) -> float:
        """x + router weight + all expert weights + idx/gates + out (bytes)."""
        return (2.0 * self.T * self.d + 2.0 * self.E * self.d + 6.0 * self.E * self.F * self.d
                + 8.0 * self.T * self.k + 2.0 * self.T * self.d)


CONFIGS = {
    "tiny": MoEConfig("tiny", T=256, d=256, E=8, k=2, F=512,
                      note="tiny MoE layer, oracle runs in seconds"),
    "mid": MoEConfig("mid", T=4096, d=2048, E=64, k=6, F=1408, zipf_s=1.0,
                     note="mid MoE layer, Zipf(1.0) expert skew"),
    "dit": MoEConfig("dit", T=32768, d=1152, E=16, k=2, F=4608, S=8, zipf_s=1.2,
                     note="DiT-MoE long-sequence layer, Zipf(1.2), 8 owner segments"),
    "fine": MoEConfig("fine", T=16384, d=4096, E=256, k=8, F=2048,
                      note="fine-grained experts, balanced routing"),
    "coarse": MoEConfig("coarse", T=8192, d=4096, E=8, k=2, F=14336,
                        note="coarse experts, balanced routing"),
}


@dataclass
class MoEInputs:
    cfg: MoEConfig
    x: torch.Tensor       # [T, d] bf16
    wr: torch.Tensor      # [E, d] bf16
    bias: torch.Tensor | None  # [E] fp32 or None
    w1: torch.Tensor      # [E, F, d] bf16
    w3: torch.Tensor      # [E, F, d] bf16
    w2: torch.Tensor      # [E, d, F] bf16
    extra: dict = field(default_factory=dict)


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu", weights: bool = True) -> MoEInputs:
    """All inputs of one layer: x~N(0,1), Wr,W1,W3~N(0,1/d), W2~N(0,1/F)."""
    T, d, E, F = cfg.T, cfg.d, cfg.E, cfg.F
    x = gaussian_bf16((T, d), 1.0, seed, TID_X, device)
    wr = gaussian_bf16((E, d), 1.0 / math.sqrt(d), seed, TID_WR, device)
    bias = None
    if cfg.zipf_s > 0:
        bias = torch.from_numpy(zipf_bias(E, cfg.zipf_s, seed)).to(device)
    if weights:
        w1 = gaussian_bf16((E, F, d), 1.0 / math.sqrt(d), seed, TID_W1, device)
        w3 = gaussian_bf16((E, F, d), 1.0 / math.sqrt(d), seed, TID_W3, device)
        w2 = gaussian_bf16((E, d, F), 1.0 / math.sqrt(F), seed, TID_W2, device)
    else:
        w1 = w3 = w2 = None
    return MoEInputs(cfg, x, wr, bias, w1, w3, w2)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor, as a contiguous numpy array (host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
