"""Seeded synthetic inputs for the MoE layer.

This module is shared by the tests, the benchmark and the CPU oracle's
callers. It holds none of the layer's arithmetic: it only turns
(seed, tensor id, element index) into numbers.

Generator
---------
Every element is a pure function of (seed, tensor id, flat element index),
so any slice of a tensor (one expert's weights, say) can be regenerated on
its own, on the CPU or on the GPU, with bit-identical results:

* ``bits``   : two rounds of the ``lowbias32`` integer hash (C. Wellons,
  "Prospecting for Hash Functions", 2018) keyed by seed and tensor id.
  Products are split into 16-bit halves so every int64 intermediate stays
  below 2**49; no step depends on overflow behaviour.
* ``normal`` : Irwin-Hall sum of four 16-bit uniforms, centred, scaled to
  unit variance, then multiplied by ``std`` in fp32. Integers up to 2**18
  convert to fp32 exactly and an fp32 multiply is correctly rounded on both
  devices, so CPU and GPU agree bit for bit, also after the cast to bf16
  (round to nearest even on both). The shape is normal to within the
  Irwin-Hall(4) approximation: mean 0, variance 1, tails cut at 3.46 sigma.
* ``uniform``: 24 random bits -> [0, 1) exactly, then ``lo + (hi-lo)*u``.

Tensor ids used by the layer workloads: x=1, Wg=2, Wnoise=3, noise=4,
sel_bias=5, W1=10, W2=11, W1s=12, W2s=13; tests use ids >= 100.
"""
from __future__ import annotations

import math

import torch

_MASK32 = 0xFFFFFFFF
_IH_SIGMA = math.sqrt(4 * (65536 ** 2 - 1) / 12.0)  # std of a sum of four U{0..65535}
_CHUNK = 1 << 24

TID_X, TID_WG, TID_WNOISE, TID_NOISE, TID_BIAS = 1, 2, 3, 4, 5
TID_W1, TID_W2, TID_W1S, TID_W2S = 10, 11, 12, 13


def _mul32(x: torch.Tensor, m: int) -> torch.Tensor:
    """(x * m) mod 2**32 for 0 <= x < 2**32 held in int64."""
    lo, hi = m & 0xFFFF, m >> 16
    return (x * lo + ((x * hi) & 0xFFFF) * 65536) & _MASK32


def _hash32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _hash32_int(v: int) -> int:
    return int(_hash32(torch.tensor([v & _MASK32], dtype=torch.int64))[0])


def _keys(seed: int, tid: int) -> tuple[int, int]:
    a = _hash32_int(seed * 0x9E3779B1 + tid)
    b = _hash32_int(a ^ (tid * 0x85EBCA77 + 0x165667B1))
    return a, b


def bits(idx: torch.Tensor, seed: int, tid: int) -> torch.Tensor:
    """32 random bits (int64 in [0, 2**32)) for each flat index in ``idx``."""
    ka, kb = _keys(seed, tid)
    lo = idx & _MASK32
    hi = idx >> 32
    h = _hash32(lo ^ ka)
    return _hash32(h ^ hi ^ kb)


def _flat_idx(n: int, offset: int, device) -> torch.Tensor:
    return torch.arange(offset, offset + n, dtype=torch.int64, device=device)


def normal(shape, seed: int, tid: int, std: float = 1.0, dtype=torch.float32,
           device="cpu", offset: int = 0) -> torch.Tensor:
    """Approximately N(0, std^2) values; element i of the flat tensor uses
    counter ``offset + i`` of stream (seed, tid)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype, device=device)
    scale = torch.tensor(float(std) / _IH_SIGMA, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        # element i consumes counters 2i and 2i+1 (two 32-bit words = four 16-bit uniforms)
        b = bits(_flat_idx(2 * m, 2 * (offset + s), device), seed, tid).view(m, 2)
        tot = (b[:, 0] & 0xFFFF) + (b[:, 0] >> 16) + (b[:, 1] & 0xFFFF) + (b[:, 1] >> 16)
        v = (tot - 131070).to(torch.float32) * scale
        out[s:s + m] = v.to(dtype)
    return out.view(*shape)


def uniform(shape, seed: int, tid: int, lo: float, hi: float, dtype=torch.float32,
            device="cpu", offset: int = 0) -> torch.Tensor:
    """Values lo + (hi-lo)*u with u = 24 random bits / 2**24, in fp32."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype, device=device)
    lo_t = torch.tensor(lo, dtype=torch.float32, device=device)
    span = torch.tensor(hi - lo, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        b = bits(_flat_idx(m, offset + s, device), seed, tid)
        u = (b >> 8).to(torch.float32) * (1.0 / 16777216.0)
        out[s:s + m] = (lo_t + span * u).to(dtype)
    return out.view(*shape)


def randint(shape, seed: int, tid: int, high: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """Integers in [0, high) (int64) from the top bits of the hash."""
    n = math.prod(shape)
    b = bits(_flat_idx(n, offset, device), seed, tid)
    return ((b * high) >> 32).view(*shape)


def zipf_logit_offset(E: int, s: float) -> torch.Tensor:
    """log of an (unnormalised) Zipf(s) pmf over experts, expert 0 most
    popular: offset[e] = -s * ln(e + 1), fp32. Added to router logits it
    skews the softmax by that pmf (the pmf's constant cancels in softmax)."""
    e = torch.arange(E, dtype=torch.float64)
    return (-s * torch.log(e + 1.0)).to(torch.float32)
