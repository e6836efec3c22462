"""Seeded synthetic inputs for the MoE layer.

This module is shared by the tests, the benchmark and the CPU oracle's
callers. It holds none of the layer's arithmetic: it only turns
(seed, tensor id, element index) into numbers.

Generator
---------
Every element is a pure function of (seed, tensor id, flat element index),
so any slice of a tensor (one expert's weights, say) can be regenerated on
its own, on the CPU or on the GPU:

* ``philox`` : the counter-based Philox4x32-10 block cipher (Salmon, Moraes,
  Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011),
  written here with int64 tensor arithmetic: every 32 x 32-bit product is
  split into 16-bit halves so no intermediate reaches 2**63. Block b of
  stream (seed, tid) encrypts the counter (b mod 2**32, b div 2**32, tid, 0)
  under the key (seed mod 2**32, seed div 2**32) and yields four 32-bit
  words; element i of a tensor takes word i mod 4 of block i div 4.
* ``normal`` : the Box-Muller transform (Box and Muller, 1958) of the two
  words of a pair, u1 = (w0 + 1) / 2**32 in (0, 1], u2 = w1 / 2**32 in
  [0, 1): sqrt(-2 ln u1) cos(2 pi u2) for the pair's first element and
  sqrt(-2 ln u1) sin(2 pi u2) for its second, times ``std``, in float64,
  rounded to float32 and then to the requested dtype. The values are
  N(0, std^2) up to the 32-bit resolution of the uniforms (|z| <= 6.66).
  CPU and GPU agree bit for bit up to the last-ulp differences of their
  float64 log / cos / sin, which change a float32 result only where the
  float64 value falls within an ulp of a float32 rounding boundary (about
  one element in 10^8, and far fewer after the cast to bf16). Where exact
  equality matters the tests copy the GPU's tensors to the host.
* ``uniform``: the top 24 bits of an element's word -> u in [0, 1) exactly,
  then ``lo + (hi-lo)*u`` in fp32.
* ``randint``: (word * high) >> 32, integers in [0, high).

Tensor ids used by the layer workloads: x=1, Wg=2, Wnoise=3, noise=4,
sel_bias=5, W1=10, W2=11, W1s=12, W2s=13; tests use ids >= 100.
"""
from __future__ import annotations

import math

import torch

_MASK32 = 0xFFFFFFFF
_CHUNK = 1 << 24          # elements generated per pass (bounds the temporaries)

# Philox4x32-10 constants (the multipliers and the Weyl key increments of the
# published definition)
_PHILOX_M0, _PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
_PHILOX_W0, _PHILOX_W1 = 0x9E3779B9, 0xBB67AE85

TID_X, TID_WG, TID_WNOISE, TID_NOISE, TID_BIAS = 1, 2, 3, 4, 5
TID_W1, TID_W2, TID_W1S, TID_W2S = 10, 11, 12, 13


def _mulhilo(m: int, c: torch.Tensor):
    """(hi, lo) 32-bit words of the 64-bit product m * c, for 0 <= c < 2**32
    held in int64 and a 32-bit constant m."""
    mh, ml = m >> 16, m & 0xFFFF
    ch, cl = c >> 16, c & 0xFFFF
    mid = cl * mh + ch * ml                # < 2**33
    low = cl * ml + (mid << 16)            # < 2**50: the product's low 32 bits + carry
    return ch * mh + (low >> 32), low & _MASK32


def philox(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox4x32 rounds on the counter words c0..c3 (int64 tensors of
    32-bit values, broadcastable) under the key (k0, k1); returns four tensors."""
    k0 &= _MASK32
    k1 &= _MASK32
    for _ in range(10):
        h0, l0 = _mulhilo(_PHILOX_M0, c0)
        h1, l1 = _mulhilo(_PHILOX_M1, c2)
        c0, c1, c2, c3 = h1 ^ c1 ^ k0, l1, h0 ^ c3 ^ k1, l0
        k0 = (k0 + _PHILOX_W0) & _MASK32
        k1 = (k1 + _PHILOX_W1) & _MASK32
    return c0, c1, c2, c3


def _blocks(b0: int, nb: int, seed: int, tid: int, device):
    """Words of blocks b0 .. b0+nb-1 of stream (seed, tid): int64 [nb, 4]."""
    b = torch.arange(b0, b0 + nb, dtype=torch.int64, device=device)
    c2 = torch.full_like(b, tid & _MASK32)
    c3 = torch.zeros_like(b)
    w = philox(b & _MASK32, b >> 32, c2, c3, seed & _MASK32, (seed >> 32) & _MASK32)
    return torch.stack(w, dim=1)


def words(n: int, seed: int, tid: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """32-bit words (int64 in [0, 2**32)) of elements offset .. offset+n-1."""
    b0 = offset // 4
    b1 = (offset + n + 3) // 4
    w = _blocks(b0, b1 - b0, seed, tid, device).view(-1)
    s = offset - 4 * b0
    return w[s:s + n]


def _normal_chunk(n: int, seed: int, tid: int, std: float, device, offset: int):
    """float64 N(0, std^2) values of elements offset .. offset+n-1. The pair
    (2q, 2q+1) shares one Box-Muller draw (cos for the first, sin for the second)."""
    p0 = offset // 2
    p1 = (offset + n + 1) // 2
    w = words(2 * (p1 - p0), seed, tid, device, 2 * p0).view(-1, 2)
    u1 = (w[:, 0].double() + 1.0) * (1.0 / 4294967296.0)
    u2 = w[:, 1].double() * (1.0 / 4294967296.0)
    rad = torch.sqrt(-2.0 * torch.log(u1))
    ang = (2.0 * math.pi) * u2
    z = torch.stack((rad * torch.cos(ang), rad * torch.sin(ang)), dim=1).view(-1)
    s = offset - 2 * p0
    return z[s:s + n] * float(std)


def normal(shape, seed: int, tid: int, std: float = 1.0, dtype=torch.float32,
           device="cpu", offset: int = 0) -> torch.Tensor:
    """N(0, std^2) values; element i of the flat tensor is element ``offset + i``
    of stream (seed, tid)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        v = _normal_chunk(m, seed, tid, std, device, offset + s)
        out[s:s + m] = v.to(torch.float32).to(dtype)
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
        b = words(m, seed, tid, device, offset + s)
        u = (b >> 8).to(torch.float32) * (1.0 / 16777216.0)
        out[s:s + m] = (lo_t + span * u).to(dtype)
    return out.view(*shape)


def randint(shape, seed: int, tid: int, high: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """Integers in [0, high) (int64, high < 2**31) from the element's word."""
    n = math.prod(shape)
    b = words(n, seed, tid, device, offset)
    return ((b * high) >> 32).view(*shape)


def zipf_logit_offset(E: int, s: float) -> torch.Tensor:
    """log of an (unnormalised) Zipf(s) pmf over experts, expert 0 most
    popular: offset[e] = -s * ln(e + 1), fp32. Added to router logits it
    skews the softmax by that pmf (the pmf's constant cancels in softmax)."""
    e = torch.arange(E, dtype=torch.float64)
    return (-s * torch.log(e + 1.0)).to(torch.float32)
