"""ctypes front end of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of bench.py, never by the product package.
Every function takes and returns numpy arrays on the host; floating-point
inputs are widened to float32 (exact for bf16 values) before the call.

Parity status: every oracle function has at least one pin in
tests/test_oracle_pins.py that does not re-use the oracle's own formula.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

RELU, GELU, SWIGLU = 0, 1, 2
ROUND_NONE, ROUND_F32, ROUND_BF16 = -1, 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double
_F = ctypes.c_float


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        sig = {
            "oracle_round": (_D, [_D, _I]),
            "oracle_softplus": (_D, [_D]),
            "oracle_activation": (_D, [_I, _D]),
            "oracle_softmax": (None, [_I, _P, _P]),
            "oracle_select": (None, [_I, _I, _I, _P, _P, _I, _P, _P]),
            "oracle_router": (None, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I,
                                     _P, _P, _P, _P, _P, _P]),
            "oracle_capacity_of": (_I, [_I, _I, _F]),
            "oracle_capacity": (None, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
            "oracle_dispatch": (None, [_I, _I, _I, _P, _P, _P]),
            "oracle_expert_ffn": (None, [_I, _I, _I, _I, _P, _P, _P, _I, _P]),
            "oracle_combine": (None, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _P]),
            "oracle_aux_stats": (None, [_I, _I, _I, _P, _P, _P, _D, _P, _P, _P, _P]),
            "oracle_bias_update": (None, [_I, _I, _I, _P, _F, _P]),
            "oracle_select_candidates": (None, [_I, _I, _I, _I, _P, _P, _I, _P, _P]),
            "oracle_capacity_policy": (None, [_I, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P,
                                              _P, _P]),
            "oracle_expert_choice": (None, [_I, _I, _I, _P, _P, _P, _P]),
            "oracle_combine_expert_choice": (None, [_I, _I, _I, _I, _P, _P, _P, _P, _I, _P]),
            "oracle_seq_aux_stats": (None, [_I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P]),
            "oracle_philox4x32_10": (None, [_P, _P, _P]),
            "oracle_draw_noise": (None, [_I, _I, ctypes.c_uint64, ctypes.c_uint64, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _f32(a):
    """Host float32 C-contiguous copy (torch tensors of any float dtype too)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ scalars

def round_to(v: float, round_dtype: int) -> float:
    return _load().oracle_round(float(v), int(round_dtype))


def softplus(u: float) -> float:
    return _load().oracle_softplus(float(u))


def activation(act: int, u: float) -> float:
    return _load().oracle_activation(int(act), float(u))


def softmax(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    p = np.empty_like(v)
    _load().oracle_softmax(v.size, _ptr(v), _ptr(p))
    return p


# ------------------------------------------------------------------ stages

def select(s, p, k: int, renorm: bool = True):
    """Top-k (lower index wins ties) on scores s[T,E] and gates from p[T,E]."""
    s, p = _f32(s), _f32(p)
    T, E = s.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().oracle_select(T, E, k, _ptr(s), _ptr(p), int(renorm), _ptr(ids), _ptr(w))
    return ids, w


def router(x, Wg, k: int, Wnoise=None, noise=None, offset=None, bias=None, renorm=True):
    """Returns dict z, H, p, s (double [T,E]), ids [T,k] int32, w [T,k] double."""
    x, Wg, Wnoise, noise = _f32(x), _f32(Wg), _f32(Wnoise), _f32(noise)
    offset, bias = _f32(offset), _f32(bias)
    T, d = x.shape
    E = Wg.shape[1]
    out = {n: np.empty((T, E), np.float64) for n in ("z", "H", "p", "s")}
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().oracle_router(T, d, E, k, _ptr(x), _ptr(Wg), _ptr(Wnoise), _ptr(noise),
                          _ptr(offset), _ptr(bias), int(renorm), _ptr(out["z"]), _ptr(out["H"]),
                          _ptr(out["p"]), _ptr(out["s"]), _ptr(ids), _ptr(w))
    out["ids"], out["w"] = ids, w
    return out


def capacity_of(T: int, E: int, capacity_factor: float) -> int:
    return _load().oracle_capacity_of(int(T), int(E), float(capacity_factor))


def capacity(ids, E: int, C: int):
    """Token-order slot assignment. Returns dict counts, kept, offsets, slot, row_token."""
    ids = _i32(ids)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot = np.empty((T, k), np.int32)
    row_token = np.full(max(T * k, 1), -1, np.int32)
    _load().oracle_capacity(T, k, E, C, _ptr(ids), _ptr(counts), _ptr(kept), _ptr(offsets),
                            _ptr(slot), _ptr(row_token))
    R = int(offsets[E])
    return dict(counts=counts, kept=kept, offsets=offsets, slot=slot, row_token=row_token[:R])


def dispatch(x, slot, R: int):
    x, slot = _f32(x), _i32(slot)
    T, d = x.shape
    k = slot.shape[1]
    xp = np.zeros((max(R, 1), d), np.float32)
    _load().oracle_dispatch(T, d, k, _ptr(x), _ptr(slot), _ptr(xp))
    return xp[:R]


def expert_ffn(X, W1e, W2e, act: int, round_dtype: int = ROUND_NONE):
    """One expert's FFN on rows X[n,d]; W1e [F1,d], W2e [d,F]. Returns double [n,d]."""
    X, W1e, W2e = _f32(X), _f32(W1e), _f32(W2e)
    n, d = X.shape
    F = W2e.shape[1]
    O = np.empty((n, d), np.float64)
    if n:
        _load().oracle_expert_ffn(n, d, F, int(act), _ptr(W1e), _ptr(W2e), _ptr(X),
                                  int(round_dtype), _ptr(O))
    return O


def combine(w, slot, O, Os=None, round_dtype: int = ROUND_NONE):
    """y[t] = sum_kept w O[t,j] + sum_s Os[s,t]; O [n,k,d], Os [S,n,d]. Returns double [n,d]."""
    w = np.ascontiguousarray(w, np.float64)
    slot = _i32(slot)
    O = np.ascontiguousarray(O, np.float64)
    n, k, d = O.shape
    S = 0 if Os is None else Os.shape[0]
    Os = None if Os is None else np.ascontiguousarray(Os, np.float64)
    y = np.empty((n, d), np.float64)
    _load().oracle_combine(n, d, k, S, _ptr(w), _ptr(slot), _ptr(O), _ptr(Os),
                           int(round_dtype), _ptr(y))
    return y


def aux_stats(p, ids, w, E: int, w_imp: float = 1.0):
    """Returns dict f, P, I ([E] double) and aux, cv2, L_imp."""
    p, ids, w = _f32(p), _i32(ids), _f32(w)
    T, k = ids.shape
    f, P, I = (np.empty(E, np.float64) for _ in range(3))
    out3 = np.empty(3, np.float64)
    _load().oracle_aux_stats(T, E, k, _ptr(p), _ptr(ids), _ptr(w), float(w_imp), _ptr(f),
                             _ptr(P), _ptr(I), _ptr(out3))
    return dict(f=f, P=P, I=I, aux=float(out3[0]), cv2=float(out3[1]), L_imp=float(out3[2]))


def bias_update(counts, bias, T: int, k: int, rate: float):
    counts = _i32(counts)
    b = _f32(bias).copy()
    _load().oracle_bias_update(counts.size, int(T), int(k), _ptr(counts), float(rate), _ptr(b))
    return b


def ffn_for_tokens(x, tok, ids, slot, W1_of, W2_of, act, round_dtype, S=0, W1s_of=None,
                   W2s_of=None):
    """Expert outputs for the tokens ``tok``: O [n,k,d] (zeros where dropped) and
    Os [S,n,d]. ``W1_of(e)`` / ``W2_of(e)`` return one expert's weights; experts
    are visited one at a time so only one expert's weights are held at once."""
    x = _f32(x)
    ids = _i32(ids)
    slot = _i32(slot)
    n = len(tok)
    k = ids.shape[1]
    d = x.shape[1]
    O = np.zeros((n, k, d), np.float64)
    need = {}
    for r, t in enumerate(tok):
        for j in range(k):
            if slot[t, j] >= 0:
                need.setdefault(int(ids[t, j]), []).append((r, j))
    for e in sorted(need):
        rows = need[e]
        X = np.stack([x[tok[r]] for r, _ in rows])
        Oe = expert_ffn(X, W1_of(e), W2_of(e), act, round_dtype)
        for q, (r, j) in enumerate(rows):
            O[r, j] = Oe[q]
    Os = np.zeros((S, n, d), np.float64) if S else None
    for s in range(S):
        Os[s] = expert_ffn(x[list(tok)], W1s_of(s), W2s_of(s), act, round_dtype)
    return O, Os


# ------------------------------------------------------- overflow policies

def select_candidates(s, p, k: int, n_cand: int, renorm: bool = True):
    """Top-n_cand candidates (the first k are the top-k choice); every gate
    uses the top-k denominator. Returns ids [T,n_cand] int32, w [T,n_cand] double."""
    s, p = _f32(s), _f32(p)
    T, E = s.shape
    ids = np.empty((T, n_cand), np.int32)
    w = np.empty((T, n_cand), np.float64)
    _load().oracle_select_candidates(T, E, k, n_cand, _ptr(s), _ptr(p), int(renorm), _ptr(ids),
                                     _ptr(w))
    return ids, w


def capacity_policy(ids, k: int, E: int, C: int, priority: int = 0, pad: bool = False):
    """Capacity with re-routing over ids [T,n_cand] (n_cand >= k) in token
    (priority 0) or rank (priority 1) order; pad gives every expert C rows.
    Returns dict counts, kept, offsets, slot, row_token (-1 on padding rows)."""
    ids = _i32(ids)
    T, n_cand = ids.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot = np.empty((T, n_cand), np.int32)
    rows = max(T * n_cand, E * C if pad else 0, 1)
    row_token = np.full(rows, -1, np.int32)
    _load().oracle_capacity_policy(T, k, n_cand, E, C, _ptr(ids), int(priority), int(pad),
                                   _ptr(counts), _ptr(kept), _ptr(offsets), _ptr(slot),
                                   _ptr(row_token))
    R = int(offsets[E])
    return dict(counts=counts, kept=kept, offsets=offsets, slot=slot, row_token=row_token[:R])


def expert_choice(p, C: int):
    """Each expert takes its C most probable tokens (lower index wins ties),
    rows in token order. Returns dict row_token [E*C], row_w [E*C] double,
    tok_row [T,E] int32 (-1 where not chosen)."""
    p = _f32(p)
    T, E = p.shape
    row_token = np.empty(max(E * C, 1), np.int32)
    row_w = np.empty(max(E * C, 1), np.float64)
    tok_row = np.empty((T, E), np.int32)
    _load().oracle_expert_choice(T, E, C, _ptr(p), _ptr(row_token), _ptr(row_w), _ptr(tok_row))
    return dict(row_token=row_token[:E * C], row_w=row_w[:E * C], tok_row=tok_row)


def combine_expert_choice(tok_row, p, O, Os=None, round_dtype: int = ROUND_NONE):
    """y[t] = sum over experts e choosing t (ascending e) of p[t,e] O[row] + sum_s Os[s,t].
    O [E*C,d] double. Returns double [T,d]."""
    tok_row, p = _i32(tok_row), _f32(p)
    O = np.ascontiguousarray(O, np.float64)
    T, E = tok_row.shape
    d = O.shape[1]
    S = 0 if Os is None else Os.shape[0]
    Os = None if Os is None else np.ascontiguousarray(Os, np.float64)
    y = np.empty((T, d), np.float64)
    _load().oracle_combine_expert_choice(T, d, E, S, _ptr(tok_row), _ptr(p), _ptr(O), _ptr(Os),
                                         int(round_dtype), _ptr(y))
    return y


def seq_aux_stats(p, ids, k: int, seq_offsets):
    """Switch aux loss inside each sequence. ids [T,stride] (first k columns
    are the top-k choice). Returns dict f, P ([n_seq,E] double), aux [n_seq], mean."""
    p, ids, so = _f32(p), _i32(ids), _i32(seq_offsets)
    T, E = p.shape
    stride = ids.shape[1]
    n_seq = so.size - 1
    f = np.empty((max(n_seq, 1), E), np.float64)
    P = np.empty((max(n_seq, 1), E), np.float64)
    aux = np.empty(max(n_seq, 1), np.float64)
    mean = ctypes.c_double()
    _load().oracle_seq_aux_stats(E, int(k), stride, _ptr(p), _ptr(ids), n_seq, _ptr(so),
                                 _ptr(f), _ptr(P), _ptr(aux), ctypes.byref(mean))
    return dict(f=f[:n_seq], P=P[:n_seq], aux=aux[:n_seq], mean=mean.value)


def philox4x32_10(ctr, key):
    """Philox4x32-10 block: four 32-bit counter words and two key words in,
    four 32-bit words out (oracle.c cites the published definition)."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def draw_noise(T: int, E: int, seed: int, counter: int = 0) -> np.ndarray:
    """The router's StandardNormal() draws eps[t, e] for the stream (seed,
    counter): Philox4x32-10 and the Box-Muller transform (oracle.c)."""
    eps = np.zeros((T, E), dtype=np.float64)
    _load().oracle_draw_noise(T, E, seed & (2**64 - 1), counter & (2**64 - 1), _ptr(eps))
    return eps
