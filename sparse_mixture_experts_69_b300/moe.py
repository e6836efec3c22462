"""Python binding of libmoe.so (include/moe.h): argument marshalling only.

Every function has the name and argument order of its C entry point. Tensors
are passed as raw device pointers (``data_ptr()``), ``None`` as NULL, and the
stream defaults to torch's current stream. All arithmetic runs in the CUDA
library; this module computes nothing. If the library has not been built the
first call raises ``MoeError``: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_RELU, MOE_GELU, MOE_SWIGLU = 0, 1, 2
MOE_TOKEN_CHOICE, MOE_EXPERT_CHOICE = 0, 1
MOE_PRIORITY_TOKEN, MOE_PRIORITY_RANK = 0, 1
MOE_COMBINE_AUTO, MOE_COMBINE_IN_GEMM, MOE_COMBINE_KERNEL = 0, 1, 2
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_NONFINITE", 6: "MOE_ERR_TIMEOUT",
          7: "MOE_ERR_DEVICE_ARG"}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("renorm_topk", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("importance_weight", ctypes.c_float), ("reroute", ctypes.c_int32),
                ("priority", ctypes.c_int32), ("pad_to_capacity", ctypes.c_int32),
                ("routing", ctypes.c_int32), ("noise_draw", ctypes.c_int32),
                ("noise_seed", ctypes.c_uint64), ("noise_counter", ctypes.c_uint64),
                ("combine_mode", ctypes.c_int32)]


@dataclass
class Config:
    """Problem statement of one layer call (fields of moe_config)."""
    T: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    n_shared: int = 0
    capacity_factor: float = 0.0
    renorm_topk: int = 1
    dtype: int = MOE_BF16
    act: int = MOE_SWIGLU
    importance_weight: float = 1.0
    reroute: int = 0
    priority: int = MOE_PRIORITY_TOKEN
    pad_to_capacity: int = 0
    routing: int = MOE_TOKEN_CHOICE
    noise_draw: int = 0
    noise_seed: int = 0
    noise_counter: int = 0
    combine_mode: int = 0

    def c(self) -> moe_config:
        return moe_config(self.T, self.d_model, self.n_experts, self.top_k, self.d_ff,
                          self.n_shared, self.capacity_factor, self.renorm_topk, self.dtype,
                          self.act, self.importance_weight, self.reroute, self.priority,
                          self.pad_to_capacity, self.routing, self.noise_draw,
                          self.noise_seed & (2**64 - 1), self.noise_counter & (2**64 - 1),
                          self.combine_mode)

    @property
    def n_cand(self) -> int:
        """Candidates per token: top_k + reroute."""
        return self.top_k + self.reroute

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == MOE_BF16 else torch.float32

    @property
    def F1(self) -> int:
        return 2 * self.d_ff if self.act == MOE_SWIGLU else self.d_ff


_lib = None
_P = ctypes.c_void_p
_CFG = ctypes.POINTER(moe_config)
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_capacity": (ctypes.c_int, [_CFG, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_int32)]),
    "moe_workspace_size": (ctypes.c_int, [_CFG, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_workspace_reset": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, _P]),
    "moe_route": (ctypes.c_int, [_CFG] + [_P] * 11 + [ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "moe_dispatch": (ctypes.c_int, [_CFG] + [_P] * 8 + [_P, ctypes.c_size_t, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_CFG] + [_P] * 9 + [_P, ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_CFG] + [_P] * 5 + [_P, ctypes.c_size_t, _P]),
    "moe_aux_stats": (ctypes.c_int, [_CFG] + [_P] * 7 + [_P, ctypes.c_size_t, _P]),
    "moe_bias_update": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_float, _P]),
    "moe_layer_fwd": (ctypes.c_int, [_CFG] + [_P] * 16 + [_P, ctypes.c_size_t, _P]),
    "moe_read_device_error": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, _P]),
    "moe_set_wait_limits": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32]),
    "moe_aux_stats_noalloc": (ctypes.c_int, [_CFG] + [_P] * 7 + [_P]),
    "moe_expert_choice_dispatch": (ctypes.c_int, [_CFG] + [_P] * 7 + [_P, ctypes.c_size_t, _P]),
    "moe_expert_choice_combine": (ctypes.c_int, [_CFG] + [_P] * 5 + [_P, ctypes.c_size_t, _P]),
    "moe_draw_noise": (ctypes.c_int, [_CFG, _P, _P]),
    "moe_seq_aux_stats": (ctypes.c_int, [_CFG, _P, _P, _P, ctypes.c_int32] + [_P] * 4 +
                          [_P, ctypes.c_size_t, _P]),
}


def lib():
    """Load libmoe.so (raises MoeError-compatible RuntimeError if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run "
                               "`python -m sparse_mixture_experts_69_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_capacity(cfg: Config):
    c, r = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_capacity(ctypes.byref(cfg.c()), ctypes.byref(c), ctypes.byref(r)),
           "moe_capacity")
    return c.value, r.value


def moe_workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg.c()), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_reset(cfg: Config, ws, stream=None):
    _check(lib().moe_workspace_reset(ctypes.byref(cfg.c()), _p(ws), ws.numel(), _s(stream)),
           "moe_workspace_reset")


def workspace(cfg: Config, device="cuda") -> torch.Tensor:
    """A zeroed workspace of moe_workspace_size bytes (torch owns the memory)."""
    return torch.zeros(moe_workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_route(cfg: Config, x, Wg, Wnoise, noise, logit_offset, sel_bias, logits, probs,
              sel_scores, topk_ids, topk_w, from_scores, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg.c()), _p(x), _p(Wg), _p(Wnoise), _p(noise),
                           _p(logit_offset), _p(sel_bias), _p(logits), _p(probs), _p(sel_scores),
                           _p(topk_ids), _p(topk_w), int(from_scores), _p(ws), ws.numel(),
                           _s(stream)), "moe_route")


def moe_dispatch(cfg: Config, x, topk_ids, counts, kept, offsets, slot, xp, row_token, ws,
                 stream=None):
    _check(lib().moe_dispatch(ctypes.byref(cfg.c()), _p(x), _p(topk_ids), _p(counts), _p(kept),
                              _p(offsets), _p(slot), _p(xp), _p(row_token), _p(ws), ws.numel(),
                              _s(stream)), "moe_dispatch")


def moe_expert_ffn(cfg: Config, xp, offsets, W1, W2, x, W1s, W2s, yp, ys, ws, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(cfg.c()), _p(xp), _p(offsets), _p(W1), _p(W2),
                                _p(x), _p(W1s), _p(W2s), _p(yp), _p(ys), _p(ws), ws.numel(),
                                _s(stream)), "moe_expert_ffn")


def moe_combine(cfg: Config, yp, slot, topk_w, ys, y, ws, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg.c()), _p(yp), _p(slot), _p(topk_w), _p(ys), _p(y),
                             _p(ws), ws.numel(), _s(stream)), "moe_combine")


def moe_aux_stats(cfg: Config, probs, topk_ids, topk_w, f, P, importance, out3, ws,
                  stream=None):
    _check(lib().moe_aux_stats(ctypes.byref(cfg.c()), _p(probs), _p(topk_ids), _p(topk_w), _p(f),
                               _p(P), _p(importance), _p(out3), _p(ws), ws.numel(), _s(stream)),
           "moe_aux_stats")


def moe_aux_stats_noalloc(cfg: Config, probs, topk_ids, topk_w, f, P, importance, out3,
                          stream=None):
    """moe_aux_stats without a workspace: the library's own device scratch is used
    (at most 512 experts; calls must not overlap on the GPU)."""
    _check(lib().moe_aux_stats_noalloc(ctypes.byref(cfg.c()), _p(probs), _p(topk_ids),
                                       _p(topk_w), _p(f), _p(P), _p(importance), _p(out3),
                                       _s(stream)), "moe_aux_stats_noalloc")


def moe_bias_update(cfg: Config, counts, bias, rate: float, stream=None):
    _check(lib().moe_bias_update(ctypes.byref(cfg.c()), _p(counts), _p(bias), float(rate),
                                 _s(stream)), "moe_bias_update")


def moe_layer_fwd(cfg: Config, x, Wg, Wnoise, noise, logit_offset, sel_bias, W1, W2, W1s, W2s,
                  y, topk_ids, topk_w, counts, aux_vecs, out3, ws, stream=None):
    _check(lib().moe_layer_fwd(ctypes.byref(cfg.c()), _p(x), _p(Wg), _p(Wnoise), _p(noise),
                               _p(logit_offset), _p(sel_bias), _p(W1), _p(W2), _p(W1s), _p(W2s),
                               _p(y), _p(topk_ids), _p(topk_w), _p(counts), _p(aux_vecs),
                               _p(out3), _p(ws), ws.numel(), _s(stream)), "moe_layer_fwd")


def moe_expert_choice_dispatch(cfg: Config, x, probs, offsets, row_token, row_w, tok_row, xp,
                               ws, stream=None):
    _check(lib().moe_expert_choice_dispatch(ctypes.byref(cfg.c()), _p(x), _p(probs),
                                            _p(offsets), _p(row_token), _p(row_w),
                                            _p(tok_row), _p(xp), _p(ws), ws.numel(), _s(stream)),
           "moe_expert_choice_dispatch")


def moe_expert_choice_combine(cfg: Config, yp, tok_row, probs, ys, y, ws, stream=None):
    _check(lib().moe_expert_choice_combine(ctypes.byref(cfg.c()), _p(yp), _p(tok_row),
                                           _p(probs), _p(ys), _p(y), _p(ws), ws.numel(),
                                           _s(stream)), "moe_expert_choice_combine")


def moe_draw_noise(cfg: Config, noise, stream=None):
    """The router's standard-normal draws for (cfg.noise_seed, cfg.noise_counter)
    into noise [T,E] float32, as the layer draws them with noise_draw = 1."""
    _check(lib().moe_draw_noise(ctypes.byref(cfg.c()), _p(noise), _s(stream)), "moe_draw_noise")


def moe_seq_aux_stats(cfg: Config, probs, topk_ids, seq_offsets, n_seq: int, f_seq, P_seq,
                      aux_seq, aux_mean, ws, stream=None):
    _check(lib().moe_seq_aux_stats(ctypes.byref(cfg.c()), _p(probs), _p(topk_ids),
                                   _p(seq_offsets), int(n_seq), _p(f_seq), _p(P_seq),
                                   _p(aux_seq), _p(aux_mean), _p(ws), ws.numel(), _s(stream)),
           "moe_seq_aux_stats")


def moe_read_device_error(cfg: Config, ws, stream=None) -> int:
    """Synchronises the stream; returns the device status (0 = MOE_OK) and clears it."""
    return lib().moe_read_device_error(ctypes.byref(cfg.c()), _p(ws), ws.numel(), _s(stream))


def moe_set_wait_limits(wait_ns: int = 0, policy_passes: int = 0,
                        hold_first_accumulator: int = 0):
    """Limits of the bounded device waits (0 restores each default) and the
    switch that makes the GEMMs' first accumulator wait run out; host only."""
    _check(lib().moe_set_wait_limits(int(wait_ns), int(policy_passes),
                                     int(hold_first_accumulator)), "moe_set_wait_limits")
