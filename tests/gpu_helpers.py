"""Shared pieces of the GPU parity tests: running the C ABI through the
binding, and the comparison rules.

Tolerances (floating point) follow the stated targets:
  router logits / probs  max |gpu - ref| <= 1e-4 * max |ref| per token row
  gates                  the probs' rule when the probs come from each side's own
                         logits (a gate is a renormalised prob, so a logit error d
                         moves it by a relative ~d); relative 1e-5 when both sides
                         get identical probs (fp32 division vs double)
  expert / layer output  max |gpu - ref| <= 2e-2 * max |ref| (bf16),
                         1e-4 * max |ref| (fp32)
  aux, cv2               relative 1e-5
Integer outputs (ids, slots, counts, offsets, rows) are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from sparse_mixture_experts_69_b300 import moe

TOL_Y = {moe.MOE_BF16: 2e-2, moe.MOE_F32: 1e-4}
TOL_LOGITS = 1e-4
TOL_GATE = 1e-5
TOL_AUX = 1e-5


def np32(t):
    return t.detach().float().cpu().numpy()


def assert_rowwise(gpu, ref, rel, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref).max(axis=1)
    scale = np.abs(ref).max(axis=1)
    bad = err > rel * np.maximum(scale, 1e-30)
    assert not bad.any(), f"{what}: {bad.sum()} rows off, worst {np.max(err / np.maximum(scale, 1e-30)):.3e}"


def assert_maxabs(gpu, ref, rel, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err <= rel * scale, f"{what}: max|d| {err:.3e} > {rel} * max|ref| {scale:.3e}"
    return err / scale if scale else 0.0


def score_tolerance(s_ref, p_ref=None, biased=False):
    """Per-token tolerance of the selection scores that the router tolerance
    allows: scores H (no selection bias) within 1e-5 of max |H|; scores p +
    bias within the probabilities' rule, TOL_LOGITS * max p of the token."""
    if biased:
        return TOL_LOGITS * np.abs(np.asarray(p_ref)).max(axis=1)
    return 1e-5 * np.maximum(np.abs(np.asarray(s_ref)).max(axis=1), 1e-30)


def check_topk_valid(ids_gpu, s_ref, k, tol_rel=1e-5, tol=None):
    """GPU ids against reference scores: equal except where the scores tie
    within the tolerance (tol: per-token absolute values; default tol_rel *
    max |s| of the token); returns the indices of tokens whose ids differ."""
    ids_gpu = np.asarray(ids_gpu)
    T = ids_gpu.shape[0]
    diff = []
    for t in range(T):
        s = s_ref[t]
        order = sorted(range(len(s)), key=lambda e: (-s[e], e))[:k]
        if list(ids_gpu[t]) == order:
            continue
        tol_t = tol_rel * max(np.abs(s).max(), 1e-30) if tol is None else float(tol[t])
        chosen = list(ids_gpu[t])
        assert len(set(chosen)) == k, f"token {t}: repeated ids {chosen}"
        # the GPU order must be non-increasing in the reference scores up to tol,
        # and nothing left out may beat the last chosen score by more than tol
        for a, b in zip(chosen, chosen[1:]):
            assert s[a] >= s[b] - tol_t, f"token {t}: order {chosen} vs scores"
        rest = [e for e in range(len(s)) if e not in chosen]
        if rest:
            assert max(s[e] for e in rest) <= min(s[e] for e in chosen) + tol_t, \
                f"token {t}: ids {chosen} are not a top-{k} (ref {order})"
        diff.append(t)
    return diff


def oracle_noise(wl, inp):
    """The router noise of a workload on the host, as the oracle takes it: the
    passed-in tensor, or, when the library draws it (noise_draw), the oracle's
    own draws for the same (seed, counter). None for a router without noise."""
    import oracle
    c = wl.cfg
    if inp["noise"] is not None:
        return inp["noise"].cpu()
    if not wl.noisy:
        return None
    eps = oracle.draw_noise(c.T, c.n_experts, c.noise_seed, c.noise_counter)
    return torch.from_numpy(eps.astype(np.float32))


def layer_outputs(wl, inp, device):
    c = wl.cfg
    T, E, k, d = c.T, c.n_experts, c.top_k, c.d_model
    out = {
        "y": torch.empty((T, d), dtype=c.torch_dtype, device=device),
        "ids": torch.empty((T, k), dtype=torch.int32, device=device),
        "w": torch.empty((T, k), dtype=torch.float32, device=device),
        "counts": torch.empty(E, dtype=torch.int32, device=device),
        "aux_vecs": torch.empty((3, E), dtype=torch.float32, device=device),
        "out3": torch.empty(3, dtype=torch.float32, device=device),
    }
    return out


def run_layer(wl, inp, device, ws=None):
    c = wl.cfg
    if ws is None:
        ws = moe.workspace(c, device)
    o = layer_outputs(wl, inp, device)
    moe.moe_layer_fwd(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                      inp["sel_bias"], inp["W1"], inp["W2"], inp["W1s"], inp["W2s"], o["y"],
                      o["ids"], o["w"], o["counts"], o["aux_vecs"], o["out3"], ws)
    st = moe.moe_read_device_error(c, ws)
    assert st == 0, moe.moe_status_string(st)
    return o, ws


def layer_vs_oracle(wl, device, inp=None):
    """Run moe_layer_fwd on workload `wl` and compare y on every token with
    the oracle fed the GPU's routing (identical router outputs): capacity,
    expert FFNs and combine are the oracle's. Returns (outputs, inputs)."""
    import oracle
    from sparse_mixture_experts_69_b300.workloads import make_inputs

    c = wl.cfg
    if inp is None:
        inp = make_inputs(wl, device)
    T, E, d, nc = c.T, c.n_experts, c.d_model, c.n_cand
    y = torch.empty((T, d), dtype=c.torch_dtype, device=device)
    ids = torch.empty((T, nc), dtype=torch.int32, device=device)
    w = torch.empty((T, nc), device=device)
    counts = torch.empty(E, dtype=torch.int32, device=device)
    ws = moe.workspace(c, device)
    moe.moe_layer_fwd(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                      inp["sel_bias"], inp["W1"], inp["W2"], inp["W1s"], inp["W2s"], y, ids, w,
                      counts, None, None, ws)
    st = moe.moe_read_device_error(c, ws)
    assert st == 0, moe.moe_status_string(st)
    ids_h = ids.cpu().numpy()
    C, _ = moe.moe_capacity(c)
    cap = oracle.capacity_policy(ids_h, c.top_k, E, C, priority=c.priority,
                                 pad=bool(c.pad_to_capacity))
    np.testing.assert_array_equal(counts.cpu().numpy(), cap["counts"])
    rd = oracle.ROUND_BF16 if c.dtype == moe.MOE_BF16 else oracle.ROUND_F32
    cpu = lambda t: None if t is None else t.cpu()
    W1, W2, W1s, W2s = cpu(inp["W1"]), cpu(inp["W2"]), cpu(inp["W1s"]), cpu(inp["W2s"])
    O, Os = oracle.ffn_for_tokens(cpu(inp["x"]), list(range(T)), ids_h, cap["slot"],
                                  lambda e: W1[e], lambda e: W2[e], c.act, rd, c.n_shared,
                                  (lambda s: W1s[s]) if c.n_shared else None,
                                  (lambda s: W2s[s]) if c.n_shared else None)
    y_ref = oracle.combine(np.asarray(np32(w), np.float64), cap["slot"], O, Os, rd)
    assert_maxabs(np32(y), y_ref, TOL_Y[c.dtype], "y")
    return dict(y=y, ids=ids, w=w, counts=counts, slot=cap["slot"], y_ref=y_ref), inp
