"""GPU parity of the next rows: candidate routing, overflow policies
(re-routing, rank priority, padding to capacity), expert-choice routing and
sequence-level statistics, each against the CPU oracle on the same seeded
inputs. Integer outputs are compared bit for bit; floating-point ones with
the tolerances of gpu_helpers."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs

from gpu_helpers import (TOL_AUX, TOL_GATE, TOL_LOGITS, TOL_Y, assert_maxabs, assert_rowwise,
                         np32, oracle_noise)

pytestmark = pytest.mark.gpu


def _cands(T, E, n, seed, skew=1.0):
    """n distinct experts per token, skewed towards low ids so experts overflow."""
    s = synth.uniform((T, E), seed, 300, 0.0, 1.0) + skew * torch.linspace(1.0, 0.0, E)
    return torch.argsort(-s, dim=1, stable=True)[:, :n].to(torch.int32).contiguous()


def _probs(T, E, seed, step=0.0):
    z = synth.normal((T, E), seed, 301)
    if step:  # coarse logits: many equal probabilities
        z = torch.round(z / step) * step
    return torch.softmax(z.double(), dim=1).float().contiguous()


# --------------------------------------------------------------- candidates

def test_route_candidates_from_scores(cuda_device):
    T, E, k, r = 1000, 64, 2, 3
    cfg = moe.Config(T=T, d_model=64, n_experts=E, top_k=k, d_ff=64, reroute=r)
    s = torch.floor(synth.uniform((T, E), 3, 310, 0.0, 6.0)).contiguous()  # ties
    p = _probs(T, E, 3)
    dev = cuda_device
    ids = torch.empty((T, k + r), dtype=torch.int32, device=dev)
    w = torch.empty((T, k + r), device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_route(cfg, None, None, None, None, None, None, None, p.to(dev), s.to(dev), ids, w, 1,
                  ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    ids_ref, w_ref = oracle.select_candidates(s, p, k, k + r)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(np32(w), w_ref, rtol=TOL_GATE)


# --------------------------------------------------------- overflow policies

def _dispatch(cfg, ids, dev, d=64):
    T, E = cfg.T, cfg.n_experts
    C, R_max = moe.moe_capacity(cfg)
    x = synth.normal((T, d), 7, 320, 1.0, torch.bfloat16, dev)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               kept=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               slot=torch.empty(ids.shape, dtype=torch.int32, device=dev),
               xp=torch.full((R_max, d), 7.0, dtype=torch.bfloat16, device=dev),
               row_token=torch.full((R_max,), -2, dtype=torch.int32, device=dev))
    ws = moe.workspace(cfg, dev)
    moe.moe_dispatch(cfg, x, ids.to(dev), out["counts"], out["kept"], out["offsets"], out["slot"],
                     out["xp"], out["row_token"], ws)
    st = moe.moe_read_device_error(cfg, ws)
    assert st == 0, moe.moe_status_string(st)
    return x, out, C


@pytest.mark.parametrize("T,E,k,r,cf,priority,pad", [
    (9000, 8, 2, 2, 1.0, 0, 0),        # several chunks per CTA, ragged tail
    (9000, 8, 2, 2, 1.0, 1, 0),
    (9000, 64, 1, 3, 1.0, 0, 1),
    (8192, 64, 1, 1, 1.0, 0, 0),       # Switch shape
    (8192, 64, 1, 1, 1.0, 1, 0),
    (8192, 256, 8, 2, 1.0, 0, 0),      # DeepSeek shape
    (8192, 256, 8, 2, 1.0, 1, 1),
    (8192, 64, 2, 0, 1.0, 1, 0),       # rank priority without re-routing
    (8192, 64, 2, 0, 1.25, 0, 1),      # plain dropping, padded
    (1, 4, 1, 1, 1.0, 0, 0),           # one token
    (37, 5, 2, 3, 0.1, 1, 1),          # every expert a candidate, C = 1
    (131072, 512, 2, 1, 1.0, 1, 0),    # largest supported T and E
])
def test_policy_capacity_bit_exact(cuda_device, T, E, k, r, cf, priority, pad):
    cfg = moe.Config(T=T, d_model=64, n_experts=E, top_k=k, d_ff=64, capacity_factor=cf,
                     reroute=r, priority=priority, pad_to_capacity=pad)
    ids = _cands(T, E, k + r, seed=T + E + r)
    x, o, C = _dispatch(cfg, ids, cuda_device)
    ref = oracle.capacity_policy(ids.numpy(), k, E, C, priority=priority, pad=bool(pad))
    for name in ("counts", "kept", "offsets", "slot"):
        np.testing.assert_array_equal(o[name].cpu().numpy(), ref[name], err_msg=name)
    R = int(ref["offsets"][-1])
    rt = o["row_token"].cpu().numpy()[:R]
    xp = o["xp"][:R].cpu()
    xh = x.cpu()
    if pad:
        for e in range(E):
            kept = int(ref["kept"][e])
            np.testing.assert_array_equal(rt[e * C:e * C + kept], ref["row_token"][e * C:e * C + kept])
            assert (xp[e * C + kept:(e + 1) * C] == 0).all(), f"padding rows of expert {e}"
            assert torch.equal(xp[e * C:e * C + kept], xh[torch.as_tensor(rt[e * C:e * C + kept]).long()])
    else:
        np.testing.assert_array_equal(rt, ref["row_token"])
        assert torch.equal(xp, xh[torch.as_tensor(rt).long()])


def _layer_policy(wl, cfg, dev, rd):
    """Run the layer with an overflow policy; check routing, then y against the
    oracle fed the GPU's candidates and gates (identical router outputs)."""
    inp = make_inputs(wl, dev)
    T, E, d, nc = cfg.T, cfg.n_experts, cfg.d_model, cfg.n_cand
    y = torch.empty((T, d), dtype=cfg.torch_dtype, device=dev)
    ids = torch.empty((T, nc), dtype=torch.int32, device=dev)
    w = torch.empty((T, nc), device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_layer_fwd(cfg, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                      inp["sel_bias"], inp["W1"], inp["W2"], inp["W1s"], inp["W2s"], y, ids, w,
                      counts, None, None, ws)
    st = moe.moe_read_device_error(cfg, ws)
    assert st == 0, moe.moe_status_string(st)
    ids_h = ids.cpu().numpy()
    C, _ = moe.moe_capacity(cfg)
    cap = oracle.capacity_policy(ids_h, cfg.top_k, E, C, priority=cfg.priority,
                                 pad=bool(cfg.pad_to_capacity))
    np.testing.assert_array_equal(counts.cpu().numpy(), cap["counts"])
    tok = list(range(T))
    W1 = lambda e: inp["W1"][e]
    W2 = lambda e: inp["W2"][e]
    W1s = (lambda s: inp["W1s"][s]) if cfg.n_shared else None
    W2s = (lambda s: inp["W2s"][s]) if cfg.n_shared else None
    O, Os = oracle.ffn_for_tokens(inp["x"], tok, ids_h, cap["slot"], W1, W2, cfg.act, rd,
                                  cfg.n_shared, W1s, W2s)
    y_ref = oracle.combine(np.asarray(np32(w), np.float64), cap["slot"], O, Os, rd)
    assert_maxabs(np32(y), y_ref, TOL_Y[cfg.dtype], "y")
    return cap


@pytest.mark.parametrize("priority,pad", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_layer_reroute_fp32(cuda_device, priority, pad):
    wl = WORKLOADS["tiny"].with_(reroute=2, priority=priority, pad_to_capacity=pad)
    cap = _layer_policy(wl, wl.cfg, cuda_device, oracle.ROUND_F32)
    # every expert overflows in this workload: all E*C rows are taken
    assert (cap["slot"] >= 0).sum() == 320


@pytest.mark.parametrize("priority,pad", [(0, 1), (1, 0)])
def test_layer_reroute_bf16(cuda_device, priority, pad):
    wl = WORKLOADS["deepseek"].with_(T=300, d_model=256, n_experts=16, top_k=2, d_ff=128,
                                     capacity_factor=1.0, reroute=2, priority=priority,
                                     pad_to_capacity=pad, bias_rate=0.0)
    _layer_policy(wl, wl.cfg, cuda_device, oracle.ROUND_BF16)


# ------------------------------------------------------------- expert choice

@pytest.mark.parametrize("T,E,cf,step", [
    (5000, 64, 2.0, 0.25),     # coarse logits: ties decided by token index
    (32768, 8, 1.0, 0.0),      # largest supported T
    (300, 16, 16.0, 0.0),      # C = T: every expert takes every token
    (77, 5, 0.1, 0.5),         # C = 2
])
def test_expert_choice_dispatch_bit_exact(cuda_device, T, E, cf, step):
    dev = cuda_device
    cfg = moe.Config(T=T, d_model=64, n_experts=E, top_k=1, d_ff=64, capacity_factor=cf,
                     routing=moe.MOE_EXPERT_CHOICE)
    C, R = moe.moe_capacity(cfg)
    p = _probs(T, E, T + E, step)
    x = synth.normal((T, 64), 9, 330, 1.0, torch.bfloat16, dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_token = torch.empty(R, dtype=torch.int32, device=dev)
    row_w = torch.empty(R, device=dev)
    tok_row = torch.empty((T, E), dtype=torch.int32, device=dev)
    xp = torch.empty((R, 64), dtype=torch.bfloat16, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_expert_choice_dispatch(cfg, x, p.to(dev), offsets, row_token, row_w, tok_row, xp, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    ref = oracle.expert_choice(p.numpy(), C)
    np.testing.assert_array_equal(offsets.cpu().numpy(), np.arange(E + 1) * C)
    np.testing.assert_array_equal(row_token.cpu().numpy(), ref["row_token"])
    np.testing.assert_array_equal(tok_row.cpu().numpy(), ref["tok_row"])
    np.testing.assert_array_equal(np32(row_w), ref["row_w"].astype(np.float32))
    assert torch.equal(xp.cpu(), x.cpu()[row_token.cpu().long()])


def test_expert_choice_combine(cuda_device):
    dev = cuda_device
    T, E, d, S, cf = 3000, 16, 256, 1, 2.0
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=1, d_ff=64, n_shared=S, capacity_factor=cf,
                     routing=moe.MOE_EXPERT_CHOICE)
    C, R = moe.moe_capacity(cfg)
    p = _probs(T, E, 5)
    ref = oracle.expert_choice(p.numpy(), C)
    yp = synth.normal((R, d), 5, 340, 1.0, torch.bfloat16, dev)
    ys = synth.normal((S, T, d), 5, 341, 1.0, torch.bfloat16, dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_expert_choice_combine(cfg, yp, torch.as_tensor(ref["tok_row"]).to(dev), p.to(dev), ys,
                                  y, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    y_ref = oracle.combine_expert_choice(ref["tok_row"], p.numpy(), np32(yp).astype(np.float64),
                                         np32(ys).astype(np.float64), oracle.ROUND_BF16)
    assert_maxabs(np32(y), y_ref, 1e-2, "y")


@pytest.mark.parametrize("name,over", [
    ("tiny", dict(capacity_factor=2.0)),
    ("deepseek", dict(T=2048, d_model=256, n_experts=16, top_k=1, d_ff=128, capacity_factor=2.0,
                      sel_bias=False, bias_rate=0.0)),
])
def test_layer_expert_choice(cuda_device, name, over):
    dev = cuda_device
    wl = WORKLOADS[name].with_(routing=moe.MOE_EXPERT_CHOICE, **over)
    cfg = wl.cfg
    inp = make_inputs(wl, dev)
    T, E, d = cfg.T, cfg.n_experts, cfg.d_model
    C, R = moe.moe_capacity(cfg)
    y = torch.empty((T, d), dtype=cfg.torch_dtype, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_layer_fwd(cfg, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                      inp["sel_bias"], inp["W1"], inp["W2"], inp["W1s"], inp["W2s"], y, None, None,
                      None, None, None, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    # identical router outputs: the oracle selects on the GPU's probabilities
    probs = torch.empty((T, E), device=dev)
    logits = torch.empty((T, E), device=dev)
    moe.moe_route(cfg, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                  inp["sel_bias"], logits, probs, None, None, None, 0, ws)
    r = oracle.router(inp["x"], inp["Wg"], 1, Wnoise=inp["Wnoise"], noise=oracle_noise(wl, inp),
                      offset=inp["logit_offset"], bias=inp["sel_bias"])
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    p_h = np32(probs)
    ref = oracle.expert_choice(p_h, C)
    rd = oracle.ROUND_BF16 if cfg.dtype == moe.MOE_BF16 else oracle.ROUND_F32
    O = np.zeros((R, d))
    for e in range(E):
        rows = ref["row_token"][e * C:(e + 1) * C]
        O[e * C:(e + 1) * C] = oracle.expert_ffn(inp["x"][torch.as_tensor(rows).long()],
                                                 inp["W1"][e], inp["W2"][e], cfg.act, rd)
    Os = None
    if cfg.n_shared:
        Os = np.stack([oracle.expert_ffn(inp["x"], inp["W1s"][s], inp["W2s"][s], cfg.act, rd)
                       for s in range(cfg.n_shared)])
    y_ref = oracle.combine_expert_choice(ref["tok_row"], p_h, O, Os, rd)
    assert_maxabs(np32(y), y_ref, TOL_Y[cfg.dtype], "y")


# ------------------------------------------------- sequence-level statistics

def test_seq_stats(cuda_device):
    dev = cuda_device
    T, E, k, r = 8192, 64, 2, 1
    cfg = moe.Config(T=T, d_model=64, n_experts=E, top_k=k, d_ff=64, reroute=r)
    lens = [0, 1, 7, 1000, 3000, 0, 4184]
    offs = torch.as_tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    assert int(offs[-1]) == T
    n = len(lens)
    p = _probs(T, E, 11)
    ids = _cands(T, E, k + r, 12)
    f = torch.empty((n, E), device=dev)
    P = torch.empty((n, E), device=dev)
    aux = torch.empty(n, device=dev)
    mean = torch.empty(1, device=dev)
    ws = moe.workspace(cfg, dev)
    outs = []
    for _ in range(2):
        moe.moe_seq_aux_stats(cfg, p.to(dev), ids.to(dev), offs.to(dev), n, f, P, aux, mean, ws)
        assert moe.moe_read_device_error(cfg, ws) == 0
        outs.append([t.clone() for t in (f, P, aux, mean)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)  # deterministic
    ref = oracle.seq_aux_stats(p.numpy(), ids.numpy(), k, offs.numpy())
    np.testing.assert_allclose(np32(f), ref["f"], rtol=TOL_AUX, atol=1e-7)
    np.testing.assert_allclose(np32(P), ref["P"], rtol=TOL_AUX, atol=1e-7)
    np.testing.assert_allclose(np32(aux), ref["aux"], rtol=TOL_AUX)
    assert float(mean) == pytest.approx(ref["mean"], rel=TOL_AUX)
    # a malformed offsets array is reported, not trusted
    bad = offs.clone()
    bad[3] = T + 5
    moe.moe_seq_aux_stats(cfg, p.to(dev), ids.to(dev), bad.to(dev), n, None, None, aux, mean, ws)
    assert moe.moe_read_device_error(cfg, ws) == 7  # MOE_ERR_DEVICE_ARG
