"""GPU parity of the stages that do not use the tensor cores: the float32
router, selection from given scores, capacity + dispatch, the float32 expert
FFN, combine, statistics, bias update and device-side error reporting.
Every input comes from the seeded generator; expected values come from the
CPU oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs

from gpu_helpers import (TOL_AUX, TOL_GATE, TOL_LOGITS, TOL_Y, assert_maxabs, assert_rowwise,
                         check_topk_valid, np32, run_layer)

pytestmark = pytest.mark.gpu


def _ids(T, E, k, seed, skew=0.0, device="cuda"):
    """k distinct experts per token from generator scores (optionally skewed to low ids)."""
    s = synth.uniform((T, E), seed, 200, 0.0, 1.0)
    if skew:
        s = s + skew * torch.linspace(1.0, 0.0, E)
    return torch.argsort(-s, dim=1, stable=True)[:, :k].to(torch.int32).contiguous().to(device)


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("T,d,E,k,noisy,offset,bias", [
    (256, 128, 8, 2, False, False, False),
    (300, 64, 64, 1, True, False, False),
    (97, 128, 256, 8, False, False, True),
    (33, 64, 1000, 4, False, True, False),
])
def test_router_f32(cuda_device, T, d, E, k, noisy, offset, bias):
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=64, dtype=moe.MOE_F32,
                     act=moe.MOE_GELU)
    x = synth.normal((T, d), 1, 101)
    Wg = synth.normal((d, E), 1, 102, 0.1)
    Wn = synth.normal((d, E), 1, 103, 0.1) if noisy else None
    noise = synth.normal((T, E), 1, 104) if noisy else None
    off = synth.zipf_logit_offset(E, 1.2) if offset else None
    b = synth.uniform((E,), 1, 105, -0.1, 0.1) if bias else None
    dev = cuda_device
    g = lambda t: None if t is None else t.to(dev)
    logits = torch.empty((T, E), device=dev)
    probs = torch.empty((T, E), device=dev)
    sel = torch.empty((T, E), device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_route(cfg, g(x), g(Wg), g(Wn), g(noise), g(off), g(b), logits, probs, sel, ids, w, 0, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    r = oracle.router(x, Wg, k, Wnoise=Wn, noise=noise, offset=off, bias=b)
    assert_rowwise(np32(logits), r["z"], TOL_LOGITS, "logits")
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    assert_rowwise(np32(sel), r["s"], TOL_LOGITS, "sel_scores")
    diff = check_topk_valid(ids.cpu().numpy(), r["s"], k)
    same = [t for t in range(T) if t not in diff]
    assert_rowwise(np32(w)[same], r["w"][same], TOL_LOGITS, "gates")


@pytest.mark.parametrize("T,E,seed,counter", [(1, 1, 0, 0), (1000, 300, 0x5EED, 7),
                                               (8192, 64, 2**64 - 1, 2**40 + 3)])
def test_draw_noise_matches_oracle(cuda_device, T, E, seed, counter):
    """moe_draw_noise against the oracle's Philox4x32-10 + Box-Muller draws:
    the 24-bit uniforms are integers on both sides, so only the float32 log,
    square root and cosine differ from the double ones."""
    cfg = moe.Config(T=T, d_model=8, n_experts=E, top_k=1, d_ff=8, noise_draw=1,
                     noise_seed=seed, noise_counter=counter)
    eps = torch.empty((T, E), device=cuda_device)
    moe.moe_draw_noise(cfg, eps)
    ref = oracle.draw_noise(T, E, seed, counter)
    err = np.abs(np32(eps) - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() < 2e-6, err.max()


@pytest.mark.parametrize("T,d,E,k,dtype", [(300, 64, 64, 1, moe.MOE_F32),
                                           (1000, 128, 32, 2, moe.MOE_BF16)])
def test_router_with_drawn_noise(cuda_device, T, d, E, k, dtype):
    """noise_draw = 1: the selection kernel draws eps itself; probs, scores and
    the top-k match the oracle router fed the oracle's draws, and passing
    moe_draw_noise's output in as the noise tensor routes bit for bit alike."""
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=64, dtype=dtype,
                     act=moe.MOE_GELU, noise_draw=1, noise_seed=99, noise_counter=5)
    td = cfg.torch_dtype
    x = synth.normal((T, d), 1, 101, 1.0, td)
    Wg = synth.normal((d, E), 1, 102, 0.1, td)
    Wn = synth.normal((d, E), 1, 103, 0.1, td)
    dev = cuda_device
    logits = torch.empty((T, E), device=dev)
    probs = torch.empty((T, E), device=dev)
    sel = torch.empty((T, E), device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_route(cfg, x.to(dev), Wg.to(dev), Wn.to(dev), None, None, None, logits, probs, sel,
                  ids, w, 0, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    noise = torch.from_numpy(oracle.draw_noise(T, E, 99, 5).astype(np.float32))
    r = oracle.router(x.float(), Wg.float(), k, Wnoise=Wn.float(), noise=noise)
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    assert_rowwise(np32(sel), r["s"], TOL_LOGITS, "sel_scores")
    check_topk_valid(ids.cpu().numpy(), r["s"], k)
    cfg_in = moe.Config(**{**cfg.__dict__, "noise_draw": 0})
    eps = torch.empty((T, E), device=dev)
    moe.moe_draw_noise(cfg, eps)
    ids2 = torch.empty_like(ids)
    w2 = torch.empty_like(w)
    moe.moe_route(cfg_in, x.to(dev), Wg.to(dev), Wn.to(dev), eps, None, None, logits, probs, sel,
                  ids2, w2, 0, ws)
    assert torch.equal(ids2, ids) and torch.equal(w2, w)


def test_noise_arguments_are_checked(cuda_device):
    """With noise_draw = 1 a noise tensor is refused; without Wnoise the router
    has no noise term and the call runs."""
    cfg = moe.Config(T=16, d_model=8, n_experts=4, top_k=1, d_ff=8, noise_draw=1)
    dev = cuda_device
    x = torch.zeros((16, 8), dtype=torch.bfloat16, device=dev)
    Wg = torch.zeros((8, 4), dtype=torch.bfloat16, device=dev)
    noise = torch.zeros((16, 4), device=dev)
    out = [torch.empty((16, 4), device=dev) for _ in range(3)]
    ids = torch.empty((16, 1), dtype=torch.int32, device=dev)
    w = torch.empty((16, 1), device=dev)
    ws = moe.workspace(cfg, dev)
    with pytest.raises(moe.MoeError):
        moe.moe_route(cfg, x, Wg, Wg, noise, None, None, *out, ids, w, 0, ws)
    moe.moe_route(cfg, x, Wg, None, None, None, None, *out, ids, w, 0, ws)


@pytest.mark.parametrize("T,E,k,renorm", [(1, 5, 2, 1), (513, 8, 2, 1), (200, 64, 1, 1),
                                          (129, 256, 8, 1), (64, 300, 32, 0), (40, 7, 7, 1)])
def test_select_from_scores_bit_exact(cuda_device, T, E, k, renorm):
    """Identical scores in, identical ids out: small integer scores force many
    ties, which the lower index must win on both sides."""
    cfg = moe.Config(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, renorm_topk=renorm,
                     dtype=moe.MOE_F32)
    s = synth.randint((T, E), 2, 110, 4).float()
    p = synth.uniform((T, E), 2, 111, 0.01, 1.0)
    dev = cuda_device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_route(cfg, None, None, None, None, None, None, None, p.to(dev), s.to(dev), ids, w, 1, ws)
    ref_ids, ref_w = oracle.select(s, p, k, renorm=bool(renorm))
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(np32(w), ref_w, rtol=TOL_GATE)


def test_softmax_example_on_gpu(cuda_device):
    """The pages' 10-logit example through the router: fp32 logits keep the
    -0.5 gap (top score 1/(1+9e^-0.5)); bf16 weights lose it (top score 1/10)."""
    dev = cuda_device
    E, d = 10, 8
    Wg = torch.zeros((d, E))
    Wg[0, :] = 128.0
    Wg[0, 0] = 128.5
    x = torch.zeros((1, d))
    x[0, 0] = 1.0
    exact = 1.0 / (1.0 + 9.0 * np.exp(-0.5))
    for dtype, expect in [(moe.MOE_F32, exact), (moe.MOE_BF16, 0.1)]:
        cfg = moe.Config(T=1, d_model=d, n_experts=E, top_k=1, d_ff=8, dtype=dtype)
        tdt = cfg.torch_dtype
        logits = torch.empty((1, E), device=dev)
        probs = torch.empty((1, E), device=dev)
        ids = torch.empty((1, 1), dtype=torch.int32, device=dev)
        w = torch.empty((1, 1), device=dev)
        ws = moe.workspace(cfg, dev)
        moe.moe_route(cfg, x.to(tdt).to(dev), Wg.to(tdt).to(dev), None, None, None, None, logits,
                      probs, None, ids, w, 0, ws)
        p0 = probs[0, 0].item()
        assert abs(p0 - expect) / expect < 1e-6, (dtype, p0, expect)
    assert 0.33 < (exact - 0.1) / exact < 0.39


# ------------------------------------------------------------ capacity, dispatch

@pytest.mark.parametrize("T,E,k,cf,d,dtype,skew", [
    (256, 8, 2, 1.25, 128, moe.MOE_F32, 0.0),
    (8192, 64, 1, 1.0, 64, moe.MOE_BF16, 0.3),
    (1, 4, 2, 1.0, 16, moe.MOE_BF16, 0.0),
    (1000, 1, 1, 0.5, 8, moe.MOE_BF16, 0.0),
    (777, 16, 16, 1.0, 24, moe.MOE_F32, 0.0),
    (3000, 256, 8, 0.0, 32, moe.MOE_BF16, 2.0),
    (513, 1000, 3, 2.0, 8, moe.MOE_BF16, 0.0),
])
def test_dispatch_bit_exact(cuda_device, T, E, k, cf, d, dtype, skew):
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=8, capacity_factor=cf,
                     dtype=dtype)
    C, R_max = moe.moe_capacity(cfg)
    assert C == oracle.capacity_of(T, E, cf) or (cf > 0 and C == T)
    dev = cuda_device
    ids = _ids(T, E, k, 3, skew, dev)
    x = synth.normal((T, d), 3, 120, 1.0, cfg.torch_dtype, dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    kept = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, k), dtype=torch.int32, device=dev)
    xp = torch.zeros((R_max, d), dtype=cfg.torch_dtype, device=dev)
    row_token = torch.full((R_max,), -7, dtype=torch.int32, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_dispatch(cfg, x, ids, counts, kept, offsets, slot, xp, row_token, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    ref = oracle.capacity(ids.cpu(), E, C)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(kept.cpu().numpy(), ref["kept"])
    np.testing.assert_array_equal(offsets.cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(slot.cpu().numpy(), ref["slot"])
    R = int(ref["offsets"][-1])
    np.testing.assert_array_equal(row_token[:R].cpu().numpy(), ref["row_token"])
    xp_ref = oracle.dispatch(x.cpu(), ref["slot"], R)
    np.testing.assert_array_equal(np32(xp[:R]), xp_ref)


def test_dispatch_flags_bad_ids(cuda_device):
    cfg = moe.Config(T=64, d_model=8, n_experts=4, top_k=2, d_ff=8, dtype=moe.MOE_BF16)
    dev = cuda_device
    ids = _ids(64, 4, 2, 4, 0.0, dev)
    ids[5, 1] = 9  # out of range
    _, R_max = moe.moe_capacity(cfg)
    ws = moe.workspace(cfg, dev)
    z = lambda n, dt=torch.int32: torch.zeros(n, dtype=dt, device=dev)
    moe.moe_dispatch(cfg, torch.zeros((64, 8), dtype=torch.bfloat16, device=dev), ids, z(4), z(4),
                     z(5), z((64, 2)), torch.zeros((R_max, 8), dtype=torch.bfloat16, device=dev),
                     z(R_max), ws)
    assert moe.moe_read_device_error(cfg, ws) == 7  # MOE_ERR_DEVICE_ARG
    assert moe.moe_read_device_error(cfg, ws) == 0  # reading clears it


# -------------------------------------------------------------- expert FFN, fp32

def _offsets_from_counts(counts):
    off = np.zeros(len(counts) + 1, np.int32)
    off[1:] = np.cumsum(counts)
    return off


def run_ffn(cfg, counts, seed, dev):
    """moe_expert_ffn on generator rows with the given per-expert row counts."""
    E, d, F, F1, S, T = cfg.n_experts, cfg.d_model, cfg.d_ff, cfg.F1, cfg.n_shared, cfg.T
    dt = cfg.torch_dtype
    _, R_max = moe.moe_capacity(cfg)
    off = _offsets_from_counts(counts)
    R = int(off[-1])
    assert R <= R_max
    xp = synth.normal((R_max, d), seed, 130, 1.0, dt, dev)
    W1 = synth.normal((E, F1, d), seed, 131, 0.05, dt, dev)
    W2 = synth.normal((E, d, F), seed, 132, 0.05, dt, dev)
    x = synth.normal((T, d), seed, 133, 1.0, dt, dev) if S else None
    W1s = synth.normal((S, F1, d), seed, 134, 0.05, dt, dev) if S else None
    W2s = synth.normal((S, d, F), seed, 135, 0.05, dt, dev) if S else None
    yp = torch.zeros((R_max, d), dtype=dt, device=dev)
    ys = torch.zeros((S, T, d), dtype=dt, device=dev) if S else None
    ws = moe.workspace(cfg, dev)
    moe.moe_expert_ffn(cfg, xp, torch.from_numpy(off).to(dev), W1, W2, x, W1s, W2s, yp, ys, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    rd = oracle.ROUND_BF16 if cfg.dtype == moe.MOE_BF16 else oracle.ROUND_F32
    xpc = xp.cpu()
    for e in range(E):
        if counts[e] == 0:
            continue
        ref = oracle.expert_ffn(xpc[off[e]:off[e + 1]], W1[e].cpu(), W2[e].cpu(), cfg.act, rd)
        assert_maxabs(np32(yp[off[e]:off[e + 1]]), ref, TOL_Y[cfg.dtype] / 2, f"expert {e}")
    for s in range(S):
        ref = oracle.expert_ffn(x.cpu(), W1s[s].cpu(), W2s[s].cpu(), cfg.act, rd)
        assert_maxabs(np32(ys[s]), ref, TOL_Y[cfg.dtype] / 2, f"shared {s}")


@pytest.mark.parametrize("act", [moe.MOE_RELU, moe.MOE_GELU, moe.MOE_SWIGLU])
def test_expert_ffn_f32(cuda_device, act):
    cfg = moe.Config(T=70, d_model=72, n_experts=5, top_k=2, d_ff=136, n_shared=1,
                     dtype=moe.MOE_F32, act=act)
    run_ffn(cfg, [0, 1, 65, 70, 3], 5, cuda_device)


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("dtype,S", [(moe.MOE_F32, 0), (moe.MOE_BF16, 2)])
def test_combine(cuda_device, dtype, S):
    T, E, k, d, cf = 300, 8, 3, 64, 1.0
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=8, n_shared=S,
                     capacity_factor=cf, dtype=dtype)
    dev = cuda_device
    C, R_max = moe.moe_capacity(cfg)
    ids = _ids(T, E, k, 6, 1.0, "cpu")
    cap = oracle.capacity(ids, E, C)
    assert (cap["slot"] < 0).any()  # some drops
    dt = cfg.torch_dtype
    yp = synth.normal((R_max, d), 6, 140, 1.0, dt, dev)
    ys = synth.normal((S, T, d), 6, 141, 1.0, dt, dev) if S else None
    w = synth.uniform((T, k), 6, 142, 0.0, 1.0)
    y = torch.empty((T, d), dtype=dt, device=dev)
    ws = moe.workspace(cfg, dev)
    slot = torch.from_numpy(cap["slot"]).to(dev)
    moe.moe_combine(cfg, yp, slot, w.to(dev), ys, y, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    ypc = yp.cpu().double().numpy()
    O = np.zeros((T, k, d))
    for t in range(T):
        for j in range(k):
            if cap["slot"][t, j] >= 0:
                O[t, j] = ypc[cap["slot"][t, j]]
    rd = oracle.ROUND_BF16 if dtype == moe.MOE_BF16 else oracle.ROUND_F32
    ref = oracle.combine(w.double().numpy(), cap["slot"], O,
                         None if ys is None else ys.cpu().double().numpy(), rd)
    assert_maxabs(np32(y), ref, TOL_Y[dtype] / 4, "combine")


# ---------------------------------------------------------------- statistics

@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (8192, 64, 1), (1000, 256, 8), (5, 3, 3)])
def test_aux_stats(cuda_device, T, E, k):
    cfg = moe.Config(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, dtype=moe.MOE_BF16,
                     importance_weight=0.01)
    dev = cuda_device
    logits = synth.normal((T, E), 7, 150)
    p = torch.softmax(logits.double(), dim=1).float()
    ids = _ids(T, E, k, 7, 0.5, "cpu")
    w = synth.uniform((T, k), 7, 151, 0.0, 1.0)
    f = torch.empty(E, device=dev)
    P = torch.empty(E, device=dev)
    I = torch.empty(E, device=dev)
    out3 = torch.empty(3, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_aux_stats(cfg, p.to(dev), ids.to(dev), w.to(dev), f, P, I, out3, ws)
    ref = oracle.aux_stats(p, ids, w, E, 0.01)
    np.testing.assert_allclose(np32(f), ref["f"], rtol=1e-6)
    np.testing.assert_allclose(np32(P), ref["P"], rtol=TOL_AUX)
    np.testing.assert_allclose(np32(I), ref["I"], rtol=TOL_AUX)
    o = np32(out3)
    assert o[0] == pytest.approx(ref["aux"], rel=TOL_AUX)
    assert o[1] == pytest.approx(ref["cv2"], rel=TOL_AUX)
    assert o[2] == pytest.approx(ref["L_imp"], rel=TOL_AUX)


def test_bias_update_bit_exact(cuda_device):
    T, E, k = 8192, 256, 8
    cfg = moe.Config(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, dtype=moe.MOE_BF16)
    dev = cuda_device
    counts = synth.randint((E,), 8, 160, 2 * T * k // E).to(torch.int32)
    counts[:4] = T * k // E  # exactly at the mean: unchanged
    bias = synth.uniform((E,), 8, 161, -0.1, 0.1)
    b = bias.to(dev)
    moe.moe_bias_update(cfg, counts.to(dev), b, 1e-3)
    ref = oracle.bias_update(counts, bias, T, k, 1e-3)
    np.testing.assert_array_equal(b.cpu().numpy(), ref)


# ---------------------------------------------------------------- tiny layer

def test_tiny_layer_full_parity(cuda_device):
    """The fp32 Tiny workload end to end against the oracle's own full
    evaluation (routing, capacity with drops, experts, combine, statistics)."""
    wl = WORKLOADS["tiny"]
    c = wl.cfg
    inp = make_inputs(wl, cuda_device)
    o, ws = run_layer(wl, inp, cuda_device)
    cpu = {k2: (None if v is None else v.cpu()) for k2, v in inp.items()}
    r = oracle.router(cpu["x"], cpu["Wg"], c.top_k)
    diff = check_topk_valid(o["ids"].cpu().numpy(), r["s"], c.top_k)
    assert not diff, f"near-tie routing differences at tokens {diff}"
    assert_rowwise(np32(o["w"]), r["w"], TOL_LOGITS, "gates")
    C, _ = moe.moe_capacity(c)
    cap = oracle.capacity(r["ids"], c.n_experts, C)
    np.testing.assert_array_equal(o["counts"].cpu().numpy(), cap["counts"])
    assert (cap["slot"] < 0).sum() == 192  # every expert overflows: 192 of 512 dropped
    O, _ = oracle.ffn_for_tokens(cpu["x"], list(range(c.T)), r["ids"], cap["slot"],
                                 lambda e: cpu["W1"][e], lambda e: cpu["W2"][e], c.act,
                                 oracle.ROUND_F32)
    y_ref = oracle.combine(r["w"], cap["slot"], O, None, oracle.ROUND_F32)
    assert_maxabs(np32(o["y"]), y_ref, TOL_Y[c.dtype], "y")
    st = oracle.aux_stats(r["p"].astype(np.float32), r["ids"], r["w"].astype(np.float32),
                          c.n_experts, c.importance_weight)
    o3 = np32(o["out3"])
    assert o3[0] == pytest.approx(st["aux"], rel=TOL_AUX)
    assert o3[1] == pytest.approx(st["cv2"], rel=TOL_AUX)
    av = np32(o["aux_vecs"])
    np.testing.assert_allclose(av[0], st["f"], rtol=1e-6)
    np.testing.assert_allclose(av[1], st["P"], rtol=TOL_AUX)
    np.testing.assert_allclose(av[2], st["I"], rtol=TOL_AUX)
    # a second call on the same workspace (counters reset by the kernels) agrees
    o2, _ = run_layer(wl, inp, cuda_device, ws)
    for key in o:
        assert torch.equal(o[key], o2[key]), key


def test_nonfinite_input_is_reported(cuda_device):
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl, cuda_device)
    inp["x"][3, 5] = float("nan")
    c = wl.cfg
    ws = moe.workspace(c, cuda_device)
    from gpu_helpers import layer_outputs
    o = layer_outputs(wl, inp, cuda_device)
    moe.moe_layer_fwd(c, inp["x"], inp["Wg"], None, None, None, None, inp["W1"], inp["W2"], None,
                      None, o["y"], o["ids"], o["w"], o["counts"], o["aux_vecs"], o["out3"], ws)
    assert moe.moe_read_device_error(c, ws) == 5  # MOE_ERR_NONFINITE
    # the context is still usable
    o2, _ = run_layer(wl, make_inputs(wl, cuda_device), cuda_device)
    assert torch.isfinite(o2["y"].float()).all()
