"""The whole layer at the workloads' full sizes, in the launch configuration the
benchmark times (moe_layer_fwd on one stream). Routing, logits and outputs are
compared with the oracle's own evaluation: on every token where the oracle
finishes in seconds, else on seeded samples of tokens (the expert FFN of a
token depends only on its own routing when nothing is dropped)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs

from gpu_helpers import (TOL_AUX, TOL_LOGITS, TOL_Y, assert_maxabs, assert_rowwise,
                         check_topk_valid, np32, oracle_noise, run_layer)

pytestmark = pytest.mark.gpu


def _route(wl, inp, dev):
    c = wl.cfg
    T, E, k = c.T, c.n_experts, c.top_k
    logits = torch.empty((T, E), device=dev)
    probs = torch.empty((T, E), device=dev)
    sel = torch.empty((T, E), device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), device=dev)
    ws = moe.workspace(c, dev)
    moe.moe_route(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                  inp["sel_bias"], logits, probs, sel, ids, w, 0, ws)
    assert moe.moe_read_device_error(c, ws) == 0
    return logits, probs, sel, ids, w


def _cpu_rows(t, rows):
    return None if t is None else t[rows].cpu()


def _oracle_router(wl, inp, tok):
    c = wl.cfg
    tok_t = torch.as_tensor(tok)
    g = lambda n: None if inp[n] is None else inp[n].cpu()
    return oracle.router(_cpu_rows(inp["x"], tok_t), g("Wg"), c.top_k, Wnoise=g("Wnoise"),
                         noise=_cpu_rows(oracle_noise(wl, inp), tok_t), offset=g("logit_offset"),
                         bias=g("sel_bias"), renorm=bool(c.renorm_topk))


def _oracle_y(wl, inp, tok, ids, w, slot):
    c = wl.cfg
    rd = oracle.ROUND_BF16 if c.dtype == moe.MOE_BF16 else oracle.ROUND_F32
    x = inp["x"][torch.as_tensor(tok)].cpu()
    O, Os = oracle.ffn_for_tokens(x, list(range(len(tok))), ids, slot,
                                  lambda e: inp["W1"][e].cpu(), lambda e: inp["W2"][e].cpu(),
                                  c.act, rd, c.n_shared,
                                  lambda s: inp["W1s"][s].cpu(), lambda s: inp["W2s"][s].cpu())
    return oracle.combine(w, slot, O, Os, rd)


def _sample(T, n, seed):
    return sorted(set(synth.randint((n,), seed, 300, T).tolist()))


def test_switch_full(cuda_device):
    """Noisy top-1, capacity 128 with drops: every token routed by the oracle."""
    wl = WORKLOADS["switch"]
    c = wl.cfg
    inp = make_inputs(wl, cuda_device)
    o, _ = run_layer(wl, inp, cuda_device)
    logits, probs, sel, _, _ = _route(wl, inp, cuda_device)
    r = _oracle_router(wl, inp, list(range(c.T)))
    assert_rowwise(np32(logits), r["z"], TOL_LOGITS, "logits")
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    ids = o["ids"].cpu().numpy()
    diff = check_topk_valid(ids, r["s"], c.top_k)
    assert len(diff) <= 2, diff
    assert np.all(np32(o["w"]) == 1.0)  # Softmax(KeepTopK(H, 1)) = 1
    C, _ = moe.moe_capacity(c)
    cap = oracle.capacity(r["ids"], c.n_experts, C)
    dropped = int((cap["slot"] < 0).sum())
    assert 200 < dropped < 600, dropped
    touched = {int(ids[t, 0]) for t in diff} | {int(r["ids"][t, 0]) for t in diff}
    if not diff:
        np.testing.assert_array_equal(o["counts"].cpu().numpy(), cap["counts"])
    tok = [t for t in _sample(c.T, 256, 1) if int(r["ids"][t, 0]) not in touched]
    slot = cap["slot"][tok]
    y_ref = _oracle_y(wl, inp, tok, r["ids"][tok], r["w"][tok], slot)
    assert_maxabs(np32(o["y"][torch.as_tensor(tok)]), y_ref, TOL_Y[c.dtype], "y")
    # dropped tokens of top-1 routing output exactly zero
    dropped_tok = [t for t in range(c.T) if cap["slot"][t, 0] < 0 and int(r["ids"][t, 0]) not in touched]
    assert dropped_tok and float(o["y"][torch.as_tensor(dropped_tok)].abs().max()) == 0.0
    st = oracle.aux_stats(r["p"].astype(np.float32), r["ids"], r["w"].astype(np.float32),
                          c.n_experts, c.importance_weight)
    o3 = np32(o["out3"])
    assert o3[0] == pytest.approx(st["aux"], rel=TOL_AUX)
    assert o3[1] == pytest.approx(st["cv2"], rel=TOL_AUX)
    av = np32(o["aux_vecs"])
    if not diff:
        np.testing.assert_allclose(av[0], st["f"], rtol=1e-6)
        np.testing.assert_allclose(av[2], st["I"], rtol=TOL_AUX)
    np.testing.assert_allclose(av[1], st["P"], rtol=TOL_AUX)


@pytest.mark.parametrize("name,n_tok", [("mixtral", 12), ("deepseek", 8), ("decode", 16)])
def test_large_config_sampled(cuda_device, name, n_tok):
    wl = WORKLOADS[name]
    c = wl.cfg
    inp = make_inputs(wl, cuda_device)
    o, ws = run_layer(wl, inp, cuda_device)
    counts = o["counts"].cpu().numpy()
    ids_all = o["ids"].cpu().numpy()
    assert counts.sum() == c.T * c.top_k
    np.testing.assert_array_equal(counts, np.bincount(ids_all.ravel(), minlength=c.n_experts))
    logits, probs, sel, ids2, _ = _route(wl, inp, cuda_device)
    np.testing.assert_array_equal(ids2.cpu().numpy(), ids_all)  # same routing, same bits
    tok = _sample(c.T, n_tok, 2) if c.T > n_tok else list(range(c.T))
    r = _oracle_router(wl, inp, tok)
    tt = torch.as_tensor(tok)
    assert_rowwise(np32(logits[tt]), r["z"], TOL_LOGITS, "logits")
    assert_rowwise(np32(probs[tt]), r["p"], TOL_LOGITS, "probs")
    diff = check_topk_valid(ids_all[tok], r["s"], c.top_k)
    keep = [i for i in range(len(tok)) if i not in diff]
    assert_rowwise(np32(o["w"][tt])[keep], r["w"][keep], TOL_LOGITS, "gates")
    tok_k = [tok[i] for i in keep]
    slot = np.zeros((len(tok_k), c.top_k), np.int32)  # dropless: every assignment kept
    y_ref = _oracle_y(wl, inp, tok_k, r["ids"][keep], r["w"][keep], slot)
    assert_maxabs(np32(o["y"][torch.as_tensor(tok_k)]), y_ref, TOL_Y[c.dtype], "y")
    if wl.bias_rate:
        # one loss-free bias update: experts above the mean load move down by the
        # rate, below it up, at it not at all (bit-exact parity is a stage test)
        bias = inp["sel_bias"].clone()
        moe.moe_bias_update(c, o["counts"], bias, wl.bias_rate)
        delta = (bias.cpu().double() - inp["sel_bias"].cpu().double()).numpy()
        over = counts * c.n_experts > c.T * c.top_k
        under = counts * c.n_experts < c.T * c.top_k
        assert np.all(delta[over] < 0) and np.all(delta[under] > 0)
        assert np.all(delta[~over & ~under] == 0)
        assert np.allclose(np.abs(delta[over | under]), wl.bias_rate, rtol=1e-3)


def test_layer_is_deterministic(cuda_device):
    wl = WORKLOADS["switch"]
    inp = make_inputs(wl, cuda_device)
    o1, ws = run_layer(wl, inp, cuda_device)
    o2, _ = run_layer(wl, inp, cuda_device, ws)
    for key in o1:
        assert torch.equal(o1[key], o2[key]), key


@pytest.mark.parametrize("act,k", [(moe.MOE_RELU, 1), (moe.MOE_SWIGLU, 2)])
def test_skewed_layer_mixes_heavy_and_light_experts(cuda_device, act, k):
    """Zipf-skewed routing gives experts from hundreds of rows down to a few
    in one grouped-GEMM launch (full, partial and single-row tiles side by
    side); top-1 without shared experts also takes the path where the down
    GEMM writes gate * output into y. Every token is checked against the
    oracle fed the GPU's routing."""
    dev = cuda_device
    wl = WORKLOADS["mixtral"].with_(T=2048, d_model=256, n_experts=32, top_k=k, d_ff=256,
                                    act=act, zipf_s=0.25)
    c = wl.cfg
    inp = make_inputs(wl, dev)
    o, ws = run_layer(wl, inp, dev)
    counts = np.bincount(o["ids"].cpu().numpy().ravel(), minlength=c.n_experts)
    assert counts.max() > 3 * 128 and ((counts > 0) & (counts <= 128)).any()  # both sizes
    ids, w = o["ids"].cpu().numpy(), np.asarray(np32(o["w"]), np.float64)
    cap = oracle.capacity(ids, c.n_experts, c.T)
    y_ref = _oracle_y(wl, inp, list(range(c.T)), ids, w, cap["slot"])
    assert_maxabs(np32(o["y"]), y_ref, TOL_Y[c.dtype], "y")


@pytest.mark.parametrize("T,E,k,cf,d,pad", [
    (4097, 64, 1, 1.0, 128, 0),   # top-1 (the down GEMM writes y), partial last block
    (1000, 256, 8, 1.0, 64, 0),   # top-8 over 256 experts, drops in every block
    (300, 16, 2, 0.5, 64, 0),     # half the assignments dropped
    (1001, 32, 2, 0.75, 64, 1),   # padded to capacity
])
def test_layer_token_order_capacity(cuda_device, T, E, k, cf, d, pad):
    """Token-order capacity inside the layer (the selection kernel counts the
    per-256-token histograms, the scan/slot kernel ranks each token), with
    drops, a partial last block and padding: counts bit-exact and y on every
    token against the oracle fed the GPU's routing."""
    from gpu_helpers import layer_vs_oracle
    wl = WORKLOADS["switch"].with_(T=T, d_model=d, n_experts=E, top_k=k, d_ff=128,
                                    capacity_factor=cf, pad_to_capacity=pad)
    o, _ = layer_vs_oracle(wl, cuda_device)
    assert (o["slot"] < 0).any()
