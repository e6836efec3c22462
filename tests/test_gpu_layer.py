"""The whole layer at the workloads' full sizes, in the launch configuration the
benchmark times (moe_layer_fwd on one stream). Router logits and
probabilities of every token are compared with the oracle's router; ids,
gates, counts and slots of every token are compared bit for bit with the
oracle's selection and capacity fed the GPU's own scores; y is compared with
the oracle fed the GPU's routing on every token of the small cases and, at
full size, on at least 256 tokens chosen to cover the grouped GEMM's tile
boundaries (a token's output depends only on its own routing and rows)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs

from gpu_helpers import (TOL_AUX, TOL_GATE, TOL_LOGITS, TOL_Y, assert_maxabs, assert_rowwise,
                         check_topk_valid, np32, oracle_noise, run_layer, score_tolerance)

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


def _identical_scores(c, sel, probs):
    """The oracle's top-k choice and gates taken on the GPU's own selection
    scores and probabilities (the "identical router logits" comparison)."""
    return oracle.select(np32(sel), np32(probs), c.top_k, bool(c.renorm_topk))


def _boundary_tokens(cap, row_cap=128):
    """Tokens whose rows sit where the grouped GEMM's tiles change: the first,
    middle and last row tile of the heaviest expert, rows 128n-1 and 128n of
    every expert that has them, every row of up to 16 experts small enough
    for the 64-row tiles, and the first and last row of every expert."""
    offsets, row_token = cap["offsets"], cap["row_token"]
    kept = np.diff(offsets)
    rows = set()
    heavy = int(np.argmax(kept))
    lo, n = int(offsets[heavy]), int(kept[heavy])
    mid = (n // 2) // row_cap * row_cap
    for r in list(range(0, min(n, 8))) + list(range(mid, min(n, mid + 8))) + \
            list(range(max(0, n - 8), n)) + [n // row_cap * row_cap - 1]:
        if 0 <= r < n:
            rows.add(lo + r)
    light = [e for e in range(len(kept)) if 0 < kept[e] <= 64][:16]
    for e in light:
        rows.update(range(int(offsets[e]), int(offsets[e + 1])))
    for e in range(len(kept)):
        a, m = int(offsets[e]), int(kept[e])
        if m == 0:
            continue
        rows.update((a, a + m - 1))
        for b in range(row_cap, m, row_cap):
            rows.update((a + b - 1, a + b))
    return sorted({int(row_token[r]) for r in rows}), heavy, light


def _dispatch_full(c, x, ids, dev):
    """moe_dispatch on the layer's ids: counts, kept, offsets, slot, xp, row_token."""
    T, E, k, d = c.T, c.n_experts, c.top_k, c.d_model
    C, R = moe.moe_capacity(c)
    o = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
             kept=torch.empty(E, dtype=torch.int32, device=dev),
             offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
             slot=torch.empty((T, k), dtype=torch.int32, device=dev),
             xp=torch.empty((R, d), dtype=c.torch_dtype, device=dev),
             row_token=torch.empty(R, dtype=torch.int32, device=dev))
    ws = moe.workspace(c, dev)
    moe.moe_dispatch(c, x, ids, o["counts"], o["kept"], o["offsets"], o["slot"], o["xp"],
                     o["row_token"], ws)
    assert moe.moe_read_device_error(c, ws) == 0
    return o, ws


def _check_stats(c, o, probs):
    """Layer statistics against the oracle's, computed from the GPU's own
    probabilities, ids and gates."""
    st = oracle.aux_stats(np32(probs), o["ids"].cpu().numpy(), np32(o["w"]), c.n_experts,
                          c.importance_weight)
    o3 = np32(o["out3"])
    assert o3[0] == pytest.approx(st["aux"], rel=TOL_AUX)
    assert o3[1] == pytest.approx(st["cv2"], rel=TOL_AUX)
    assert o3[2] == pytest.approx(st["L_imp"], rel=TOL_AUX)
    av = np32(o["aux_vecs"])
    np.testing.assert_allclose(av[0], st["f"], rtol=1e-6)
    np.testing.assert_allclose(av[1], st["P"], rtol=TOL_AUX)
    np.testing.assert_allclose(av[2], st["I"], rtol=TOL_AUX)
    return st


@pytest.mark.parametrize("name", ["switch", "switch_drawn"])
def test_switch_full(cuda_device, name):
    """Noisy top-1, capacity 128 with drops (router noise passed in from the
    host, or drawn by the library): every token routed by the oracle."""
    wl = WORKLOADS[name]
    c = wl.cfg
    inp = make_inputs(wl, cuda_device)
    o, _ = run_layer(wl, inp, cuda_device)
    logits, probs, sel, _, _ = _route(wl, inp, cuda_device)
    r = _oracle_router(wl, inp, list(range(c.T)))
    assert_rowwise(np32(logits), r["z"], TOL_LOGITS, "logits")
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    ids = o["ids"].cpu().numpy()
    # bit-exact on identical scores, valid against the oracle's own scores
    ids_ref, w_ref = _identical_scores(c, sel, probs)
    np.testing.assert_array_equal(ids, ids_ref)
    diff = check_topk_valid(ids, r["s"], c.top_k)
    assert len(diff) <= 2, diff
    assert np.all(np32(o["w"]) == 1.0)  # Softmax(KeepTopK(H, 1)) = 1
    C, _ = moe.moe_capacity(c)
    cap = oracle.capacity(ids_ref, c.n_experts, C)
    np.testing.assert_array_equal(o["counts"].cpu().numpy(), cap["counts"])
    dropped = int((cap["slot"] < 0).sum())
    assert 200 < dropped < 600, dropped
    tok = sorted(set(_sample(c.T, 256, 1)) | set(_boundary_tokens(cap)[0]))
    y_ref = _oracle_y(wl, inp, tok, ids[tok], w_ref[tok], cap["slot"][tok])
    assert_maxabs(np32(o["y"][torch.as_tensor(tok)]), y_ref, TOL_Y[c.dtype], "y")
    # dropped tokens of top-1 routing output exactly zero
    dropped_tok = np.nonzero(cap["slot"][:, 0] < 0)[0]
    assert float(o["y"][torch.as_tensor(dropped_tok)].abs().max()) == 0.0
    _check_stats(c, o, probs)
    # the oracle's own statistics (its own probabilities and routing)
    st = oracle.aux_stats(r["p"].astype(np.float32), r["ids"], r["w"].astype(np.float32),
                          c.n_experts, c.importance_weight)
    assert np32(o["out3"])[0] == pytest.approx(st["aux"], rel=1e-4)


@pytest.mark.parametrize("name", ["mixtral", "deepseek", "decode"])
def test_large_config_full(cuda_device, name):
    """The Mixtral-, DeepSeek- and decode-shaped layers at full size:
    logits and probabilities of every token against the oracle's router;
    ids, gates, counts, offsets, slots and rows of every token bit-exact
    against the oracle's selection and capacity on the GPU's own scores; y
    against the oracle on at least 256 tokens that include every tile
    boundary kind; statistics and the bias update against the oracle."""
    dev = cuda_device
    wl = WORKLOADS[name]
    c = wl.cfg
    T, E, k = c.T, c.n_experts, c.top_k
    inp = make_inputs(wl, dev)
    o, ws = run_layer(wl, inp, dev)
    logits, probs, sel, _, _ = _route(wl, inp, dev)
    r = _oracle_router(wl, inp, list(range(T)))
    assert_rowwise(np32(logits), r["z"], TOL_LOGITS, "logits")
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    ids = o["ids"].cpu().numpy()
    ids_ref, w_ref = _identical_scores(c, sel, probs)
    np.testing.assert_array_equal(ids, ids_ref)
    assert_rowwise(np32(o["w"]), w_ref, TOL_GATE, "gates")
    # the oracle's own routing differs only where its scores tie within what
    # the router tolerance allows
    tol = score_tolerance(r["s"], r["p"], biased=wl.sel_bias)
    diff = check_topk_valid(ids, r["s"], k, tol=tol)
    srt = -np.sort(-r["s"], axis=1)[:, :k + 1]
    gaps = (srt[:, :-1] - srt[:, 1:]).min(axis=1)
    assert set(diff) <= set(np.nonzero(gaps < tol)[0].tolist())
    C, R = moe.moe_capacity(c)
    cap = oracle.capacity(ids_ref, E, C)
    np.testing.assert_array_equal(o["counts"].cpu().numpy(), cap["counts"])
    dp, _ = _dispatch_full(c, inp["x"], o["ids"], dev)
    for key in ("counts", "kept", "offsets", "slot"):
        np.testing.assert_array_equal(dp[key].cpu().numpy(), cap[key], err_msg=key)
    n = int(cap["offsets"][-1])
    np.testing.assert_array_equal(dp["row_token"][:n].cpu().numpy(), cap["row_token"])
    # xp[row] is x[row_token[row]], byte for byte
    assert torch.equal(dp["xp"][:n], inp["x"][dp["row_token"][:n].long()])
    # y on boundary tokens plus a seeded sample, at least 256 tokens
    btok, heavy, light = _boundary_tokens(cap)
    tok = sorted(set(btok) | set(_sample(T, 256, 2)))
    if len(tok) < min(256, T):
        tok = sorted(set(tok) | set(range(min(256, T))))
    assert len(tok) >= min(256, T)
    if E > 64:
        assert len(light) >= 8  # the 64-row MMA path is covered
    y_ref = _oracle_y(wl, inp, tok, ids[tok], np.asarray(np32(o["w"]), np.float64)[tok],
                      cap["slot"][tok])
    assert_maxabs(np32(o["y"][torch.as_tensor(tok)]), y_ref, TOL_Y[c.dtype], "y")
    _check_stats(c, o, probs)
    if wl.bias_rate:
        bias = inp["sel_bias"].clone()
        moe.moe_bias_update(c, o["counts"], bias, wl.bias_rate)
        want = oracle.bias_update(o["counts"].cpu(), inp["sel_bias"].cpu(), T, k, wl.bias_rate)
        np.testing.assert_array_equal(bias.cpu().numpy(), want)


def test_deepseek_whole_experts(cuda_device):
    """moe_expert_ffn at the DeepSeek shape: every row of the heaviest routed
    expert (dozens of 128-row tiles and a partial last one), every row of the
    four lightest non-empty experts (64-row tiles) and every row of the
    shared expert's first tile, against the oracle's expert FFN."""
    dev = cuda_device
    wl = WORKLOADS["deepseek"]
    c = wl.cfg
    inp = make_inputs(wl, dev)
    _, _, _, ids, _ = _route(wl, inp, dev)
    dp, ws = _dispatch_full(c, inp["x"], ids, dev)
    C, R = moe.moe_capacity(c)
    yp = torch.empty((R, c.d_model), dtype=c.torch_dtype, device=dev)
    ys = torch.empty((c.n_shared, c.T, c.d_model), dtype=c.torch_dtype, device=dev)
    moe.moe_expert_ffn(c, dp["xp"], dp["offsets"], inp["W1"], inp["W2"], inp["x"], inp["W1s"],
                       inp["W2s"], yp, ys, ws)
    assert moe.moe_read_device_error(c, ws) == 0
    offsets = dp["offsets"].cpu().numpy()
    kept = np.diff(offsets)
    heavy = int(np.argmax(kept))
    lightest = [int(e) for e in np.argsort(kept, kind="stable") if kept[e] > 0][:4]
    assert kept[heavy] > 20 * 128 and all(kept[e] <= 64 for e in lightest)
    for e in [heavy] + lightest:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        ref = oracle.expert_ffn(dp["xp"][lo:hi].cpu(), inp["W1"][e].cpu(), inp["W2"][e].cpu(),
                                c.act, oracle.ROUND_BF16)
        assert_maxabs(np32(yp[lo:hi]), ref, TOL_Y[c.dtype], f"expert {e} ({hi - lo} rows)")
    ref = oracle.expert_ffn(inp["x"][:128].cpu(), inp["W1s"][0].cpu(), inp["W2s"][0].cpu(),
                            c.act, oracle.ROUND_BF16)
    assert_maxabs(np32(ys[0, :128]), ref, TOL_Y[c.dtype], "shared expert")


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


@pytest.mark.parametrize("name,kw", [
    ("mixtral", dict(T=3000, d_model=512, d_ff=512)),
    ("deepseek", dict(T=2000, d_model=512, d_ff=256, n_experts=64, capacity_factor=1.0)),
    ("decode", dict(d_model=512, d_ff=256)),
    ("switch_reroute", dict(T=4096, d_model=256, d_ff=256, top_k=2, n_shared=1)),
])
def test_folded_combine_equals_the_combine_kernel(cuda_device, name, kw):
    """The combine folded into the down GEMM and the separate combine kernel
    add the same bf16 rows with the same gates in the same order, so y is
    equal bit for bit (shared experts, drops and re-routed candidates
    included); both match the oracle fed the GPU's routing."""
    from gpu_helpers import layer_vs_oracle
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, cuda_device)
    ys = []
    for mode in (moe.MOE_COMBINE_IN_GEMM, moe.MOE_COMBINE_KERNEL):
        o, _ = layer_vs_oracle(wl.with_(combine_mode=mode), cuda_device, inp)
        ys.append(o["y"])
    assert torch.equal(ys[0], ys[1])


@pytest.mark.parametrize("k,T,act", [(1, 8192, moe.MOE_RELU), (2, 4096, moe.MOE_SWIGLU),
                                     (2, 4096, moe.MOE_GELU)])
def test_pair_tiles_with_ragged_experts(cuda_device, k, T, act):
    """Experts that hold 1024 rows or more on average (R_max >= 1024 E) run
    the expert GEMMs on CTA pairs: 256-row tiles, each CTA holding 128 rows
    and half of the weight tile, one pair MMA (M = 256) per K step. A strong
    Zipf skew puts experts of thousands of rows (full tiles and a last tile
    of 129..255 rows), of at most 128 rows (the odd CTA's rows all belong to
    the next expert and are not stored) and of a handful of rows into the
    same launches; y of every token matches the oracle fed the GPU's routing
    (top-1: the down GEMM scatters gate * output into y; top-2: the combine
    kernel)."""
    from gpu_helpers import layer_vs_oracle
    wl = WORKLOADS["mixtral"].with_(T=T, d_model=256, d_ff=256, zipf_s=1.5, top_k=k, act=act)
    c = wl.cfg
    assert c.T * k >= 1024 * c.n_experts
    o, _ = layer_vs_oracle(wl, cuda_device)
    counts = np.bincount(o["ids"].cpu().numpy().ravel(), minlength=c.n_experts)
    assert counts.max() > 8 * 256 and ((counts > 0) & (counts <= 128)).any()


@pytest.mark.parametrize("mode", [moe.MOE_COMBINE_KERNEL, moe.MOE_COMBINE_IN_GEMM])
def test_split_launch_for_mixed_expert_sizes(cuda_device, mode):
    """Layers whose experts hold 256..1023 rows on average but of very mixed
    sizes (DeepSeek-shaped: the selection bias sends most tokens to a few
    experts) run each expert projection as two launches: experts of fewer
    than 512 rows on single CTAs, the others and the shared expert on CTA
    pairs. Here 9 experts hold 630..2048 rows and 9 hold 1..297; y of every
    token matches the oracle fed the GPU's routing, with the combine kernel
    and with the combine folded into the (two) down launches."""
    from gpu_helpers import layer_vs_oracle
    wl = WORKLOADS["deepseek"].with_(T=2048, d_model=256, d_ff=256, n_experts=32,
                                     combine_mode=mode)
    c = wl.cfg
    assert 256 * c.n_experts <= c.T * c.top_k < 1024 * c.n_experts
    o, _ = layer_vs_oracle(wl, cuda_device)
    counts = o["counts"].cpu().numpy()
    assert (counts >= 512).sum() >= 4 and ((counts > 0) & (counts < 512)).sum() >= 4


@pytest.mark.parametrize("kind", ["all_few_row", "all_many_row"])
def test_split_launch_with_one_kind_of_expert(cuda_device, kind):
    """The same layer shape class (256..1023 rows per expert on average) when
    every expert falls on one side of 512 rows, so that one of the two
    launches of each projection has no tile: uniform routing over 16 experts
    (about 256 rows each, no shared expert: the many-row launch is empty),
    and 8 experts of about 700 rows with a shared expert (the few-row launch
    is empty). y of every token matches the oracle."""
    from gpu_helpers import layer_vs_oracle
    base = WORKLOADS["deepseek"].with_(d_model=256, d_ff=256, sel_bias=False, bias_rate=0.0)
    if kind == "all_few_row":
        wl = base.with_(T=2048, n_experts=16, top_k=2, n_shared=0)
    else:
        wl = base.with_(T=2800, n_experts=8, top_k=2)
    c = wl.cfg
    assert 256 * c.n_experts <= c.T * c.top_k < 1024 * c.n_experts
    o, _ = layer_vs_oracle(wl, cuda_device)
    counts = o["counts"].cpu().numpy()
    if kind == "all_few_row":
        assert counts.max() < 512
    else:
        assert counts.min() >= 512
