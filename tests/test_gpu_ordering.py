"""Launch ordering of the layer on one stream. Its kernels overlap through
programmatic dependent launch, and two kinds of launch read inputs before
waiting for the kernel ahead of them (the router-weight copy and the expert
GEMMs' first weight tiles and tile table). These tests change those inputs
with the kernel right before the call, and run the layer inside a CUDA graph,
and check every output against the plain eager result. A last test runs two
layers concurrently on two streams with their own workspaces."""
import pytest
import torch

from sparse_mixture_experts_69_b300 import moe
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs

from gpu_helpers import run_layer

pytestmark = pytest.mark.gpu


def _small(name):
    return WORKLOADS[name].with_(T=1024, d_model=256, d_ff=512)


@pytest.mark.parametrize("name", ["switch", "deepseek", "decode", "mixtral"])
def test_inputs_written_just_before_the_call(cuda_device, name):
    """Wg, W1, W2 and x are overwritten by device kernels on the same stream
    immediately before moe_layer_fwd: the result must be the one for the new
    values, equal bit for bit to a run on freshly allocated copies."""
    wl = _small(name) if name != "decode" else WORKLOADS["decode"].with_(d_model=256, d_ff=512)
    dev = cuda_device
    inp = make_inputs(wl, dev)
    fresh = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    for k in ("Wg", "W1", "W2", "x"):
        fresh[k] = (fresh[k].float() * -0.5).to(fresh[k].dtype)
    ref, _ = run_layer(wl, fresh, dev)
    # first a run on the old values (so a stale copy of the old weights exists
    # in the workspace), then the in-place update on the stream, then the call
    old, ws = run_layer(wl, inp, dev)
    for k in ("Wg", "W1", "W2", "x"):
        inp[k].mul_(-0.5)
    new, _ = run_layer(wl, inp, dev, ws)
    for key in ref:
        assert torch.equal(new[key], ref[key]), key
    assert not torch.equal(new["y"], old["y"])


@pytest.mark.parametrize("name", ["switch", "deepseek"])
def test_layer_in_a_cuda_graph(cuda_device, name):
    """Three back-to-back layer calls captured in one CUDA graph and replayed
    give the eager outputs bit for bit."""
    wl = _small(name)
    c = wl.cfg
    dev = cuda_device
    inp = make_inputs(wl, dev)
    ref, ws = run_layer(wl, inp, dev)
    T, E, k, d = c.T, c.n_experts, c.top_k, c.d_model
    y = torch.empty((T, d), dtype=c.torch_dtype, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    aux_vecs = torch.empty((3, E), device=dev)
    out3 = torch.empty(3, device=dev)

    def call():
        moe.moe_layer_fwd(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"],
                          inp["logit_offset"], inp["sel_bias"], inp["W1"], inp["W2"], inp["W1s"],
                          inp["W2s"], y, ids, w, counts, aux_vecs, out3, ws)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            for _ in range(3):
                call()
    torch.cuda.synchronize()
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_read_device_error(c, ws) == 0
    for key, got in (("y", y), ("ids", ids), ("w", w), ("counts", counts),
                     ("aux_vecs", aux_vecs), ("out3", out3)):
        assert torch.equal(got, ref[key]), key


@pytest.mark.parametrize("name", ["switch", "deepseek", "mixtral"])
def test_back_to_back_calls_with_different_router_weights(cuda_device, name):
    """Two layer calls, then two moe_route calls, queued back to back on one
    stream with one workspace and different router weights: the second
    call's router-weight copy overwrites the workspace copy the first call's
    router GEMM reads, so it must not start before that GEMM is done. Each
    result equals a run of its own."""
    wl = _small(name)
    c = wl.cfg
    dev = cuda_device
    inp_a = make_inputs(wl, dev)
    inp_b = dict(inp_a)
    inp_b["Wg"] = (inp_a["Wg"].float().flip(1) * 1.5).to(inp_a["Wg"].dtype).contiguous()
    ref_a, _ = run_layer(wl, inp_a, dev)
    ref_b, _ = run_layer(wl, inp_b, dev)
    ws = moe.workspace(c, dev)
    outs = []
    for inp in (inp_a, inp_b):
        o = {k: torch.empty_like(v) for k, v in ref_a.items()}
        moe.moe_layer_fwd(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"],
                          inp["logit_offset"], inp["sel_bias"], inp["W1"], inp["W2"], inp["W1s"],
                          inp["W2s"], o["y"], o["ids"], o["w"], o["counts"], o["aux_vecs"],
                          o["out3"], ws)
        outs.append(o)
    torch.cuda.synchronize()
    assert moe.moe_read_device_error(c, ws) == 0
    for got, ref in zip(outs, (ref_a, ref_b)):
        for key in ref:
            assert torch.equal(got[key], ref[key]), key
    assert not torch.equal(outs[0]["ids"], outs[1]["ids"])

    T, E, k = c.T, c.n_experts, c.top_k
    routes = []
    for inp in (inp_a, inp_b):
        r = dict(logits=torch.empty((T, E), device=dev), probs=torch.empty((T, E), device=dev),
                 ids=torch.empty((T, k), dtype=torch.int32, device=dev),
                 w=torch.empty((T, k), device=dev))
        moe.moe_route(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                      inp["sel_bias"], r["logits"], r["probs"], None, r["ids"], r["w"], 0, ws)
        routes.append(r)
    torch.cuda.synchronize()
    for r, ref in zip(routes, (ref_a, ref_b)):
        assert torch.equal(r["ids"], ref["ids"])
        assert torch.equal(r["w"], ref["w"])


def test_concurrent_layers_on_two_streams(cuda_device):
    """Two layers with their own workspaces, enqueued alternately on two
    streams (four calls each, so their kernels overlap on the GPU), give the
    same bits as the same calls made one at a time: the library keeps no state
    outside a call's workspace (the CTA-pair GEMMs' tile counters included).
    One layer runs its expert GEMMs on CTA pairs, the other as the two-launch
    FFN of mixed expert sizes."""
    from gpu_helpers import layer_outputs
    dev = cuda_device
    wls = [WORKLOADS["mixtral"].with_(T=2048, d_model=256, n_experts=2, top_k=1, d_ff=256,
                                      name="pairs"),
           WORKLOADS["deepseek"].with_(T=2048, d_model=256, n_experts=32, d_ff=256,
                                       name="split")]
    inps = [make_inputs(wl, dev) for wl in wls]
    refs = [run_layer(wl, inp, dev)[0] for wl, inp in zip(wls, inps)]
    streams = [torch.cuda.Stream(dev) for _ in wls]
    wss = [moe.workspace(wl.cfg, dev) for wl in wls]
    outs = [layer_outputs(wl, inp, dev) for wl, inp in zip(wls, inps)]
    torch.cuda.synchronize()
    for _ in range(4):
        for wl, inp, o, ws, st in zip(wls, inps, outs, wss, streams):
            moe.moe_layer_fwd(wl.cfg, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"],
                              inp["logit_offset"], inp["sel_bias"], inp["W1"], inp["W2"],
                              inp["W1s"], inp["W2s"], o["y"], o["ids"], o["w"], o["counts"],
                              o["aux_vecs"], o["out3"], ws, st)
    torch.cuda.synchronize()
    for wl, o, ref, ws in zip(wls, outs, refs, wss):
        assert moe.moe_read_device_error(wl.cfg, ws) == 0
        for key in ("y", "ids", "w", "counts", "aux_vecs", "out3"):
            assert torch.equal(o[key], ref[key]), (wl.name, key)
