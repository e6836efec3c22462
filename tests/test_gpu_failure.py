"""Failure detection on the device without faulting the GPU: the library's
bounded waits are made to run out on purpose (moe_set_wait_limits), the
kernel reports MOE_ERR_TIMEOUT through the workspace status word and
returns, and the same CUDA context then runs the path again, within the
default limits, with results that match the oracle.

- The tensor-core GEMM kernels bound every pipeline wait in time. With the
  hold switch on, each CTA's first "accumulator ready" signal is withheld
  (a signal nothing else gives), so the epilogue's wait for it runs out
  after the limit (1 ms here) in every CTA; aborting CTAs let their own
  copies and matrix operations finish before they free tensor memory and
  exit.
- The capacity kernel with re-routing bounds its fixed-point loop in
  passes. One pass cannot settle when an expert overflows (the first pass
  starts from "no expert is full"); its slots then stay in range."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs

from gpu_helpers import TOL_Y, assert_maxabs, layer_vs_oracle, np32

pytestmark = pytest.mark.gpu
MOE_ERR_TIMEOUT = 6


def _routed(wl, inp, dev, ws):
    c = wl.cfg
    T, E, nc, d = c.T, c.n_experts, c.n_cand, c.d_model
    C, R = moe.moe_capacity(c)
    o = dict(logits=torch.empty((T, E), device=dev), probs=torch.empty((T, E), device=dev),
             ids=torch.empty((T, nc), dtype=torch.int32, device=dev),
             w=torch.empty((T, nc), device=dev),
             counts=torch.empty(E, dtype=torch.int32, device=dev),
             kept=torch.empty(E, dtype=torch.int32, device=dev),
             offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
             slot=torch.empty((T, nc), dtype=torch.int32, device=dev),
             xp=torch.zeros((R, d), dtype=c.torch_dtype, device=dev),
             row_token=torch.empty(R, dtype=torch.int32, device=dev))
    moe.moe_route(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"],
                  inp["sel_bias"], o["logits"], o["probs"], None, o["ids"], o["w"], 0, ws)
    return o


def _dispatch(c, inp, o, ws):
    moe.moe_dispatch(c, inp["x"], o["ids"], o["counts"], o["kept"], o["offsets"], o["slot"],
                     o["xp"], o["row_token"], ws)


def test_gemm_wait_limit_runs_out_and_the_context_stays_usable(cuda_device):
    dev = cuda_device
    wl = WORKLOADS["deepseek"].with_(name="small", T=700, d_model=256, n_experts=16, top_k=4,
                                     d_ff=256, n_shared=1)
    c = wl.cfg
    inp = make_inputs(wl, dev)
    ws = moe.workspace(c, dev)
    o = _routed(wl, inp, dev, ws)
    _dispatch(c, inp, o, ws)
    assert moe.moe_read_device_error(c, ws) == 0
    C, R = moe.moe_capacity(c)
    yp = torch.zeros((R, c.d_model), dtype=c.torch_dtype, device=dev)
    ys = torch.zeros((c.n_shared, c.T, c.d_model), dtype=c.torch_dtype, device=dev)

    def ffn():
        moe.moe_expert_ffn(c, o["xp"], o["offsets"], inp["W1"], inp["W2"], inp["x"], inp["W1s"],
                           inp["W2s"], yp, ys, ws)

    moe.moe_set_wait_limits(1_000_000, 0, 1)
    try:
        ffn()
        st = moe.moe_read_device_error(c, ws)
    finally:
        moe.moe_set_wait_limits(0, 0, 0)
    assert st == MOE_ERR_TIMEOUT, moe.moe_status_string(st)
    # the status word was cleared by the read; the same context runs the FFN again
    ffn()
    assert moe.moe_read_device_error(c, ws) == 0
    offsets = o["offsets"].cpu().numpy()
    xp = o["xp"].float().cpu().numpy()
    for e in range(c.n_experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        ref = oracle.expert_ffn(xp[lo:hi], inp["W1"][e].cpu(), inp["W2"][e].cpu(), c.act,
                                oracle.ROUND_BF16)
        assert_maxabs(np32(yp[lo:hi]), ref, TOL_Y[c.dtype], f"expert {e}")
    ref = oracle.expert_ffn(inp["x"].cpu(), inp["W1s"][0].cpu(), inp["W2s"][0].cpu(), c.act,
                            oracle.ROUND_BF16)
    assert_maxabs(np32(ys[0]), ref, TOL_Y[c.dtype], "shared expert")
    # and the whole layer, router GEMM included
    layer_vs_oracle(wl, dev, inp)


def test_policy_pass_limit_runs_out_and_the_context_stays_usable(cuda_device):
    dev = cuda_device
    wl = WORKLOADS["switch_reroute"].with_(T=4096, d_model=64, d_ff=64, n_experts=32)
    c = wl.cfg
    inp = make_inputs(wl, dev)
    ws = moe.workspace(c, dev)
    o = _routed(wl, inp, dev, ws)
    assert moe.moe_read_device_error(c, ws) == 0
    C, R = moe.moe_capacity(c)
    moe.moe_set_wait_limits(0, 1, 0)
    try:
        _dispatch(c, inp, o, ws)
        st = moe.moe_read_device_error(c, ws)
    finally:
        moe.moe_set_wait_limits(0, 0, 0)
    assert st == MOE_ERR_TIMEOUT, moe.moe_status_string(st)
    slot = o["slot"].cpu().numpy()
    assert slot.min() >= -1 and slot.max() < R  # the unsettled slots stay in range
    _dispatch(c, inp, o, ws)
    assert moe.moe_read_device_error(c, ws) == 0
    ref = oracle.capacity_policy(o["ids"].cpu().numpy(), c.top_k, c.n_experts, C,
                                 priority=c.priority)
    assert (ref["counts"] > C).any()  # an expert overflows: one pass could not settle
    for key in ("counts", "kept", "offsets", "slot"):
        np.testing.assert_array_equal(o[key].cpu().numpy(), ref[key], err_msg=key)
    n = int(ref["offsets"][-1])
    np.testing.assert_array_equal(o["row_token"][:n].cpu().numpy(), ref["row_token"])
    layer_vs_oracle(wl, dev, inp)
