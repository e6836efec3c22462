"""Edge cases of the layer on the GPU, each against the oracle: the largest
supported expert count and top-k, top-k equal to E (the sparse layer is then
the dense mixture), a capacity of one row, a single token, every token on
one expert, and batch sizes on both sides of the one-launch capacity scan's
limit (256 token blocks)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth
from sparse_mixture_experts_69_b300.workloads import WORKLOADS, Workload, make_inputs

from gpu_helpers import TOL_Y, assert_maxabs, layer_vs_oracle, np32

pytestmark = pytest.mark.gpu


def _wl(name="edge", **cfg):
    base = dict(T=96, d_model=64, n_experts=8, top_k=2, d_ff=64, capacity_factor=0.0,
                dtype=moe.MOE_BF16, act=moe.MOE_SWIGLU)
    base.update(cfg)
    return Workload(name, moe.Config(**base))


def test_largest_expert_count_and_top_k(cuda_device):
    layer_vs_oracle(_wl(n_experts=1024, top_k=32, T=96), cuda_device)


@pytest.mark.parametrize("dtype", [moe.MOE_F32, moe.MOE_BF16])
def test_top_k_equal_to_E_is_the_dense_mixture(cuda_device, dtype):
    """With k = E and no capacity limit every token visits every expert with
    gate p_e (renormalised over all E, i.e. p_e itself): y = sum_e p_e E_e(x)."""
    wl = _wl(n_experts=8, top_k=8, T=64, dtype=dtype, act=moe.MOE_GELU)
    o, inp = layer_vs_oracle(wl, cuda_device)
    rd = oracle.ROUND_BF16 if dtype == moe.MOE_BF16 else oracle.ROUND_F32
    x = inp["x"].cpu()
    w = np.asarray(np32(o["w"]), np.float64)
    ids = o["ids"].cpu().numpy()
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-5)
    dense = np.zeros((64, 64))
    for e in range(8):
        Oe = oracle.expert_ffn(x, inp["W1"][e].cpu(), inp["W2"][e].cpu(), wl.cfg.act, rd)
        g = np.array([w[t, list(ids[t]).index(e)] for t in range(64)])
        dense += g[:, None] * Oe
    assert_maxabs(np32(o["y"]), dense, TOL_Y[dtype], "dense mixture")


def test_capacity_of_one_row(cuda_device):
    """C = 1: one token per expert survives; every other token's output is zero."""
    wl = _wl(T=64, top_k=1, capacity_factor=0.01, act=moe.MOE_RELU)
    assert moe.moe_capacity(wl.cfg)[0] == 1
    o, _ = layer_vs_oracle(wl, cuda_device)
    kept = (o["slot"] >= 0).any(axis=1)
    assert kept.sum() <= wl.cfg.n_experts
    assert (np32(o["y"])[~kept] == 0).all()


def test_single_token_with_shared_experts(cuda_device):
    layer_vs_oracle(_wl(T=1, n_shared=2, top_k=3), cuda_device)


def test_every_token_on_one_expert(cuda_device):
    """A logit offset no softmax gap can overcome sends all tokens to expert 0."""
    wl = _wl(T=300, top_k=1, act=moe.MOE_RELU)
    inp = make_inputs(wl, cuda_device)
    inp["logit_offset"] = torch.tensor([60.0] + [0.0] * 7, device=cuda_device)
    o, _ = layer_vs_oracle(wl, cuda_device, inp)
    assert (o["ids"].cpu().numpy() == 0).all()


@pytest.mark.parametrize("T", [65536, 65537])
def test_dispatch_at_the_capacity_scan_block_limit(cuda_device, T):
    """256 token blocks take the one-launch scan + slots; 257 take the
    separate scan and slot kernels. Both bit-exact."""
    E, k, cf, d = 64, 2, 1.0, 16
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=8, capacity_factor=cf)
    C, R_max = moe.moe_capacity(cfg)
    dev = cuda_device
    s = synth.uniform((T, E), 9, 200, 0.0, 1.0) + 0.3 * torch.linspace(1.0, 0.0, E)
    ids = torch.argsort(-s, dim=1, stable=True)[:, :k].to(torch.int32).contiguous()
    x = synth.normal((T, d), 9, 121, 1.0, torch.bfloat16, dev)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               kept=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               slot=torch.empty((T, k), dtype=torch.int32, device=dev))
    xp = torch.zeros((R_max, d), dtype=torch.bfloat16, device=dev)
    row_token = torch.full((R_max,), -7, dtype=torch.int32, device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_dispatch(cfg, x, ids.to(dev), out["counts"], out["kept"], out["offsets"], out["slot"],
                     xp, row_token, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    ref = oracle.capacity(ids.numpy(), E, C)
    for n in ("counts", "kept", "offsets", "slot"):
        np.testing.assert_array_equal(out[n].cpu().numpy(), ref[n], err_msg=n)
    R = int(ref["offsets"][-1])
    np.testing.assert_array_equal(row_token[:R].cpu().numpy(), ref["row_token"])
    assert torch.equal(xp[:R].cpu(), x.cpu()[torch.as_tensor(ref["row_token"]).long()])
