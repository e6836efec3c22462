"""moe_aux_stats_noalloc: the statistics entry point for callers that cannot
give the library a workspace (a plugin in a host framework that owns all
device memory, or code where allocating is not allowed). It uses a device
array inside libmoe.so instead. Its results must match moe_aux_stats, which
takes a caller-allocated workspace, on back-to-back calls; the array is
shared by all calls and keeps the previous call's contents, so the second
call also shows that each call starts from a cleared array.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth

from gpu_helpers import TOL_AUX, np32


def _inputs(T, E, k, seed, dev):
    logits = synth.normal((T, E), seed, 500)
    probs = torch.softmax(logits.double(), dim=1).float()
    s = synth.uniform((T, E), seed, 501, 0.0, 1.0) + torch.linspace(0.5, 0.0, E)
    ids = torch.argsort(-s, dim=1, stable=True)[:, :k].to(torch.int32).contiguous()
    w = synth.uniform((T, k), seed, 502, 0.0, 1.0)
    return probs.to(dev), ids.to(dev), w.to(dev)


def _outs(E, dev):
    return [torch.full((E,), -1.0, device=dev) for _ in range(3)] + [
        torch.full((3,), -1.0, device=dev)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_on_consecutive_calls(cuda_device):
    dev = cuda_device
    for call, (T, E, k) in enumerate([(8192, 256, 8), (3000, 64, 2)]):
        cfg = moe.Config(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, dtype=moe.MOE_BF16,
                         importance_weight=0.01)
        probs, ids, w = _inputs(T, E, k, 40 + call, dev)
        f0, P0, I0, o0 = _outs(E, dev)
        moe.moe_aux_stats(cfg, probs, ids, w, f0, P0, I0, o0, moe.workspace(cfg, dev))
        f1, P1, I1, o1 = _outs(E, dev)
        moe.moe_aux_stats_noalloc(cfg, probs, ids, w, f1, P1, I1, o1)
        torch.cuda.synchronize()
        ref = oracle.aux_stats(probs.cpu(), ids.cpu(), w.cpu(), E, cfg.importance_weight)
        ref3 = [ref["aux"], ref["cv2"], ref["L_imp"]]
        for a, b, r, name in [(f1, f0, ref["f"], "f"), (P1, P0, ref["P"], "P"),
                              (I1, I0, ref["I"], "importance"), (o1, o0, ref3, "aux/cv2/L")]:
            np.testing.assert_allclose(np32(a), r, rtol=TOL_AUX, atol=0,
                                       err_msg=f"call {call} {name} vs the oracle")
            np.testing.assert_allclose(np32(a), np32(b), rtol=TOL_AUX, err_msg=f"call {call} {name}")
        assert np32(o1)[0] > 0.0  # outputs were written


def test_noalloc_rejects_more_experts_than_its_scratch_holds():
    cfg = moe.Config(T=64, d_model=8, n_experts=513, top_k=2, d_ff=8, dtype=moe.MOE_BF16)
    A = 1 << 20  # never dereferenced: the size check comes first
    st = moe.lib().moe_aux_stats_noalloc(ctypes.byref(cfg.c()), A, A, A, None, None, None, A,
                                         None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
    # the workspace version accepts that size
    assert moe.moe_workspace_size(cfg) > 0
