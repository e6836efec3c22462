"""GPU parity of the tensor-core (tcgen05) kernels: the bf16 router GEMM and
the grouped expert GEMMs, on shapes that span several tiles, ragged expert
row counts (0, 1, 127, 128, 129, ...), ragged N and K tails and shared experts."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_69_b300 import moe, synth

from gpu_helpers import TOL_GATE, TOL_LOGITS, assert_rowwise, check_topk_valid, np32
from test_gpu_stages import run_ffn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,d,E,k,noisy,offset,bias", [
    (300, 256, 8, 2, False, True, False),
    (1000, 200, 40, 3, False, False, False),
    (8192, 1024, 64, 1, True, False, False),
    (129, 7168, 256, 8, False, False, True),
    (64, 4096, 64, 6, False, False, False),
    (77, 512, 300, 4, False, False, False),
    # 256-wide routers run on CTA pairs (256-row tiles): a ragged last pair
    # tile with the K range split, an unsplit one with a column tail and the
    # logit offset, and a noisy router whose 2E = 256 columns hold z and zn
    (1000, 7168, 256, 8, False, False, True),
    (300, 256, 200, 4, False, True, False),
    (500, 512, 128, 2, True, False, False),
    # a memory-bound router of 79 full-height tiles runs one 68-row tile per
    # SM instead (148 tiles, the last of 4 rows)
    (10000, 512, 16, 2, False, True, False),
])
def test_router_bf16(cuda_device, T, d, E, k, noisy, offset, bias):
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=64, dtype=moe.MOE_BF16)
    dev = cuda_device
    bf = torch.bfloat16
    x = synth.normal((T, d), 11, 101, 1.0, bf)
    Wg = synth.normal((d, E), 11, 102, 0.02, bf)
    Wn = synth.normal((d, E), 11, 103, 0.02, bf) if noisy else None
    noise = synth.normal((T, E), 11, 104) if noisy else None
    off = synth.zipf_logit_offset(E, 1.2) if offset else None
    b = synth.uniform((E,), 11, 105, -0.1, 0.1) if bias else None
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
    assert len(diff) <= max(1, T // 1000), diff
    same = [t for t in range(T) if t not in diff]
    assert_rowwise(np32(w)[same], r["w"][same], TOL_LOGITS, "gates")


@pytest.mark.parametrize("T,d,E,k,reroute,bias,renorm,offset", [
    (300, 64, 8, 2, 0, False, 1, False),
    (257, 128, 32, 8, 0, True, 1, False),
    (129, 64, 17, 3, 2, False, 0, False),
    (5, 64, 1, 1, 0, False, 1, False),
    (1000, 192, 2, 2, 0, True, 1, True),
    (2000, 256, 8, 2, 6, False, 1, True),
    # one short tile per SM (148 tiles of 68 rows, the last of 4)
    (10000, 512, 16, 2, 0, False, 1, False),
])
def test_selection_in_router_gemm(cuda_device, T, d, E, k, reroute, bias, renorm, offset):
    """Routers of at most 32 columns with one K part select in the GEMM's
    epilogue, one token per thread. Small integer x and Wg make every logit
    an exact integer (many ties, which the lower index must win): logits equal
    the oracle's exactly, and on the GPU's own scores and probabilities the
    ids of all n_cand candidates are bit-exact against the oracle's
    selection, the gates within the division's rounding."""
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, reroute=reroute, renorm_topk=renorm,
                     d_ff=64, dtype=moe.MOE_BF16)
    nc = k + reroute
    dev = cuda_device
    bf = torch.bfloat16
    x = (synth.randint((T, d), 12, 101, 5) - 2).to(bf)
    Wg = (synth.randint((d, E), 12, 102, 3) - 1).to(bf)
    off = synth.zipf_logit_offset(E, 1.2) if offset else None
    b = synth.uniform((E,), 12, 105, -0.1, 0.1) if bias else None
    g = lambda t: None if t is None else t.to(dev)
    logits = torch.empty((T, E), device=dev)
    probs = torch.empty((T, E), device=dev)
    sel = torch.empty((T, E), device=dev)
    ids = torch.empty((T, nc), dtype=torch.int32, device=dev)
    w = torch.empty((T, nc), device=dev)
    ws = moe.workspace(cfg, dev)
    moe.moe_route(cfg, g(x), g(Wg), None, None, g(off), g(b), logits, probs, sel, ids, w, 0, ws)
    assert moe.moe_read_device_error(cfg, ws) == 0
    r = oracle.router(x, Wg, k, offset=off, bias=b, renorm=bool(renorm))
    if offset:
        assert_rowwise(np32(logits), r["z"], TOL_LOGITS, "logits")
    else:
        np.testing.assert_array_equal(np32(logits), r["z"].astype(np.float32))
    assert_rowwise(np32(probs), r["p"], TOL_LOGITS, "probs")
    assert_rowwise(np32(sel), r["s"], TOL_LOGITS, "sel_scores")
    ref_ids, ref_w = oracle.select_candidates(np32(sel), np32(probs), k, nc, renorm=bool(renorm))
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    # a gate is an fp32 quotient: relative rounding, except in the subnormal
    # range (far-down candidates), where it is at most one step of 2**-149
    np.testing.assert_allclose(np32(w), ref_w, rtol=TOL_GATE, atol=2.0**-149)


@pytest.mark.parametrize("act", [moe.MOE_RELU, moe.MOE_GELU, moe.MOE_SWIGLU])
def test_expert_ffn_bf16_ragged(cuda_device, act):
    """Per-expert rows 0, 1, 127, 128, 129, 300; d=200 (K tail), F=136 (N tail)."""
    cfg = moe.Config(T=200, d_model=200, n_experts=6, top_k=4, d_ff=136, n_shared=2,
                     dtype=moe.MOE_BF16, act=act)
    run_ffn(cfg, [0, 1, 127, 128, 129, 300], 21, cuda_device)


@pytest.mark.parametrize("act", [moe.MOE_RELU, moe.MOE_SWIGLU])
def test_expert_ffn_bf16_many_tiles(cuda_device, act):
    """More tiles than SMs, so the persistent CTAs loop and both TMEM
    accumulator buffers are reused several times."""
    cfg = moe.Config(T=1024, d_model=1024, n_experts=8, top_k=2, d_ff=2048, n_shared=0,
                     dtype=moe.MOE_BF16, act=act)
    counts = [512, 100, 300, 0, 260, 380, 200, 296]
    run_ffn(cfg, counts, 22, cuda_device)


def test_expert_ffn_bf16_single_row_experts(cuda_device):
    """Decode-like: one or two rows per expert, 64 experts."""
    cfg = moe.Config(T=64, d_model=512, n_experts=64, top_k=2, d_ff=256, n_shared=1,
                     dtype=moe.MOE_BF16, act=moe.MOE_SWIGLU)
    counts = [2 if e % 3 == 0 else (1 if e % 3 == 1 else 0) for e in range(64)]
    run_ffn(cfg, counts, 23, cuda_device)
