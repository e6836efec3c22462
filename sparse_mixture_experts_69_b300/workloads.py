"""The five synthetic MoE-layer workloads and their seeded inputs.

Shapes follow the models the pages name (Switch top-1, Mixtral top-2,
DeepSeek-V3 fine-grained + shared, a decode batch); every value comes from
``synth`` (counter-based, CPU/GPU bit-identical). Nothing here computes any
part of the layer.

  tiny     T=256   d=128  E=8   k=2 F=256   GELU,   cf=1.25 (C=40), fp32
  switch   T=8192  d=1024 E=64  k=1 F=4096  ReLU,   cf=1.0 (C=128), noisy KeepTopK
           with the noise tensor [T,E] generated on the host and passed in, bf16
  mixtral  T=16384 d=4096 E=8   k=2 F=14336 SwiGLU, dropless, Zipf(1.2) logit offset, bf16
  deepseek T=8192  d=7168 E=256 k=8 F=2048  SwiGLU, 1 shared, dropless, selection bias
           U(-0.1,0.1), one bias update at rate 1e-3, bf16
  decode   T=64    d=4096 E=64  k=6 F=1408  SwiGLU, 2 shared, dropless, bf16

Variants of the Switch layer (same inputs):
  switch_drawn    the router noise drawn by the library in the selection kernel
                  (noise_draw = 1) instead of passed in
  switch_reroute  a full expert sends the token to its next candidate (1 extra)
  switch_rank     the same, every token's first choice served before any second
  switch_pad      plain dropping, every expert's block padded to C = 128 rows
  switch_ec       expert choice: each expert takes its 128 most probable tokens

Input recipe: x ~ N(0,1); Wg, Wnoise, W1, W2, W1s, W2s ~ N(0, 0.02^2). The
router noise [T,E] ~ N(0,1) of the Switch layers is generated here and passed
in; switch_drawn has the library draw it from (noise_seed, noise_counter)
(moe_draw_noise) instead.
"""
from __future__ import annotations

import dataclasses

import torch

from . import synth
from .moe import (MOE_BF16, MOE_EXPERT_CHOICE, MOE_F32, MOE_GELU, MOE_PRIORITY_RANK,
                  MOE_RELU, MOE_SWIGLU, Config)

W_STD = 0.02


@dataclasses.dataclass
class Workload:
    name: str
    cfg: Config
    noisy: bool = False          # KeepTopK noise: Wnoise, plus a noise tensor unless
                                 # cfg.noise_draw (then the library draws it)
    zipf_s: float = 0.0          # > 0: logit offset -s ln(e+1)
    sel_bias: bool = False       # selection bias ~ U(-0.1, 0.1)
    bias_rate: float = 0.0       # > 0: one bias update per step
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        """Copy with some Config fields (T, d_model, ...) or Workload fields replaced."""
        cfg_kw = {k: v for k, v in kw.items() if k in Config.__dataclass_fields__}
        wl_kw = {k: v for k, v in kw.items() if k not in cfg_kw}
        return dataclasses.replace(self, cfg=dataclasses.replace(self.cfg, **cfg_kw), **wl_kw)


WORKLOADS = {
    "tiny": Workload("tiny", Config(T=256, d_model=128, n_experts=8, top_k=2, d_ff=256,
                                    capacity_factor=1.25, dtype=MOE_F32, act=MOE_GELU)),
    "switch": Workload("switch", Config(T=8192, d_model=1024, n_experts=64, top_k=1, d_ff=4096,
                                        capacity_factor=1.0, dtype=MOE_BF16, act=MOE_RELU),
                       noisy=True),
    "mixtral": Workload("mixtral", Config(T=16384, d_model=4096, n_experts=8, top_k=2,
                                          d_ff=14336, capacity_factor=0.0, dtype=MOE_BF16,
                                          act=MOE_SWIGLU), zipf_s=1.2),
    "deepseek": Workload("deepseek", Config(T=8192, d_model=7168, n_experts=256, top_k=8,
                                            d_ff=2048, n_shared=1, capacity_factor=0.0,
                                            dtype=MOE_BF16, act=MOE_SWIGLU),
                         sel_bias=True, bias_rate=1e-3),
    "decode": Workload("decode", Config(T=64, d_model=4096, n_experts=64, top_k=6, d_ff=1408,
                                        n_shared=2, capacity_factor=0.0, dtype=MOE_BF16,
                                        act=MOE_SWIGLU)),
}
WORKLOADS["switch_drawn"] = WORKLOADS["switch"].with_(name="switch_drawn", noise_draw=1,
                                                      noise_seed=0x5EED)
WORKLOADS["switch_reroute"] = WORKLOADS["switch"].with_(name="switch_reroute", reroute=1)
WORKLOADS["switch_rank"] = WORKLOADS["switch"].with_(name="switch_rank", reroute=1,
                                                     priority=MOE_PRIORITY_RANK)
WORKLOADS["switch_pad"] = WORKLOADS["switch"].with_(name="switch_pad", pad_to_capacity=1)
WORKLOADS["switch_ec"] = WORKLOADS["switch"].with_(name="switch_ec", routing=MOE_EXPERT_CHOICE)


def make_inputs(wl: Workload, device="cuda", experts: bool = True) -> dict:
    """All layer inputs of a workload as tensors on ``device`` (expert weights
    left out, as None, when ``experts`` is False)."""
    c = wl.cfg
    dt = c.torch_dtype
    T, d, E, F, F1, S = c.T, c.d_model, c.n_experts, c.d_ff, c.F1, c.n_shared
    s = wl.seed
    out = {
        "x": synth.normal((T, d), s, synth.TID_X, 1.0, dt, device),
        "Wg": synth.normal((d, E), s, synth.TID_WG, W_STD, dt, device),
        "Wnoise": None, "noise": None, "logit_offset": None, "sel_bias": None,
        "W1": synth.normal((E, F1, d), s, synth.TID_W1, W_STD, dt, device) if experts else None,
        "W2": synth.normal((E, d, F), s, synth.TID_W2, W_STD, dt, device) if experts else None,
        "W1s": None, "W2s": None,
    }
    if wl.noisy:
        out["Wnoise"] = synth.normal((d, E), s, synth.TID_WNOISE, W_STD, dt, device)
        if not c.noise_draw:
            out["noise"] = synth.normal((T, E), s, synth.TID_NOISE, 1.0, torch.float32,
                                        "cpu").to(device)
    if wl.zipf_s > 0:
        out["logit_offset"] = synth.zipf_logit_offset(E, wl.zipf_s).to(device)
    if wl.sel_bias:
        out["sel_bias"] = synth.uniform((E,), s, synth.TID_BIAS, -0.1, 0.1).to(device)
    if S and experts:
        out["W1s"] = synth.normal((S, F1, d), s, synth.TID_W1S, W_STD, dt, device)
        out["W2s"] = synth.normal((S, d, F), s, synth.TID_W2S, W_STD, dt, device)
    return out
