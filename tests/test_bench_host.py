"""The bench's launch accounting on the host: which expert-GEMM kernels and how
many launches a layer makes, as the library chooses them from the layer's
shape (the roofline's per-launch figures and the line's gpu_launches depend on
it). The per-step sequences follow the ncu launch lists of each workload."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_mixture_experts_69_b300 import moe  # noqa: E402
from sparse_mixture_experts_69_b300.workloads import WORKLOADS  # noqa: E402


@pytest.mark.parametrize("name,launches,kernel", [
    ("mixtral", 2, "grouped_gemm_pair_kernel"),       # 2048+ rows per expert: CTA pairs
    ("deepseek", 4, "grouped_gemm_tc_kernel + grouped_gemm_pair_kernel"),  # mixed sizes
    ("switch", 2, "grouped_gemm_tc_kernel"),
    ("decode", 2, "grouped_gemm_tc_kernel"),          # T <= 128
    ("tiny", 2, "grouped_gemm_simt_kernel"),          # fp32
])
def test_ffn_kernels_follow_the_layer_shape(name, launches, kernel):
    wl = WORKLOADS[name]
    n, k = bench.ffn_kernels(wl, moe.moe_capacity(wl.cfg)[1])
    assert n == launches
    assert k.startswith(kernel)


@pytest.mark.parametrize("name,per_step", [
    # transpose, router GEMM (it selects too), scan + slots, permute, up, down, combine
    ("mixtral", 7),
    # the same with two launches per projection, and the bias update
    ("deepseek", 11),
    # no combine launch: the top-1 down GEMM writes y
    ("switch", 7),
    ("decode", 8),
    # re-routing: one capacity kernel instead of scan + slots, and a combine
    # launch (a token has two candidates, so the down GEMM cannot scatter)
    ("switch_reroute", 8),
])
def test_launches_per_step(name, per_step):
    assert bench.launches_per_step(WORKLOADS[name]) == per_step


@pytest.mark.parametrize("T,d,E,noisy,fused", [
    (16384, 4096, 8, False, True),    # Mixtral-shaped: 148 tiles of 111 rows
    (2048, 256, 8, False, True),      # 4 K blocks: no split
    (2048, 4096, 8, False, False),    # 16 tiles: K split in 4 parts
    (10000, 512, 16, False, True),    # 148 tiles of 68 rows
    (8192, 1024, 32, True, False),    # noisy
    (64, 4096, 64, False, False),     # more than 32 experts
])
def test_router_selects_in_gemm(T, d, E, noisy, fused):
    c = WORKLOADS["mixtral"].with_(T=T, d_model=d, n_experts=E).cfg
    assert bench.router_selects_in_gemm(c, noisy) == fused
