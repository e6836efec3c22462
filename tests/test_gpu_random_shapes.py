"""The whole layer on seeded random shapes, every token against the oracle fed
the GPU's routing (counts bit-exact, y within the dtype's tolerance).

The shapes are drawn once from a fixed seed: odd expert counts and token
counts that leave ragged row tiles, d and F that are multiples of 8 but not of
the tile widths, 0-2 shared experts, dropless and capacity-limited layers, all
three activations and both dtypes. A few fixed cases make sure every
tensor-core path appears: expert GEMMs on CTA pairs (experts of 1024+ rows),
the two-launch FFN of mixed expert sizes (256..1023 rows per expert), and the
256-wide router on CTA pairs."""
import numpy as np
import pytest

from sparse_mixture_experts_69_b300 import moe
from sparse_mixture_experts_69_b300.workloads import Workload

pytestmark = pytest.mark.gpu


def _random_cases(n, seed=20261203):
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        E = int(rng.choice([1, 2, 3, 8, 17, 64, 130]))
        k = int(rng.randint(1, min(E, 8) + 1))
        T = int(rng.choice([1, 7, 100, 129, 300, 777]))
        d = int(rng.choice([64, 136, 264]))
        F = int(rng.choice([64, 200, 264]))
        S = int(rng.choice([0, 0, 1, 2]))
        cf = float(rng.choice([0.0, 0.0, 1.25, 2.0]))
        act = int(rng.choice([moe.MOE_RELU, moe.MOE_GELU, moe.MOE_SWIGLU]))
        dtype = moe.MOE_F32 if i % 4 == 3 else moe.MOE_BF16
        cases.append((f"r{i}", T, d, E, k, F, S, cf, act, dtype))
    return cases


FIXED = [
    # experts of 1024+ rows on average: CTA-pair expert GEMMs, ragged last tiles
    ("pairs", 2100, 136, 2, 1, 200, 1, 0.0, moe.MOE_SWIGLU, moe.MOE_BF16),
    ("pairs-relu", 3001, 64, 3, 2, 72, 0, 0.0, moe.MOE_RELU, moe.MOE_BF16),
    # 256..1023 rows per expert: two launches per projection
    ("split", 1000, 136, 8, 3, 200, 2, 0.0, moe.MOE_GELU, moe.MOE_BF16),
    # 256 experts: router GEMM on CTA pairs (T not a multiple of 256)
    ("router-pairs", 300, 264, 256, 8, 64, 1, 0.0, moe.MOE_SWIGLU, moe.MOE_BF16),
]


CASES = FIXED + _random_cases(12)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_layer_on_random_shapes(cuda_device, case):
    from gpu_helpers import layer_vs_oracle
    name, T, d, E, k, F, S, cf, act, dtype = case
    cfg = moe.Config(T=T, d_model=d, n_experts=E, top_k=k, d_ff=F, n_shared=S,
                     capacity_factor=cf, dtype=dtype, act=act)
    wl = Workload(name, cfg, seed=100 + CASES.index(case))
    o, _ = layer_vs_oracle(wl, cuda_device)
    counts = o["counts"].cpu().numpy()
    assert counts.sum() == T * k
