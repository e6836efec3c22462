"""The C ABI without a GPU: the library loads, exports every entry point that
include/moe.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from sparse_mixture_experts_69_b300 import build as moe_build
from sparse_mixture_experts_69_b300 import moe
from sparse_mixture_experts_69_b300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_layer_fwd",
               "moe_aux_stats", "moe_bias_update", "moe_workspace_size", "moe_status_string",
               "moe_read_device_error"]:
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(moe.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name
        assert name in moe._SIGS, f"binding lacks {name}"


def test_status_strings(lib):
    for code, name in moe.STATUS.items():
        assert moe.moe_status_string(code).startswith(name)
    assert moe.moe_status_string(99) == "unknown moe_status"


@pytest.mark.parametrize("name,C,R", [("tiny", 40, 320), ("switch", 128, 8192),
                                      ("mixtral", 16384, 32768), ("deepseek", 8192, 65536),
                                      ("decode", 64, 384)])
def test_capacity_of_the_workloads(lib, name, C, R):
    assert moe.moe_capacity(WORKLOADS[name].cfg) == (C, R)


def _cfg(**kw):
    base = dict(T=64, d_model=64, n_experts=8, top_k=2, d_ff=64, n_shared=0,
                capacity_factor=1.0, renorm_topk=1, dtype=moe.MOE_BF16, act=moe.MOE_SWIGLU)
    base.update(kw)
    return moe.Config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(top_k=9), 1), (dict(top_k=0), 1), (dict(T=0), 1), (dict(n_experts=0), 1),
    (dict(dtype=7), 1), (dict(act=3), 1), (dict(renorm_topk=2), 1), (dict(n_shared=-1), 1),
    (dict(capacity_factor=float("nan")), 1),
    (dict(d_model=60), 2), (dict(d_ff=100), 2), (dict(n_experts=2048, top_k=2), 2),
    (dict(top_k=33, n_experts=64), 2), (dict(n_shared=65), 2),
    # overflow policies and expert choice
    (dict(reroute=-1), 1), (dict(top_k=2, reroute=7), 1), (dict(priority=2), 1),
    (dict(pad_to_capacity=2), 1), (dict(routing=2), 1),
    (dict(routing=1, reroute=1), 1), (dict(routing=1, priority=1), 1),
    (dict(n_experts=64, top_k=8, reroute=25), 2),
    (dict(n_experts=600, reroute=1), 2), (dict(T=131073, priority=1), 2),
    (dict(T=32769, routing=1), 2),
])
def test_invalid_configs_rejected(lib, kw, status):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(_cfg(**kw))
    assert ei.value.status == status


def test_rows_bound_of_padding_and_expert_choice(lib):
    # dropping: min(T k, E C); padded or expert choice: E C
    assert moe.moe_capacity(_cfg(capacity_factor=0.5)) == (4, 32)
    assert moe.moe_capacity(_cfg(capacity_factor=4.0)) == (32, 128)
    assert moe.moe_capacity(_cfg(capacity_factor=4.0, pad_to_capacity=1)) == (32, 256)
    assert moe.moe_capacity(_cfg(capacity_factor=2.0, routing=moe.MOE_EXPERT_CHOICE)) == (16, 128)
    # candidates widen the per-token arrays in the workspace
    assert moe.moe_workspace_size(_cfg(reroute=2)) > moe.moe_workspace_size(_cfg())


def test_workspace_grows_with_the_problem(lib):
    a = moe.moe_workspace_size(_cfg())
    b = moe.moe_workspace_size(_cfg(T=128))
    c = moe.moe_workspace_size(_cfg(n_shared=2))
    assert 0 < a < b and a < c
    assert moe.moe_workspace_size(WORKLOADS["deepseek"].cfg) > 2 * 65536 * 7168 * 2


class _FakeTensor:
    """A device pointer stand-in: host validation must reject before using it."""

    def __init__(self, addr, n=1 << 40):
        self.addr, self.n = addr, n

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n


def test_host_validation_before_any_launch(lib):
    cfg = _cfg()
    L = moe.lib()
    c = ctypes.byref(cfg.c())
    A = 1 << 20  # aligned fake address, never dereferenced
    big = moe.moe_workspace_size(cfg)
    # NULL workspace
    assert L.moe_dispatch(c, A, A, A, A, A, A, A, A, None, big, None) == 1
    # workspace too small
    assert L.moe_dispatch(c, A, A, A, A, A, A, A, A, A, big - 1, None) == 3
    # missing required output
    assert L.moe_dispatch(c, A, A, None, A, A, A, A, A, A, big, None) == 1
    # misaligned activation pointer
    assert L.moe_dispatch(c, A + 4, A, A, A, A, A, A, A, A, big, None) == 2
    # noisy router needs both Wnoise and noise
    assert L.moe_route(c, A, A, A, None, None, None, A, A, None, A, A, 0, A, big, None) == 1
    # shared experts need their weights
    cs = _cfg(n_shared=1)
    bs = moe.moe_workspace_size(cs)
    assert L.moe_expert_ffn(ctypes.byref(cs.c()), A, A, A, A, A, None, A, A, A, A, bs, None) == 1
    assert L.moe_layer_fwd(c, A, A, None, None, None, None, None, A, None, None, A, None, None,
                           None, None, None, A, big, None) == 1
    assert L.moe_bias_update(c, None, A, 1e-3, None) == 1
    assert L.moe_bias_update(c, A, A, float("inf"), None) == 1


def test_host_validation_of_the_next_entry_points(lib):
    L = moe.lib()
    A = 1 << 20
    ec = _cfg(routing=moe.MOE_EXPERT_CHOICE, capacity_factor=2.0)
    big = moe.moe_workspace_size(ec)
    c = ctypes.byref(ec.c())
    # token-choice calls refuse an expert-choice config and vice versa
    assert L.moe_dispatch(c, A, A, A, A, A, A, A, A, A, big, None) == 1
    assert L.moe_combine(c, A, A, A, None, A, A, big, None) == 1
    tc = _cfg()
    tbig = moe.moe_workspace_size(tc)
    assert L.moe_expert_choice_dispatch(ctypes.byref(tc.c()), A, A, A, A, A, A, A, A, tbig,
                                        None) == 1
    assert L.moe_expert_choice_combine(ctypes.byref(tc.c()), A, A, A, None, A, A, tbig,
                                       None) == 1
    # missing outputs, misaligned rows
    assert L.moe_expert_choice_dispatch(c, A, A, A, None, A, A, A, A, big, None) == 1
    assert L.moe_expert_choice_dispatch(c, A + 4, A, A, A, A, A, A, A, big, None) == 2
    # the layer refuses token-choice outputs under expert choice
    assert L.moe_layer_fwd(c, A, A, None, None, None, None, A, A, None, None, A, A, None,
                           None, None, None, A, big, None) == 1
    # sequence statistics: need at least one sequence and the outputs
    assert L.moe_seq_aux_stats(ctypes.byref(tc.c()), A, A, A, 0, None, None, A, A, A, tbig,
                               None) == 1
    assert L.moe_seq_aux_stats(ctypes.byref(tc.c()), A, A, A, 4, None, None, None, A, A, tbig,
                               None) == 1
