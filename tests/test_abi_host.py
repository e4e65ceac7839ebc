"""The C ABI on the CPU: the library loads, exports every function the header
declares, and its host-only logic (argument checks, launch planning, status
strings) behaves as documented.  No CUDA call is made."""
import os
import re

import pytest

import entropy_bounded_softmax_gb300 as cs
from entropy_bounded_softmax_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "entropy_bounded_softmax.h")
GB300 = dict(sm_count=152, smem_per_block_optin=232448, smem_per_sm=233472,
             max_cluster=16)
C = _lib.CONSTANTS


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cs_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = _lib.load()
    declared = header_functions()
    assert "cs_constrained_softmax" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(_lib.exported_names()) == declared


def test_status_codes_follow_the_page():
    import json
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "kernel_api_constants.json")))
    codes = g["error_codes"]
    assert C["CS_OK"] == codes["SUCCESS"]
    for name in ("NAN_INPUT", "INF_INPUT", "ENTROPY_OVERFLOW",
                 "DIM_MISMATCH", "OOM"):
        assert C[f"CS_ERR_{name}"] == codes[name]
    assert cs.cs_status_string(C["CS_ERR_INVALID_ARG"]) == "invalid argument"
    assert cs.version().endswith("sm_103a")


def test_binding_defaults_follow_the_page():
    import inspect
    import json
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "kernel_api_constants.json")))["defaults"]
    sig = inspect.signature(cs.constrained_softmax)
    assert sig.parameters["entropy_bound"].default == g["entropy_bound"]
    assert sig.parameters["t_min"].default == g["temperature_min"]
    assert sig.parameters["t_max"].default == g["temperature_max"]
    assert sig.parameters["max_iter"].default == g["max_iterations"]


A, B = 1 << 20, 1 << 30   # two far-apart fake device addresses


@pytest.mark.parametrize("args,status", [
    ((A, B, 4, 10, 0.2, 0.01, 10.0, 20, None), 0),
    ((A, B, 0, 10, 0.2, 0.01, 10.0, 20, None), 0),
    ((None, None, 0, 10, 0.2, 0.01, 10.0, 20, None), 0),
    ((A, B, -1, 10, 0.2, 0.01, 10.0, 20, None), 6),
    ((A, B, 4, 0, 0.2, 0.01, 10.0, 20, None), 6),
    ((A, B, 2**62, 1000, 0.2, 0.01, 10.0, 20, None), 6),
    ((A, B, 4, 900000, 0.2, 0.01, 10.0, 20, None), 7),
    ((None, B, 4, 10, 0.2, 0.01, 10.0, 20, None), 8),
    ((A, None, 4, 10, 0.2, 0.01, 10.0, 20, None), 8),
    ((A, A + 40, 4, 10, 0.2, 0.01, 10.0, 20, None), 8),     # overlap
    ((A, A + 160, 4, 10, 0.2, 0.01, 10.0, 20, None), 0),    # adjacent
    ((A, B, 4, 10, 0.2, 0.01, 10.0, 20, A + 8), 8),         # t_out overlap
    ((A, B, 4, 10, float("nan"), 0.01, 10.0, 20, None), 8),
    ((A, B, 4, 10, float("inf"), 0.01, 10.0, 20, None), 0),
    ((A, B, 4, 10, -1.0, 0.01, 10.0, 20, None), 0),
    ((A, B, 4, 10, 0.2, 0.0, 10.0, 20, None), 8),
    ((A, B, 4, 10, 0.2, 1e-45, 10.0, 20, None), 8),         # subnormal
    ((A, B, 4, 10, 0.2, float("inf"), float("inf"), 20, None), 8),
    ((A, B, 4, 10, 0.2, 2.0**64, float("inf"), 20, None), 0),  # the cap
    ((A, B, 4, 10, 0.2, 2.0**65, float("inf"), 20, None), 8),  # above it
    ((A, B, 4, 10, 0.2, 0.01, 0.001, 20, None), 8),
    ((A, B, 4, 10, 0.2, 0.01, float("nan"), 20, None), 8),
    ((A, B, 4, 10, 0.2, 0.01, float("inf"), 20, None), 0),
    ((A, B, 4, 10, 0.2, 0.01, 10.0, -1, None), 8),
    ((A, B, 4, 10, 0.2, 0.01, 10.0, 1025, None), 8),
    ((A, B, 4, 10, 0.2, 0.01, 10.0, 0, None), 0),
])
def test_check_args(args, status):
    assert cs.cs_check_args(*args) == status


def plan(batch, classes, variant=0, param=0, threads=0, strict=0, **dev):
    d = dict(GB300, **dev)
    st, p = cs.cs_plan_host(batch, classes,
                            cs.options(variant, param, threads, strict),
                            d["sm_count"], d["smem_per_block_optin"],
                            d["smem_per_sm"], d["max_cluster"])
    return st, p.as_dict()


def test_auto_plans_for_the_workloads():
    st, p = plan(65536, 64)
    assert st == 0 and p["variant"] == C["CS_VARIANT_ROWGROUP"]
    assert p["lanes_per_row"] * p["elems_per_lane"] >= 64
    st, p = plan(32, 50000)
    assert st == 0 and p["variant"] == C["CS_VARIANT_CLUSTER"]
    assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
    st, p = plan(4096, 32000)
    assert st == 0 and p["cluster_size"] >= 1
    st, p = plan(256, 131072)
    assert st == 0 and p["cluster_size"] >= 3
    assert p["slice_len"] * p["cluster_size"] >= 131072
    assert p["grid_ctas"] == 256 * p["cluster_size"]


def test_middle_width_plans():
    # Up to 1024 classes: one warp a row, 32 classes a lane.
    for classes in (513, 1000, 1024):
        st, p = plan(4, classes)
        assert st == 0 and p["variant"] == C["CS_VARIANT_ROWGROUP"]
        assert p["lanes_per_row"] == 32 and p["elems_per_lane"] == 32
    st, p = plan(4, 1025)
    assert st == 0 and p["variant"] == C["CS_VARIANT_CLUSTER"]
    # Many one-CTA rows: 64-thread CTAs; few rows: at least 128.
    st, p = plan(4096, 2000)
    assert st == 0 and p["cluster_size"] == 1 and p["threads_per_cta"] == 64
    st, p = plan(4096, 8000)
    assert st == 0 and p["threads_per_cta"] == 128
    st, p = plan(4, 2000)
    assert st == 0 and p["threads_per_cta"] >= 128
    # The backward keeps its row-group kernel to 512 classes.
    st, p = cs.cs_plan_backward_host(4, 1000, None, *GB300.values())
    assert st == 0 and p.as_dict()["variant"] == C["CS_VARIANT_CLUSTER"]


def test_fan_only_for_one_wave_cluster_plans():
    # Few rows: the fan (temperatures evaluated with T = 1) and clusters of
    # a power of two that keep at most two CTAs on an SM.
    st, p = plan(32, 50000)
    assert st == 0 and p["fan_points"] == 3
    assert p["cluster_size"] == 8 and p["threads_per_cta"] == 128
    assert p["grid_ctas"] <= 2 * GB300["sm_count"]
    # strict bisects from the whole interval: no fan, the widened plan.
    st, p = plan(32, 50000, strict=1)
    assert st == 0 and p["fan_points"] == 0 and p["cluster_size"] == 10
    # Throughput launches (more than one wave) and one-CTA rows: none.
    for batch, classes in ((4096, 32000), (256, 131072), (65536, 64),
                           (4, 1000)):
        st, p = plan(batch, classes)
        assert st == 0 and p["fan_points"] == 0, (batch, classes)
    # Forced plans keep their shape; the fan follows the same rule.
    st, p = plan(32, 50000, variant=C["CS_VARIANT_CLUSTER"], param=10)
    assert st == 0 and p["cluster_size"] == 10 and p["fan_points"] == 3
    st, p = plan(32, 50000, variant=C["CS_VARIANT_CLUSTER"], param=4,
                 threads=512)
    assert st == 0 and p["fan_points"] == 0


@pytest.mark.parametrize("classes", [1, 3, 17, 64, 511, 512, 513, 1000,
                                     4099, 32000, 50001, 131072, 600000,
                                     850000])
def test_plans_hold_the_row(classes):
    st, p = plan(8, classes)
    assert st == 0
    if p["variant"] == C["CS_VARIANT_ROWGROUP"]:
        assert p["lanes_per_row"] * p["elems_per_lane"] >= classes
        assert p["lanes_per_row"] in (1, 2, 4, 8, 16, 32)
    else:
        n = p["cluster_size"]
        assert 1 <= n <= 16
        assert p["slice_len"] % 4 == 0
        assert n * p["slice_len"] >= classes
        assert (n - 1) * p["slice_len"] < classes or n == 1 or classes < 4 * n
        assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
        assert p["smem_bytes"] >= 4 * p["slice_len"]
        assert p["threads_per_cta"] % 32 == 0 and p["threads_per_cta"] <= 1024


def test_forced_variants_and_limits():
    st, _ = plan(8, 64, C["CS_VARIANT_ROWGROUP"], 1)
    assert st == C["CS_ERR_OOM"]          # 64 classes in one lane
    st, p = plan(8, 32, C["CS_VARIANT_ROWGROUP"], 1)
    assert st == 0 and p["elems_per_lane"] == 32
    st, _ = plan(8, 4096, C["CS_VARIANT_ROWGROUP"], 32)
    assert st == C["CS_ERR_OOM"]          # 128 classes per lane
    st, _ = plan(8, 64, C["CS_VARIANT_ROWGROUP"], 3)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = plan(8, 64, C["CS_VARIANT_CLUSTER"], 17)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = plan(8, 131072, C["CS_VARIANT_CLUSTER"], 1)
    assert st == C["CS_ERR_OOM"]
    st, p = plan(8, 131072, C["CS_VARIANT_CLUSTER"], 16)
    assert st == 0 and p["slice_len"] == 8192
    st, _ = plan(8, 131072, C["CS_VARIANT_CLUSTER"], 8, max_cluster=4)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = plan(8, 64, C["CS_VARIANT_AUTO"], 4)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = plan(8, 64, 7, 0)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = plan(8, 850000, C["CS_VARIANT_CLUSTER"], 0, max_cluster=8)
    assert st == C["CS_ERR_OOM"]
    for bad in (dict(threads=48), dict(threads=544), dict(threads=100),
                dict(strict=2)):
        st, _ = plan(8, 50000, C["CS_VARIANT_CLUSTER"], 0, **bad)
        assert st == C["CS_ERR_INVALID_ARG"], bad
    st, _ = plan(8, 64, C["CS_VARIANT_ROWGROUP"], 0, threads=256)
    assert st == C["CS_ERR_INVALID_ARG"]


def test_null_options_mean_automatic():
    st1, p1 = cs.cs_plan_host(32, 50000, None, 152, 232448, 233472, 16)
    st2, p2 = plan(32, 50000)
    assert st1 == st2 == 0 and p1.as_dict() == p2


def test_strict_option_is_checked():
    st, _ = plan(32, 50000, strict=1)
    assert st == 0
    st, _ = plan(32, 50000, strict=2)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, p = plan(8, 4096, C["CS_VARIANT_CLUSTER"], 2, threads=512)
    assert st == 0 and p["threads_per_cta"] == 512 and p["cluster_size"] == 2
    st, _ = plan(8, 4096, C["CS_VARIANT_CLUSTER"], 2, threads=1024)
    assert st == C["CS_ERR_INVALID_ARG"]


# ------------------------------------------------------------------ backward
@pytest.mark.parametrize("args,status", [
    ((A, B, A + 4096, B + 4096, 4, 10), 0),
    ((A, A, A + 4096, B, 4, 10), 0),            # probs == grad_out
    ((A, B, B + 4096, A, 4, 10), 0),            # in place over probs
    ((A, B, A + 4096, B, 4, 10), 0),            # in place over grad_out
    ((None, None, None, None, 0, 10), 0),
    ((A, B, A + 4096, B + 4096, -1, 10), 6),
    ((A, B, A + 4096, B + 4096, 4, 0), 6),
    ((A, B, A + 4096, B + 4096, 2**62, 1000), 6),
    ((A, B, A + 4096, B + 4096, 4, 900000), 7),
    ((None, B, A + 4096, B + 4096, 4, 10), 8),
    ((A, None, A + 4096, B + 4096, 4, 10), 8),
    ((A, B, None, B + 4096, 4, 10), 8),
    ((A, B, A + 4096, None, 4, 10), 8),
    ((A, B, A + 4096, A + 4, 4, 10), 8),        # grad overlaps probs
    ((A, B, A + 4096, B + 156, 4, 10), 8),      # grad overlaps grad_out
    ((A, B, B + 4100, B + 4096, 4, 10), 8),     # t overlaps grad
    ((A, B, A + 8, B + 4096, 4, 10), 0),        # t overlaps probs (reads)
    ((A, B, A + 4096, B + 160, 4, 10), 0),      # adjacent
])
def test_check_backward_args(args, status):
    assert cs.cs_check_backward_args(*args) == status


def bplan(batch, classes, variant=0, param=0, threads=0, strict=0, **dev):
    d = dict(GB300, **dev)
    st, p = cs.cs_plan_backward_host(
        batch, classes, cs.options(variant, param, threads, strict),
        d["sm_count"], d["smem_per_block_optin"], d["smem_per_sm"],
        d["max_cluster"])
    return st, p.as_dict()


def test_backward_plans_for_the_workloads():
    st, p = bplan(65536, 64)
    assert st == 0 and p["variant"] == C["CS_VARIANT_ROWGROUP"]
    assert p["lanes_per_row"] * p["elems_per_lane"] >= 64 + 6
    st, p = bplan(4096, 32000)
    assert st == 0 and p["variant"] == C["CS_VARIANT_CLUSTER"]
    assert (p["cluster_size"], p["slice_len"], p["staged_tensors"]) == \
        (4, 8000, 2)
    assert p["grid_ctas"] == 4096 * 4 and p["ctas_per_sm"] >= 3
    st, p = bplan(32, 50000)
    assert st == 0 and p["grid_ctas"] >= GB300["sm_count"]
    st, p = bplan(256, 131072)
    assert st == 0 and (p["cluster_size"], p["slice_len"]) == (16, 8192)
    st, p = bplan(4, 850000)
    assert st == 0 and p["cluster_size"] == 16 and p["staged_tensors"] == 1


@pytest.mark.parametrize("classes", [1, 3, 17, 64, 511, 512, 513, 1000,
                                     4099, 8193, 32000, 50001, 131072,
                                     464000, 600000, 850000])
@pytest.mark.parametrize("batch", [1, 8, 4096])
def test_backward_plans_hold_the_row(classes, batch):
    st, p = bplan(batch, classes)
    assert st == 0
    if p["variant"] == C["CS_VARIANT_ROWGROUP"]:
        # Room for the row at its worst alignment (3 floats of lead-in).
        assert p["lanes_per_row"] * p["elems_per_lane"] >= classes + 6 - 3
        assert p["elems_per_lane"] in (4, 8, 16, 32)
        assert p["grid_ctas"] * p["threads_per_cta"] >= \
            batch * p["lanes_per_row"]
    else:
        n, L = p["cluster_size"], p["slice_len"]
        assert 1 <= n <= 16 and L % 4 == 0 and n * L >= classes
        assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
        assert p["smem_bytes"] >= 512 + (L // 4 + 1) * 16 * p["staged_tensors"]
        assert p["staged_tensors"] in (1, 2)
        assert 64 <= p["threads_per_cta"] <= 512
        assert p["threads_per_cta"] % 32 == 0
        assert p["grid_ctas"] == batch * n


def test_backward_forced_variants_and_limits():
    st, p = bplan(8, 50001, C["CS_VARIANT_CLUSTER"], 1)
    assert st == 0 and p["staged_tensors"] == 1
    st, p = bplan(8, 20000, C["CS_VARIANT_CLUSTER"], 1)
    assert st == 0 and p["staged_tensors"] == 2
    st, _ = bplan(8, 131072, C["CS_VARIANT_CLUSTER"], 1)
    assert st == C["CS_ERR_OOM"]
    st, _ = bplan(8, 100, C["CS_VARIANT_ROWGROUP"], 1)
    assert st == C["CS_ERR_OOM"]
    st, p = bplan(8, 26, C["CS_VARIANT_ROWGROUP"], 1)
    assert st == 0 and p["elems_per_lane"] == 32
    st, _ = bplan(8, 64, C["CS_VARIANT_ROWGROUP"], 3)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = bplan(8, 64, C["CS_VARIANT_CLUSTER"], 17)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = bplan(8, 850000, C["CS_VARIANT_CLUSTER"], 0, max_cluster=8)
    assert st == C["CS_ERR_OOM"]
    for bad in (dict(threads=48), dict(threads=544), dict(threads=100),
                dict(strict=1)):
        st, _ = bplan(8, 50000, C["CS_VARIANT_CLUSTER"], 0, **bad)
        assert st == C["CS_ERR_INVALID_ARG"], bad
    st, _ = bplan(8, 64, C["CS_VARIANT_AUTO"], 4)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = bplan(8, 64, C["CS_VARIANT_ROWGROUP"], 0, threads=256)
    assert st == C["CS_ERR_INVALID_ARG"]
    st1, p1 = cs.cs_plan_backward_host(32, 50000, None, 152, 232448, 233472,
                                       16)
    assert st1 == 0 and p1.as_dict() == bplan(32, 50000)[1]


# ----------------------------------------------------------------- attention
@pytest.mark.parametrize("args,status", [
    ((A, B, None, 2, 2, 8, 0), 0),
    ((A, A, None, 2, 2, 8, 1), 0),                # in place
    ((A, B, A + 8192, 2, 2, 8, 0), 0),            # mask beside the scores
    ((None, None, None, 0, 2, 8, 0), 0),
    ((None, None, None, 2, 0, 8, 0), 0),
    ((None, None, None, 2, 2, 0, 0), 0),
    ((A, B, None, -1, 2, 8, 0), 6),
    ((A, B, None, 2, -2, 8, 0), 6),
    ((A, B, None, 2, 2, -8, 0), 6),
    ((A, B, None, 2, 2, 8, 2), 8),                # causal not 0/1
    ((A, B, None, 1, 1, 60000, 0), 7),
    ((None, B, None, 2, 2, 8, 0), 8),
    ((A, None, None, 2, 2, 8, 0), 8),
    ((A, A + 16, None, 2, 2, 8, 0), 8),           # partial overlap
    ((A, B, B + 64, 2, 2, 8, 0), 8),              # mask overlaps out
    ((A, B, A + 64, 2, 2, 8, 0), 0),              # mask overlaps scores
])
def test_check_attention_args(args, status):
    assert cs.cs_check_attention_args(*args) == status


def aplan(batch, heads, S, aligned=1, variant=0, param=0, threads=0,
          strict=0):
    st, p = cs.cs_plan_attention_host(
        batch, heads, S, aligned, cs.options(variant, param, threads, strict),
        GB300["sm_count"], GB300["smem_per_block_optin"],
        GB300["smem_per_sm"])
    return st, p.as_dict()


def test_attention_plans_for_the_workloads():
    st, p = aplan(32, 8, 512)
    assert st == 0 and p["variant"] == C["CS_VARIANT_ROWGROUP"]
    assert (p["lanes_per_row"], p["elems_per_lane"]) == (32, 16)
    assert p["grid_ctas"] * p["threads_per_cta"] == 32 * 8 * 512 * 32
    st, p = aplan(2, 8, 4096)
    assert st == 0 and p["variant"] == C["CS_VARIANT_CLUSTER"]
    assert p["cluster_size"] == 1 and p["grid_ctas"] == 2 * 8 * 4096
    assert p["smem_bytes"] >= 512 + 4096 * 4


@pytest.mark.parametrize("S", [1, 2, 3, 5, 64, 127, 512, 1017, 1018, 1024,
                               1025, 4096, 57344])
@pytest.mark.parametrize("aligned", [0, 1])
def test_attention_plans_hold_the_row(S, aligned):
    st, p = aplan(1, 1, S, aligned)
    assert st == 0
    if p["variant"] == C["CS_VARIANT_ROWGROUP"]:
        q = (S + 3) // 4 if aligned else (S + 6) // 4
        assert p["lanes_per_row"] * p["elems_per_lane"] >= 4 * q
    else:
        assert p["smem_bytes"] <= GB300["smem_per_block_optin"]
        assert p["smem_bytes"] >= 512 + 16 * ((S + 6) // 4)
        assert 64 <= p["threads_per_cta"] <= 512
        assert p["threads_per_cta"] % 32 == 0


def test_attention_forced_variants_and_limits():
    st, _ = aplan(1, 1, 100, 1, C["CS_VARIANT_ROWGROUP"], 1)
    assert st == C["CS_ERR_OOM"]
    st, p = aplan(1, 1, 32, 1, C["CS_VARIANT_ROWGROUP"], 1)
    assert st == 0 and p["elems_per_lane"] == 32
    st, _ = aplan(1, 1, 64, 1, C["CS_VARIANT_ROWGROUP"], 3)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = aplan(1, 1, 64, 1, C["CS_VARIANT_CLUSTER"], 2)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, p = aplan(1, 1, 64, 1, C["CS_VARIANT_CLUSTER"], 1, 96)
    assert st == 0 and p["threads_per_cta"] == 96
    for bad in (dict(threads=48), dict(threads=544), dict(strict=1)):
        st, _ = aplan(1, 1, 2048, 1, C["CS_VARIANT_CLUSTER"], 0, **bad)
        assert st == C["CS_ERR_INVALID_ARG"], bad
    st, _ = aplan(1, 1, 64, 1, C["CS_VARIANT_AUTO"], 4)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = aplan(1, 1, 64, 2)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = aplan(1, 1, 60000)
    assert st == C["CS_ERR_OOM"]


# ---------------------------------------------------------- biencoder_attention
Q0, K0, V0, O0 = 1 << 20, 1 << 24, 1 << 26, 1 << 28


@pytest.mark.parametrize("args,status", [
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 0),
    ((None, None, None, None, 0, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 0),
    ((Q0, K0, V0, O0, 2, 8, 0, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 6),
    ((Q0, K0, V0, O0, -1, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 6),
    ((Q0, K0, V0, O0, 2, 8, 257, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 7),
    ((Q0, K0, V0, O0, 2, 8, 64, 260, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 7),
    ((Q0, K0, V0, O0, 2, 8, 64, 62, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 8),
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, float("inf"), 0.2, 0.01, 10.0, 20, None, None), 8),
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, float("nan"), 0.01, 10.0, 20, None, None), 8),
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.0, 10.0, 20, None, None), 8),
    ((Q0 + 4, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 8),
    ((Q0, K0, V0, Q0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 8),
    ((Q0, K0, V0, K0 + 16, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, None), 8),
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, O0 + 64, None), 8),
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, None, V0), 8),
    ((Q0, K0, V0, O0, 2, 8, 64, 64, 4, 0.125, 0.2, 0.01, 10.0, 20, 1 << 30, (1 << 30) + 16384 * 4), 0),
])
def test_check_biencoder_args(args, status):
    assert cs.cs_check_biencoder_args(*args) == status


def test_biencoder_plans():
    st, p = cs.cs_plan_biencoder_host(32, 512, 64, 64, 8, None, 232448)
    p = p.as_dict()
    assert st == 0 and p["lanes_per_row"] == 4 and p["threads_per_cta"] == 256
    assert p["elems_per_lane"] == 16
    assert p["grid_ctas"] == 32 * 8 * (512 // 128)
    st, p = cs.cs_plan_biencoder_host(4, 1024, 256, 64, 8, None, 232448)
    assert st == 0 and p.lanes_per_row == 16 and p.elems_per_lane == 16
    assert p.smem_bytes <= 232448
    st, _ = cs.cs_plan_biencoder_host(4, 1024, 256, 128, 8, None, 232448)
    assert st == C["CS_ERR_OOM"]            # keys and values exceed smem
    for K in (1, 8, 9, 16, 17, 64, 65, 256):
        # by default sixteen items a lane, on the fewest lanes that hold K
        st, p = cs.cs_plan_biencoder_host(1, 10, K, 16, 1, None, 232448)
        assert st == 0 and 16 * p.lanes_per_row >= K
        assert p.lanes_per_row == 1 or 8 * p.lanes_per_row < K
        assert p.elems_per_lane == 16
    st, _ = cs.cs_plan_biencoder_host(1, 10, 40, 16, 1,
                                      cs.options(C["CS_VARIANT_ROWGROUP"], 2),
                                      232448)
    assert st == C["CS_ERR_OOM"]            # two lanes hold at most 32 items
    st, p = cs.cs_plan_biencoder_host(1, 10, 40, 16, 1,
                                      cs.options(C["CS_VARIANT_ROWGROUP"], 4),
                                      232448)
    assert st == 0 and (p.lanes_per_row, p.elems_per_lane) == (4, 16)
    st, p = cs.cs_plan_biencoder_host(1, 10, 40, 16, 1,
                                      cs.options(C["CS_VARIANT_ROWGROUP"], 8),
                                      232448)
    assert st == 0 and (p.lanes_per_row, p.elems_per_lane) == (8, 8)
    st, _ = cs.cs_plan_biencoder_host(1, 10, 40, 16, 1,
                                      cs.options(C["CS_VARIANT_CLUSTER"], 1),
                                      232448)
    assert st == C["CS_ERR_INVALID_ARG"]


def test_evaluation_counts_only_for_the_forward():
    """cs_options.evals_out is an output of cs_constrained_softmax_ex; the
    planners of the other operations reject it."""
    opt = cs.options(0, 0, 0, 0, A)
    st, _ = cs.cs_plan_host(4, 1000, opt, *GB300.values())
    assert st == 0
    st, _ = cs.cs_plan_backward_host(4, 1000, opt, *GB300.values())
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = cs.cs_plan_attention_host(1, 1, 64, 1, opt, 152, 232448, 233472)
    assert st == C["CS_ERR_INVALID_ARG"]
    st, _ = cs.cs_plan_biencoder_host(1, 8, 64, 64, 1, opt, 232448)
    assert st == C["CS_ERR_INVALID_ARG"]


def test_biencoder_plans_step3_on_the_tensor_cores():
    """The page's shape (64 context items, d_head 64) runs step 3 as a
    tensor-core kernel; a longer context, a larger head or the fused
    variant run one kernel."""
    def bplan(K, D, opt=None):
        st, p = cs.cs_plan_biencoder_host(32, 512, K, D, 8, opt, 232448)
        assert st == 0
        return p.as_dict()
    p = bplan(64, 64)
    assert p["tensor_cores"] == 1 and p["staged_tensors"] == 2
    assert bplan(12, 12)["tensor_cores"] == 1
    assert bplan(256, 64)["tensor_cores"] == 0      # context longer than the head
    assert bplan(64, 128)["tensor_cores"] == 0      # head above 64
    fused = bplan(64, 64, cs.options(C["CS_VARIANT_FUSED"], 0))
    assert fused["tensor_cores"] == 0 and fused["staged_tensors"] == 3
    assert fused["lanes_per_row"] == p["lanes_per_row"] == 4
