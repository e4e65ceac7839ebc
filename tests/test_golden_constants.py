"""The values the page prints, held against the oracle (CPU only)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "kernel_api_constants.json")


def load():
    with open(GOLDEN) as f:
        return json.load(f)


def test_oracle_flags_use_page_codes(oracle_lib):
    codes = load()["error_codes"]
    assert oracle.FLAG_NONE == codes["SUCCESS"]
    assert oracle.FLAG_NAN_INPUT == codes["NAN_INPUT"]
    assert oracle.FLAG_INF_INPUT == codes["INF_INPUT"]
    assert oracle.FLAG_ENTROPY_OVERFLOW == codes["ENTROPY_OVERFLOW"]
    x = np.array([[0.0, np.nan], [0.0, np.inf], [1.0, 1.0]], np.float32)
    r = oracle.constrained_softmax(x, lib=oracle_lib)
    assert list(r.flags) == [codes["NAN_INPUT"], codes["INF_INPUT"],
                             codes["ENTROPY_OVERFLOW"]]


def test_oracle_defaults_match_page():
    import inspect
    d = load()["defaults"]
    sig = inspect.signature(oracle.constrained_softmax)
    assert sig.parameters["entropy_bound"].default == d["entropy_bound"]
    assert sig.parameters["t_min"].default == d["temperature_min"]
    assert sig.parameters["t_max"].default == d["temperature_max"]
    assert sig.parameters["max_iter"].default == d["max_iterations"]


def test_search_is_at_least_as_precise_as_page_states():
    """The page quotes ~1e-5 after 20 halvings of [0.01, 10]; searching
    only [0.01, min(1, 10)] (temperatures above 1 cannot lower H) makes the
    final bracket ten times narrower."""
    g = load()["search_precision"]
    lo, hi = g["interval"]
    page_width = (hi - lo) / 2 ** g["iterations"]
    assert abs(page_width - g["stated_precision"]) / g["stated_precision"] < 0.05
    ours = oracle.final_interval(lo, hi, g["iterations"])
    assert ours <= page_width and ours <= g["stated_precision"]
