"""Repeated launches on the same logits agree bit for bit.

Every thread of a row's cluster (or lane group) reduces the same partial
sums in one fixed order, whatever order the CTAs, warps and pushes arrive
in, and so takes the same search decisions; two launches must therefore
write the same probabilities, temperatures and error bits.  The cases cover
the fan launch, one-CTA rows, clusters of 2, 8 and 16 CTAs, and the
row-group kernel at 4 and 32 lanes a row."""
import numpy as np
import pytest

import oracle
from gpu_parity import compare, run_gpu

pytestmark = pytest.mark.gpu

# (variant, param, batch, classes)
CASES = [
    ("auto", 0, 32, 50000),
    ("cluster", 1, 40, 4099),
    ("cluster", 2, 24, 32000),
    ("cluster", 8, 6, 131072),
    ("cluster", 16, 3, 50001),
    ("rowgroup", 4, 512, 64),
    ("rowgroup", 32, 64, 1000),
]


@pytest.mark.parametrize("variant,param,B,C", CASES,
                         ids=[f"{c[0]}{c[1]}_{c[2]}x{c[3]}" for c in CASES])
def test_repeated_launches_agree(variant, param, B, C):
    x = np.random.default_rng(B * 7 + C).normal(0.0, 2.0, (B, C)).astype(np.float32)
    p1, T1, m1 = run_gpu(x, variant=variant, param=param)
    p2, T2, m2 = run_gpu(x, variant=variant, param=param)
    assert np.array_equal(p1.view(np.uint32), p2.view(np.uint32))
    assert np.array_equal(T1.view(np.uint32), T2.view(np.uint32))
    assert m1 == m2
    # And the launch is right, not just repeatable.
    compare(x, p1, T1, m1, oracle.constrained_softmax(x))
