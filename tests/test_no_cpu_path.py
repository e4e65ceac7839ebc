"""The product path has no CPU fallback: every public operation refuses
tensors that are not on a CUDA device, and loading the library from a path
where it is absent raises instead of substituting anything.  CPU only."""
import os

import pytest

torch = pytest.importorskip("torch")

import entropy_bounded_softmax_gb300 as cs
from entropy_bounded_softmax_gb300 import _lib


def test_forward_refuses_cpu_tensors():
    with pytest.raises(ValueError):
        cs.constrained_softmax(torch.zeros(2, 8))


def test_backward_refuses_cpu_tensors():
    p = torch.full((2, 8), 0.125)
    with pytest.raises(ValueError):
        cs.constrained_softmax_backward(p, p.clone(), torch.ones(2))


def test_attention_refuses_cpu_tensors():
    with pytest.raises(ValueError):
        cs.attention_softmax(torch.zeros(1, 1, 4, 4))


def test_biencoder_refuses_cpu_tensors():
    q = torch.zeros(1, 1, 4, 8)
    with pytest.raises(ValueError):
        cs.biencoder_attention(q, q, q)


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError):
        _lib.load(os.path.join(str(tmp_path), "libcsoftmax.so"))


def test_autograd_function_is_built_on_the_kernels():
    fn = cs.ConstrainedSoftmaxFunction
    assert issubclass(fn, torch.autograd.Function)
    with pytest.raises(ValueError):
        fn.apply(torch.zeros(2, 8, requires_grad=True))
