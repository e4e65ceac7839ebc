"""Entropy-bounded softmax (``constrained_softmax``) for GB300 (sm_103a).

For each row of a [batch, num_classes] fp32 logit matrix: softmax and its
entropy; if the entropy exceeds ``entropy_bound`` the temperature is bisected
on [t_min, min(1, t_max)] for ``max_iter`` steps and softmax(l / T) is
written ("BURT-IMMA CUDA Kernel API Reference", section 2.1);
:func:`attention_softmax` is section 2.6's masked, optionally causal row
softmax of attention scores.  The backward
(section 6.3, with the 1/T of softmax(l / T) restored) gives the gradient
with respect to the logits; :class:`ConstrainedSoftmaxFunction` joins the two
for autograd.

PyTorch supplies device memory and the current stream; the computation runs
in the hand-written CUDA kernels of ``libcsoftmax.so`` behind a C ABI
(``include/entropy_bounded_softmax.h``).  There is no CPU path: the calls
raise if the library is missing or the tensors are not on a CUDA device.
"""
from __future__ import annotations

from . import _lib
from ._lib import (CONSTANTS, cs_attention_softmax, cs_attention_softmax_ex,
                   cs_biencoder_attention, cs_biencoder_attention_ex,
                   cs_check_biencoder_args, cs_plan_biencoder_host,
                   cs_check_args, cs_check_attention_args,
                   cs_check_backward_args, cs_constrained_softmax,
                   cs_constrained_softmax_backward,
                   cs_constrained_softmax_backward_ex,
                   cs_constrained_softmax_ex, cs_get_error,
                   cs_constrained_softmax_bf16, cs_constrained_softmax_bf16_ex,
                   cs_check_args_bf16,
                   cs_plan_attention_host, cs_plan_attention_launch,
                   cs_plan_backward_host, cs_plan_backward_launch,
                   cs_plan_host, cs_plan_launch, cs_probe_ex2,
                   cs_probe_ex2_sink_floats, cs_status_string,
                   cs_test_wait_timeout, cs_version, options)

__all__ = [
    "constrained_softmax", "constrained_softmax_backward",
    "ConstrainedSoftmaxFunction", "get_error", "plan", "plan_backward",
    "version", "CsError", "ERROR_BITS", "VARIANTS", "options",
    "cs_constrained_softmax", "cs_constrained_softmax_ex",
    "cs_constrained_softmax_bf16", "cs_constrained_softmax_bf16_ex",
    "cs_check_args_bf16",
    "cs_constrained_softmax_backward", "cs_constrained_softmax_backward_ex",
    "cs_get_error", "cs_plan_launch", "cs_plan_host",
    "cs_plan_backward_launch", "cs_plan_backward_host", "cs_check_args",
    "cs_check_backward_args", "cs_probe_ex2", "cs_probe_ex2_sink_floats",
    "cs_test_wait_timeout", "cs_version", "cs_status_string",
    "attention_softmax", "plan_attention", "cs_attention_softmax",
    "cs_attention_softmax_ex", "cs_plan_attention_launch",
    "cs_plan_attention_host", "cs_check_attention_args",
    "biencoder_attention", "cs_biencoder_attention",
    "cs_biencoder_attention_ex", "cs_plan_biencoder_host",
    "cs_check_biencoder_args",
]

# Defaults of section 2.1's signature.
DEFAULT_ENTROPY_BOUND = 0.20
DEFAULT_T_MIN = 0.01
DEFAULT_T_MAX = 10.0
DEFAULT_MAX_ITER = 20

VARIANTS = {"auto": CONSTANTS["CS_VARIANT_AUTO"],
            "rowgroup": CONSTANTS["CS_VARIANT_ROWGROUP"],
            "cluster": CONSTANTS["CS_VARIANT_CLUSTER"]}
ERROR_BITS = {name: 1 << CONSTANTS[f"CS_ERR_{name}"]
              for name in ("NAN_INPUT", "INF_INPUT", "ENTROPY_OVERFLOW",
                           "TIMEOUT")}


class CsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} "
                         f"({_lib.cs_status_string(status)})")


def _stream_handle(device) -> int:
    """The raw cudaStream_t of the current stream of a CUDA device."""
    import torch
    idx = device.index if device.index is not None else torch.cuda.current_device()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _on_device(device):
    """A context that makes `device` current: none when it already is (the
    common case, and the cheapest: the call is on every step's path)."""
    import contextlib
    import torch
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def constrained_softmax(logits, entropy_bound: float = DEFAULT_ENTROPY_BOUND,
                        t_min: float = DEFAULT_T_MIN,
                        t_max: float = DEFAULT_T_MAX,
                        max_iter: int = DEFAULT_MAX_ITER,
                        return_t: bool = False, out=None, t_out=None,
                        variant: str = "auto", param: int = 0,
                        threads: int = 0, strict: bool = False,
                        evals_out=None):
    """Entropy-bounded softmax of a CUDA [batch, num_classes] tensor of fp32
    logits, or of bf16 logits (``cs_constrained_softmax_bf16``: promoted
    exactly to fp32 on load; the probabilities are fp32 either way).

    Returns the probabilities (and the per-row temperature if ``return_t``).
    ``out``/``t_out`` may be given to write into existing tensors.  The call
    is asynchronous on the current stream; per-row conditions (NaN/Inf rows,
    unsatisfiable bounds) are read with :func:`get_error`.
    ``variant``/``param``/``threads``/``strict`` are the launch options
    of ``cs_constrained_softmax_ex`` (defaults: automatic); ``evals_out``, an
    int32 [batch] tensor on the same device, receives how many temperatures
    each row's exponentials were evaluated at.
    """
    import torch
    if not isinstance(logits, torch.Tensor):
        raise TypeError("logits must be a torch.Tensor")
    if logits.device.type != "cuda":
        raise ValueError("logits must be on a CUDA device")
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    if logits.dim() != 2:
        raise ValueError("logits must be 2-D [batch, num_classes]")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    batch, num_classes = logits.shape
    if out is None:
        out = torch.empty(logits.shape, dtype=torch.float32,
                          device=logits.device)
    elif (out.shape != logits.shape or out.dtype != torch.float32
          or out.device != logits.device or not out.is_contiguous()):
        raise ValueError("out must be a contiguous float32 tensor shaped like "
                         "logits on the same device")
    t_ptr = None
    if return_t or t_out is not None:
        if t_out is None:
            t_out = torch.empty(batch, dtype=torch.float32,
                                device=logits.device)
        elif (t_out.shape != (batch,) or t_out.dtype != torch.float32
              or t_out.device != logits.device or not t_out.is_contiguous()):
            raise ValueError("t_out must be a contiguous float32 [batch] "
                             "tensor on the logits' device")
        t_ptr = t_out.data_ptr()
    e_ptr = None
    if evals_out is not None:
        if (not isinstance(evals_out, torch.Tensor)
                or evals_out.shape != (batch,)
                or evals_out.dtype != torch.int32
                or evals_out.device != logits.device
                or not evals_out.is_contiguous()):
            raise ValueError("evals_out must be a contiguous int32 [batch] "
                             "tensor on the logits' device")
        e_ptr = evals_out.data_ptr()
    entry = (cs_constrained_softmax_bf16_ex
             if logits.dtype == torch.bfloat16 else cs_constrained_softmax_ex)
    with _on_device(logits.device):
        st = entry(
            logits.data_ptr(), out.data_ptr(), batch, num_classes,
            float(entropy_bound), float(t_min), float(t_max), int(max_iter),
            t_ptr, options(VARIANTS[variant], param, threads, int(strict),
                           e_ptr),
            _stream_handle(logits.device))
    if st != 0:
        raise CsError(st, "cs_constrained_softmax")
    return (out, t_out) if return_t else out


def _check_like(name, x, ref) -> None:
    import torch
    if (not isinstance(x, torch.Tensor) or x.shape != ref.shape
            or x.dtype != torch.float32 or x.device != ref.device
            or not x.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous float32 tensor shaped "
                         "like probs on the same device")


def constrained_softmax_backward(probs, grad_output, t, out=None,
                                 variant: str = "auto", param: int = 0,
                                 threads: int = 0):
    """Gradient with respect to the logits: (1/T) p (g - <g, p>) per row.

    ``probs`` and ``t`` are the forward's output and temperatures
    (``constrained_softmax(..., return_t=True)``), ``grad_output`` the
    upstream gradient; all on one CUDA device, fp32, contiguous.  Rows whose
    T is NaN (rows the forward zeroed) get zeros.  ``out`` may be given, and
    may be ``probs`` or ``grad_output`` itself (in place).  Asynchronous on
    the current stream.
    """
    import torch
    if not isinstance(probs, torch.Tensor) or probs.device.type != "cuda":
        raise ValueError("probs must be a CUDA tensor")
    if probs.dim() != 2:
        raise ValueError("probs must be 2-D [batch, num_classes]")
    _check_like("probs", probs, probs)
    _check_like("grad_output", grad_output, probs)
    batch, num_classes = probs.shape
    if (not isinstance(t, torch.Tensor) or t.shape != (batch,)
            or t.dtype != torch.float32 or t.device != probs.device
            or not t.is_contiguous()):
        raise ValueError("t must be a contiguous float32 [batch] tensor on "
                         "probs' device")
    if out is None:
        out = torch.empty_like(probs)
    else:
        _check_like("out", out, probs)
    with _on_device(probs.device):
        st = cs_constrained_softmax_backward_ex(
            probs.data_ptr(), grad_output.data_ptr(), t.data_ptr(),
            out.data_ptr(), batch, num_classes,
            options(VARIANTS[variant], param, threads, 0),
            _stream_handle(probs.device))
    if st != 0:
        raise CsError(st, "cs_constrained_softmax_backward")
    return out


def attention_softmax(scores, mask=None, causal: bool = False, out=None,
                      variant: str = "auto", param: int = 0,
                      threads: int = 0):
    """Section 2.6 attention_softmax of CUDA fp32 scores [B, H, S, S].

    ``mask`` is None or an additive fp32 mask of shape [B, S] or
    [B, 1, 1, S] (0 attends; -inf, or the page's -1e9, masks); ``causal``
    removes keys j > i from row i.  ``out`` may be given, ``scores`` itself
    included (in place).  Asynchronous on the current stream; rows with
    NaN/Inf inputs are zeroed and reported by :func:`get_error`.
    """
    import torch
    if not isinstance(scores, torch.Tensor) or scores.device.type != "cuda":
        raise ValueError("scores must be a CUDA tensor")
    if (scores.dtype != torch.float32 or scores.dim() != 4
            or scores.shape[2] != scores.shape[3] or not scores.is_contiguous()):
        raise ValueError("scores must be a contiguous float32 [B, H, S, S] "
                         "tensor")
    B, H, S, _ = scores.shape
    m_ptr = None
    if mask is not None:
        if (not isinstance(mask, torch.Tensor) or mask.dtype != torch.float32
                or mask.device != scores.device or not mask.is_contiguous()
                or mask.numel() != B * S
                or tuple(mask.shape) not in ((B, S), (B, 1, 1, S))):
            raise ValueError("mask must be a contiguous float32 [B, S] or "
                             "[B, 1, 1, S] tensor on the scores' device")
        m_ptr = mask.data_ptr()
    if out is None:
        out = torch.empty_like(scores)
    elif (out.shape != scores.shape or out.dtype != torch.float32
          or out.device != scores.device or not out.is_contiguous()):
        raise ValueError("out must be a contiguous float32 tensor shaped like "
                         "scores on the same device")
    with _on_device(scores.device):
        st = cs_attention_softmax_ex(
            scores.data_ptr(), out.data_ptr(), m_ptr, B, H, S,
            int(bool(causal)), options(VARIANTS[variant], param, threads, 0),
            _stream_handle(scores.device))
    if st != 0:
        raise CsError(st, "cs_attention_softmax")
    return out


def biencoder_attention(query, keys, values, scale=None,
                        entropy_bound: float = DEFAULT_ENTROPY_BOUND,
                        t_min: float = DEFAULT_T_MIN,
                        t_max: float = DEFAULT_T_MAX,
                        max_iter: int = DEFAULT_MAX_ITER, out=None,
                        return_attn: bool = False, return_t: bool = False,
                        lanes: int = 0, fused: bool = False):
    """Section 2.5 biencoder_attention: scores = query @ keys^T * scale
    (default 1/sqrt(d_head)), the constrained softmax of every score row,
    then attn @ values (on the tensor cores for d_head <= 64 and
    context_len <= d_head unless ``fused``, which runs all three steps in
    one kernel on the FMA pipes).  query [B, H, Q, D], keys and values
    [B, H, K, D], CUDA fp32 contiguous.  Returns the output [B, H, Q, D]
    (and the weights [B, H, Q, K] and temperatures [B, H, Q] when asked).
    Asynchronous on the current stream."""
    import math
    import torch
    for name, x in (("query", query), ("keys", keys), ("values", values)):
        if (not isinstance(x, torch.Tensor) or x.device.type != "cuda"
                or x.dtype != torch.float32 or x.dim() != 4
                or not x.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA float32 "
                             "4-D tensor")
    B, H, Q, D = query.shape
    K = keys.shape[2]
    if keys.shape != (B, H, K, D) or values.shape != (B, H, K, D):
        raise ValueError("keys and values must be [B, H, K, D]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(query)
    attn = t = None
    if return_attn:
        attn = torch.empty((B, H, Q, K), dtype=torch.float32,
                           device=query.device)
    if return_t:
        t = torch.empty((B, H, Q), dtype=torch.float32, device=query.device)
    variant = (CONSTANTS["CS_VARIANT_FUSED"] if fused
               else VARIANTS["rowgroup"] if lanes else 0)
    opt = options(variant, lanes, 0, 0)
    with _on_device(query.device):
        st = cs_biencoder_attention_ex(
            query.data_ptr(), keys.data_ptr(), values.data_ptr(),
            out.data_ptr(), B, Q, K, D, H, float(scale), float(entropy_bound),
            float(t_min), float(t_max), int(max_iter),
            attn.data_ptr() if attn is not None else None,
            t.data_ptr() if t is not None else None, opt,
            _stream_handle(query.device))
    if st != 0:
        raise CsError(st, "cs_biencoder_attention")
    res = (out,) + ((attn,) if return_attn else ()) + ((t,) if return_t else ())
    return res if len(res) > 1 else out


def plan_attention(batch: int, heads: int, seq_len: int, aligned: bool = True,
                   variant: str = "auto", param: int = 0,
                   threads: int = 0) -> dict:
    """The attention_softmax launch plan on the current device."""
    st, p = cs_plan_attention_launch(batch, heads, seq_len, int(aligned),
                                     options(VARIANTS[variant], param,
                                             threads, 0))
    if st != 0:
        raise CsError(st, "cs_plan_attention_launch")
    return p.as_dict()


def _autograd_function():
    import torch

    class ConstrainedSoftmaxFunction(torch.autograd.Function):
        """Autograd wrapper of section 6.3: forward = constrained_softmax,
        backward = constrained_softmax_backward at the forward's
        temperatures.  ``apply(logits, entropy_bound, t_min, t_max,
        max_iter)``; only the logits receive a gradient."""

        @staticmethod
        def forward(ctx, logits, entropy_bound=DEFAULT_ENTROPY_BOUND,
                    t_min=DEFAULT_T_MIN, t_max=DEFAULT_T_MAX,
                    max_iter=DEFAULT_MAX_ITER):
            out, t = constrained_softmax(logits.contiguous(), entropy_bound,
                                         t_min, t_max, max_iter,
                                         return_t=True)
            ctx.save_for_backward(out, t)
            return out

        @staticmethod
        def backward(ctx, grad_output):
            out, t = ctx.saved_tensors
            grad = constrained_softmax_backward(out, grad_output.contiguous(),
                                                t)
            return grad, None, None, None, None

    return ConstrainedSoftmaxFunction


def __getattr__(name):
    # The autograd class needs torch; it is built on first use so that the
    # package imports without torch (the C ABI tests run without it).
    if name == "ConstrainedSoftmaxFunction":
        cls = _autograd_function()
        globals()[name] = cls
        return cls
    raise AttributeError(name)


def get_error(device=None) -> set[str]:
    """Synchronise the current stream, read and clear the device error word;
    returns the names of the conditions seen since the last call."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    with _on_device(dev):
        st, mask = cs_get_error(_stream_handle(dev))
    if st != 0:
        raise CsError(st, "cs_get_error")
    return {name for name, bit in ERROR_BITS.items() if mask & bit}


def plan(batch: int, num_classes: int, variant: str = "auto",
         param: int = 0, threads: int = 0, strict: bool = False) -> dict:
    """The launch plan for this shape on the current device."""
    st, p = cs_plan_launch(batch, num_classes,
                           options(VARIANTS[variant], param, threads,
                                   int(strict)))
    if st != 0:
        raise CsError(st, "cs_plan_launch")
    return p.as_dict()


def plan_backward(batch: int, num_classes: int, variant: str = "auto",
                  param: int = 0, threads: int = 0) -> dict:
    """The backward's launch plan for this shape on the current device."""
    st, p = cs_plan_backward_launch(batch, num_classes,
                                    options(VARIANTS[variant], param,
                                            threads, 0))
    if st != 0:
        raise CsError(st, "cs_plan_backward_launch")
    return p.as_dict()


def version() -> str:
    return cs_version()
