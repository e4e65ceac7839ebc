"""ctypes binding of libcsoftmax.so: one Python function per C ABI entry
point, with the same name and arguments (pointers as integers, streams as
integers).  Argument marshalling only: every step of the operation runs in
the library's CUDA kernels.  Loading fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libcsoftmax.so")
HEADER = os.path.join(os.path.dirname(PKG), "include",
                      "entropy_bounded_softmax.h")

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class cs_options(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int32),
        ("param", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("strict", ctypes.c_int32),
        ("evals_out", ctypes.c_void_p),
    ]


class cs_plan(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int32),
        ("lanes_per_row", ctypes.c_int32),
        ("elems_per_lane", ctypes.c_int32),
        ("cluster_size", ctypes.c_int32),
        ("slice_len", ctypes.c_int32),
        ("threads_per_cta", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("grid_ctas", ctypes.c_int64),
        ("staged_tensors", ctypes.c_int32),
        ("tensor_cores", ctypes.c_int32),
        ("fan_points", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def _header_constants() -> dict[str, int]:
    """The #define'd integer constants of the public header."""
    out = {}
    with open(HEADER) as f:
        for line in f:
            m = re.match(r"#define\s+(CS_[A-Z0-9_]+)\s+(-?\d+)", line)
            if m:
                out[m.group(1)] = int(m.group(2))
    return out


CONSTANTS = _header_constants()
globals().update(CONSTANTS)

_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float

_SIGNATURES = {
    "cs_constrained_softmax": (_I32, [_VP, _VP, _I64, _I32, _F32, _F32, _F32,
                                      _I32, _VP, _VP]),
    "cs_constrained_softmax_ex": (_I32, [_VP, _VP, _I64, _I32, _F32, _F32,
                                         _F32, _I32, _VP,
                                         ctypes.POINTER(cs_options), _VP]),
    "cs_constrained_softmax_bf16": (_I32, [_VP, _VP, _I64, _I32, _F32, _F32,
                                           _F32, _I32, _VP, _VP]),
    "cs_constrained_softmax_bf16_ex": (_I32, [_VP, _VP, _I64, _I32, _F32,
                                              _F32, _F32, _I32, _VP,
                                              ctypes.POINTER(cs_options),
                                              _VP]),
    "cs_check_args_bf16": (_I32, [_VP, _VP, _I64, _I32, _F32, _F32, _F32,
                                  _I32, _VP]),
    "cs_get_error": (_I32, [ctypes.POINTER(_I32), _VP]),
    "cs_plan_launch": (_I32, [_I64, _I32, ctypes.POINTER(cs_options),
                              ctypes.POINTER(cs_plan)]),
    "cs_plan_host": (_I32, [_I64, _I32, ctypes.POINTER(cs_options), _I32,
                            _I32, _I32, _I32, ctypes.POINTER(cs_plan)]),
    "cs_check_args": (_I32, [_VP, _VP, _I64, _I32, _F32, _F32, _F32, _I32,
                             _VP]),
    "cs_constrained_softmax_backward": (_I32, [_VP, _VP, _VP, _VP, _I64,
                                               _I32, _VP]),
    "cs_constrained_softmax_backward_ex": (_I32, [_VP, _VP, _VP, _VP, _I64,
                                                  _I32,
                                                  ctypes.POINTER(cs_options),
                                                  _VP]),
    "cs_plan_backward_launch": (_I32, [_I64, _I32, ctypes.POINTER(cs_options),
                                       ctypes.POINTER(cs_plan)]),
    "cs_plan_backward_host": (_I32, [_I64, _I32, ctypes.POINTER(cs_options),
                                     _I32, _I32, _I32, _I32,
                                     ctypes.POINTER(cs_plan)]),
    "cs_check_backward_args": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32]),
    "cs_attention_softmax": (_I32, [_VP, _VP, _VP, _I32, _I32, _I32, _I32,
                                    _VP]),
    "cs_attention_softmax_ex": (_I32, [_VP, _VP, _VP, _I32, _I32, _I32, _I32,
                                       ctypes.POINTER(cs_options), _VP]),
    "cs_plan_attention_launch": (_I32, [_I32, _I32, _I32, _I32,
                                        ctypes.POINTER(cs_options),
                                        ctypes.POINTER(cs_plan)]),
    "cs_plan_attention_host": (_I32, [_I32, _I32, _I32, _I32,
                                      ctypes.POINTER(cs_options), _I32, _I32,
                                      _I32, ctypes.POINTER(cs_plan)]),
    "cs_check_attention_args": (_I32, [_VP, _VP, _VP, _I32, _I32, _I32,
                                       _I32]),
    "cs_biencoder_attention": (_I32, [_VP, _VP, _VP, _VP, _I32, _I32, _I32,
                                      _I32, _I32, _F32, _F32, _VP]),
    "cs_biencoder_attention_ex": (_I32, [_VP, _VP, _VP, _VP, _I32, _I32,
                                         _I32, _I32, _I32, _F32, _F32, _F32,
                                         _F32, _I32, _VP, _VP,
                                         ctypes.POINTER(cs_options), _VP]),
    "cs_plan_biencoder_host": (_I32, [_I32, _I32, _I32, _I32, _I32,
                                      ctypes.POINTER(cs_options), _I32,
                                      ctypes.POINTER(cs_plan)]),
    "cs_check_biencoder_args": (_I32, [_VP, _VP, _VP, _VP, _I32, _I32, _I32,
                                       _I32, _I32, _F32, _F32, _F32, _F32,
                                       _I32, _VP, _VP]),
    "cs_probe_ex2": (_I32, [_VP, _I32, ctypes.POINTER(_I64), _VP]),
    "cs_probe_ex2_sink_floats": (_I32, []),
    "cs_test_wait_timeout": (_I32, [_I64, _VP]),
    "cs_version": (ctypes.c_char_p, []),
    "cs_status_string": (ctypes.c_char_p, [_I32]),
}


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libcsoftmax.so (built by ``build.py``); raise if it is absent."""
    global _lib
    if _lib is not None and path is None:   # the common case: no lock
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIBRARY
        if not os.path.exists(p):
            raise RuntimeError(
                f"libcsoftmax.so not found at {p}: build it first "
                "(python -m entropy_bounded_softmax_gb300.build); there is no "
                "fallback implementation")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def exported_names() -> list[str]:
    return list(_SIGNATURES)


# Same-named thin wrappers over the C entry points.
def cs_constrained_softmax(logits, out, batch, num_classes, entropy_bound,
                           t_min, t_max, max_iter, t_out, stream) -> int:
    return load().cs_constrained_softmax(logits, out, batch, num_classes,
                                         entropy_bound, t_min, t_max,
                                         max_iter, t_out, stream)


def options(variant=0, param=0, threads=0, strict=0, evals_out=None):
    """A cs_options struct (all zero = automatic); evals_out: an optional
    device pointer (integer) for the per-row evaluation counts."""
    return cs_options(int(variant), int(param), int(threads), int(strict),
                      evals_out)


def _opt_ref(opt):
    return None if opt is None else ctypes.byref(opt)


def cs_constrained_softmax_ex(logits, out, batch, num_classes, entropy_bound,
                              t_min, t_max, max_iter, t_out, opt,
                              stream) -> int:
    return load().cs_constrained_softmax_ex(
        logits, out, batch, num_classes, entropy_bound, t_min, t_max,
        max_iter, t_out, _opt_ref(opt), stream)


def cs_constrained_softmax_bf16(logits, out, batch, num_classes,
                                entropy_bound, t_min, t_max, max_iter, t_out,
                                stream) -> int:
    return load().cs_constrained_softmax_bf16(logits, out, batch, num_classes,
                                              entropy_bound, t_min, t_max,
                                              max_iter, t_out, stream)


def cs_constrained_softmax_bf16_ex(logits, out, batch, num_classes,
                                   entropy_bound, t_min, t_max, max_iter,
                                   t_out, opt, stream) -> int:
    return load().cs_constrained_softmax_bf16_ex(
        logits, out, batch, num_classes, entropy_bound, t_min, t_max,
        max_iter, t_out, _opt_ref(opt), stream)


def cs_check_args_bf16(logits, out, batch, num_classes, entropy_bound, t_min,
                       t_max, max_iter, t_out) -> int:
    return load().cs_check_args_bf16(logits, out, batch, num_classes,
                                     entropy_bound, t_min, t_max, max_iter,
                                     t_out)


def cs_get_error(stream) -> tuple[int, int]:
    mask = _I32(0)
    st = load().cs_get_error(ctypes.byref(mask), stream)
    return st, mask.value


def cs_plan_launch(batch, num_classes, opt=None):
    p = cs_plan()
    st = load().cs_plan_launch(batch, num_classes, _opt_ref(opt),
                               ctypes.byref(p))
    return st, p


def cs_plan_host(batch, num_classes, opt, sm_count, smem_per_block_optin,
                 smem_per_sm, max_cluster):
    p = cs_plan()
    st = load().cs_plan_host(batch, num_classes, _opt_ref(opt), sm_count,
                             smem_per_block_optin, smem_per_sm, max_cluster,
                             ctypes.byref(p))
    return st, p


def cs_check_args(logits, out, batch, num_classes, entropy_bound, t_min,
                  t_max, max_iter, t_out) -> int:
    return load().cs_check_args(logits, out, batch, num_classes,
                                entropy_bound, t_min, t_max, max_iter, t_out)


def cs_constrained_softmax_backward(probs, grad_out, t, grad_in, batch,
                                    num_classes, stream) -> int:
    return load().cs_constrained_softmax_backward(probs, grad_out, t, grad_in,
                                                  batch, num_classes, stream)


def cs_constrained_softmax_backward_ex(probs, grad_out, t, grad_in, batch,
                                       num_classes, opt, stream) -> int:
    return load().cs_constrained_softmax_backward_ex(
        probs, grad_out, t, grad_in, batch, num_classes, _opt_ref(opt), stream)


def cs_plan_backward_launch(batch, num_classes, opt=None):
    p = cs_plan()
    st = load().cs_plan_backward_launch(batch, num_classes, _opt_ref(opt),
                                        ctypes.byref(p))
    return st, p


def cs_plan_backward_host(batch, num_classes, opt, sm_count,
                          smem_per_block_optin, smem_per_sm, max_cluster):
    p = cs_plan()
    st = load().cs_plan_backward_host(batch, num_classes, _opt_ref(opt),
                                      sm_count, smem_per_block_optin,
                                      smem_per_sm, max_cluster,
                                      ctypes.byref(p))
    return st, p


def cs_check_backward_args(probs, grad_out, t, grad_in, batch,
                           num_classes) -> int:
    return load().cs_check_backward_args(probs, grad_out, t, grad_in, batch,
                                         num_classes)


def cs_attention_softmax(scores, out, mask, batch, heads, seq_len, causal,
                         stream) -> int:
    return load().cs_attention_softmax(scores, out, mask, batch, heads,
                                       seq_len, causal, stream)


def cs_attention_softmax_ex(scores, out, mask, batch, heads, seq_len, causal,
                            opt, stream) -> int:
    return load().cs_attention_softmax_ex(scores, out, mask, batch, heads,
                                          seq_len, causal, _opt_ref(opt),
                                          stream)


def cs_plan_attention_launch(batch, heads, seq_len, aligned, opt=None):
    p = cs_plan()
    st = load().cs_plan_attention_launch(batch, heads, seq_len, aligned,
                                         _opt_ref(opt), ctypes.byref(p))
    return st, p


def cs_plan_attention_host(batch, heads, seq_len, aligned, opt, sm_count,
                           smem_per_block_optin, smem_per_sm):
    p = cs_plan()
    st = load().cs_plan_attention_host(batch, heads, seq_len, aligned,
                                       _opt_ref(opt), sm_count,
                                       smem_per_block_optin, smem_per_sm,
                                       ctypes.byref(p))
    return st, p


def cs_check_attention_args(scores, out, mask, batch, heads, seq_len,
                            causal) -> int:
    return load().cs_check_attention_args(scores, out, mask, batch, heads,
                                          seq_len, causal)


def cs_biencoder_attention(query, keys, values, output, batch_size,
                           query_len, context_len, d_head, num_heads, scale,
                           entropy_bound, stream) -> int:
    return load().cs_biencoder_attention(query, keys, values, output,
                                         batch_size, query_len, context_len,
                                         d_head, num_heads, scale,
                                         entropy_bound, stream)


def cs_biencoder_attention_ex(query, keys, values, output, batch_size,
                              query_len, context_len, d_head, num_heads,
                              scale, entropy_bound, t_min, t_max, max_iter,
                              attn_out, t_out, opt, stream) -> int:
    return load().cs_biencoder_attention_ex(
        query, keys, values, output, batch_size, query_len, context_len,
        d_head, num_heads, scale, entropy_bound, t_min, t_max, max_iter,
        attn_out, t_out, _opt_ref(opt), stream)


def cs_plan_biencoder_host(batch_size, query_len, context_len, d_head,
                           num_heads, opt, smem_per_block_optin):
    p = cs_plan()
    st = load().cs_plan_biencoder_host(batch_size, query_len, context_len,
                                       d_head, num_heads, _opt_ref(opt),
                                       smem_per_block_optin, ctypes.byref(p))
    return st, p


def cs_check_biencoder_args(query, keys, values, output, batch_size,
                            query_len, context_len, d_head, num_heads, scale,
                            entropy_bound, t_min, t_max, max_iter, attn_out,
                            t_out) -> int:
    return load().cs_check_biencoder_args(
        query, keys, values, output, batch_size, query_len, context_len,
        d_head, num_heads, scale, entropy_bound, t_min, t_max, max_iter,
        attn_out, t_out)


def cs_probe_ex2(sink, iters, stream) -> tuple[int, int]:
    count = _I64(0)
    st = load().cs_probe_ex2(sink, iters, ctypes.byref(count), stream)
    return st, count.value


def cs_probe_ex2_sink_floats() -> int:
    return load().cs_probe_ex2_sink_floats()


def cs_test_wait_timeout(limit_ns, stream) -> int:
    return load().cs_test_wait_timeout(limit_ns, stream)


def cs_version() -> str:
    return load().cs_version().decode()


def cs_status_string(status: int) -> str:
    return load().cs_status_string(status).decode()
