"""The (O, P) forward as a PyTorch operator, with its backward.

FlagOS-OP PR #10 ("feat: add sdpa_math operator", overview and the A1 item)
registers the math backend's SDPA as a framework operator that returns
(out, attn_probs) and has a backward through both outputs.  This module does the
same for the GB300 kernels:

* ``torch.ops.sdpa_gb300.sdpa_math(q, k, v, attn_mask, is_causal, scale)``:
  a ``torch.library`` custom op on CUDA returning (O, P), with a fake (meta)
  implementation for shape propagation and an autograd formula that calls the
  library's backward (gradients of q, k, v through dout and dprobs, GQA
  gradients summed back to the key/value heads).  An attention mask is a
  constant: it gets no gradient.
* ``enable_aten_override()``: routes ``aten::_scaled_dot_product_attention_math``
  on CUDA (what ``F.scaled_dot_product_attention`` runs under the MATH backend)
  to that op, so existing PyTorch code uses these kernels unchanged.  Cases the
  operation does not define (dropout, a dropout mask, head counts that neither
  match nor form groups) raise instead of running anything else.

Everything here marshals arguments (mask broadcasting, innermost-stride
copies); the work runs in the library's kernels.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch
from torch import Tensor

from . import prepare_mask, sdpa_math_backward, sdpa_math_fwd_ex, _mask_kind

_NS = "sdpa_gb300"


def _inner_contig(t: Tensor) -> Tensor:
    return t if t.stride(-1) == 1 else t.contiguous()


def _prepare_mask(attn_mask: Optional[Tensor], B: int, Hq: int, Sq: int, Skv: int,
                  dtype: torch.dtype) -> Optional[Tensor]:
    """Broadcast a mask to [1|B, 1|Hq, Sq, Skv] (the shape the library takes)."""
    return prepare_mask(attn_mask, B, Hq, Sq, Skv, dtype)


def _default_scale(q: Tensor, scale: Optional[float]) -> float:
    if scale is not None:
        return float(scale)
    return 1.0 / math.sqrt(q.shape[-1]) if q.shape[-1] > 0 else 1.0


@torch.library.custom_op(f"{_NS}::sdpa_math", mutates_args=(), device_types="cuda")
def sdpa_math_op(q: Tensor, k: Tensor, v: Tensor, attn_mask: Optional[Tensor], is_causal: bool,
                 scale: Optional[float]) -> Tuple[Tensor, Tensor]:
    """(O, P) of the math-backend SDPA forward on CUDA tensors."""
    B, Hq, Sq, _ = q.shape
    Skv = k.shape[-2]
    q, k, v = _inner_contig(q), _inner_contig(k), _inner_contig(v)
    mask = _prepare_mask(attn_mask, B, Hq, Sq, Skv, q.dtype)
    O = q.new_empty((B, Hq, Sq, v.shape[-1]))
    P = q.new_empty((B, Hq, Sq, Skv))
    # the library launches on the current device: make it the tensors' device
    with torch.cuda.device(q.device):
        sdpa_math_fwd_ex(q, k, v, mask, _mask_kind(mask), is_causal, _default_scale(q, scale), O, P, None,
                         "auto", torch.cuda.current_stream(q.device))
    return O, P


@sdpa_math_op.register_fake
def _(q, k, v, attn_mask, is_causal, scale):
    B, Hq, Sq, _ = q.shape
    return q.new_empty((B, Hq, Sq, v.shape[-1])), q.new_empty((B, Hq, Sq, k.shape[-2]))


def _setup_context(ctx, inputs, output):
    q, k, v, _, _, scale = inputs
    _, P = output
    ctx.save_for_backward(q, k, v, P)
    ctx.scale = _default_scale(q, scale)


def _backward(ctx, dO, dP):
    q, k, v, P = ctx.saved_tensors
    if dO is None:
        dO = torch.zeros(q.shape[:3] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    q, k, v, P = (_inner_contig(t) for t in (q, k, v, P))
    dO = _inner_contig(dO.to(q.dtype))
    if dP is not None:
        dP = _inner_contig(dP.to(q.dtype))
    with torch.cuda.device(q.device):
        dq, dk, dv = sdpa_math_backward(q, k, v, P, dO, dP, scale=ctx.scale,
                                        stream=torch.cuda.current_stream(q.device))
    return dq, dk, dv, None, None, None


sdpa_math_op.register_autograd(_backward, setup_context=_setup_context)


def _aten_math_override(query, key, value, attn_mask=None, dropout_p=0.0, is_causal=False, dropout_mask=None, *,
                        scale=None, enable_gqa=False):
    """The CUDA kernel behind ``aten::_scaled_dot_product_attention_math``:
    same arguments and (out, attn_probs) result, computed by the custom op."""
    if dropout_p != 0.0 or dropout_mask is not None:
        raise NotImplementedError("sdpa_gb300: dropout is not part of the materialised (O, P) forward")
    if query.dim() != 4 or key.dim() != 4 or value.dim() != 4:
        raise NotImplementedError("sdpa_gb300: q, k and v must be [B, H, S, D]")
    Hq, Hkv = query.shape[1], key.shape[1]
    if Hq != Hkv and not (enable_gqa and Hq % Hkv == 0) and Hkv != 1:
        raise ValueError(f"sdpa_gb300: {Hq} query heads and {Hkv} key/value heads need enable_gqa and "
                         f"Hq % Hkv == 0")
    return torch.ops.sdpa_gb300.sdpa_math(query, key, value, attn_mask, bool(is_causal), scale)


_override_lib: Optional[torch.library.Library] = None


def enable_aten_override() -> None:
    """Run ``aten::_scaled_dot_product_attention_math`` on CUDA tensors through
    the custom op (forward and backward).  Registered for AutogradCUDA (calls
    under autograd) and for CUDA (calls that skip the autograd keys, e.g. under
    ``torch.inference_mode()``).  Idempotent."""
    global _override_lib
    if _override_lib is not None:
        return
    lib = torch.library.Library("aten", "IMPL")
    lib.impl("_scaled_dot_product_attention_math", _aten_math_override, "AutogradCUDA")
    lib.impl("_scaled_dot_product_attention_math", _aten_math_override, "CUDA")
    _override_lib = lib


def disable_aten_override() -> None:
    """Give ``aten::_scaled_dot_product_attention_math`` back to PyTorch."""
    global _override_lib
    if _override_lib is not None:
        _override_lib._destroy()
        _override_lib = None


def aten_override_enabled() -> bool:
    return _override_lib is not None
