"""Host-side checks of the PyTorch operator (no GPU): registration, schema,
shape propagation through the fake implementation, mask marshalling, and the
aten override's dispatch entry and refusals."""
import pytest
import torch

from sdpa_forward_materialised_gb300 import torch_op as T

KEY = "aten::_scaled_dot_product_attention_math"


def test_schema():
    s = str(torch.ops.sdpa_gb300.sdpa_math.default._schema)
    assert s.startswith("sdpa_gb300::sdpa_math(Tensor q, Tensor k, Tensor v, Tensor? attn_mask, bool is_causal")
    assert s.endswith("-> (Tensor, Tensor)")


@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
def test_fake_shapes_gqa_and_distinct_value_dim(dt):
    q = torch.empty(2, 8, 5, 64, device="meta", dtype=dt)
    k = torch.empty(2, 2, 9, 64, device="meta", dtype=dt)
    v = torch.empty(2, 2, 9, 48, device="meta", dtype=dt)
    O, P = torch.ops.sdpa_gb300.sdpa_math(q, k, v, None, False, None)
    assert O.shape == (2, 8, 5, 48) and P.shape == (2, 8, 5, 9)
    assert O.dtype == dt and P.dtype == dt


def test_prepare_mask_broadcasts_to_library_shape():
    B, Hq, Sq, Skv = 2, 4, 3, 5
    m2 = torch.rand(Sq, Skv) < 0.5
    out = T._prepare_mask(m2, B, Hq, Sq, Skv, torch.float16)
    assert out.shape == (1, 1, Sq, Skv) and out.stride(-1) == 1 and torch.equal(out[0, 0], m2)
    pad = torch.rand(B, 1, 1, Skv) < 0.5  # a key-padding mask broadcast over the queries
    out = T._prepare_mask(pad, B, Hq, Sq, Skv, torch.float16)
    assert out.shape == (B, 1, Sq, Skv) and out.stride(2) != 0
    assert torch.equal(out, pad.expand(B, 1, Sq, Skv))
    add = torch.randn(1, Hq, Sq, Skv, dtype=torch.float64)
    out = T._prepare_mask(add, B, Hq, Sq, Skv, torch.float16)
    assert out.dtype == torch.float32 and out.shape == (1, Hq, Sq, Skv)
    assert T._prepare_mask(None, B, Hq, Sq, Skv, torch.float16) is None


def test_override_refuses_dropout_and_bad_heads():
    q = torch.zeros(1, 4, 2, 8)
    k = torch.zeros(1, 3, 2, 8)
    with pytest.raises(NotImplementedError, match="dropout"):
        T._aten_math_override(q, q, q, dropout_p=0.1)
    with pytest.raises(NotImplementedError, match="dropout"):
        T._aten_math_override(q, q, q, dropout_mask=torch.ones(1))
    with pytest.raises(ValueError, match="enable_gqa"):
        T._aten_math_override(q, k, k, enable_gqa=True)
    k2 = torch.zeros(1, 2, 2, 8)
    with pytest.raises(ValueError, match="enable_gqa"):
        T._aten_math_override(q, k2, k2, enable_gqa=False)


def test_override_enable_disable_dispatch_entry():
    assert not T.aten_override_enabled()
    has = lambda key: torch._C._dispatch_has_kernel_for_dispatch_key(KEY, key)
    assert not has("AutogradCUDA") and not has("CUDA")
    T.enable_aten_override()
    try:
        T.enable_aten_override()  # idempotent
        # under autograd, and for calls that skip the autograd keys (inference mode)
        assert T.aten_override_enabled() and has("AutogradCUDA") and has("CUDA")
    finally:
        T.disable_aten_override()
    assert not T.aten_override_enabled() and not has("AutogradCUDA") and not has("CUDA")
    # CPU tensors never reach the override: the stock math path still runs there
    q = torch.randn(1, 2, 3, 4)
    o, p = torch.ops.aten._scaled_dot_product_attention_math(q, q, q)
    assert o.shape == (1, 2, 3, 4) and p.shape == (1, 2, 3, 3)
