"""The Python binding refuses tensors the C ABI would misread (host memory, a
missing required operand) before anything reaches the library; no GPU needed."""
import pytest
import torch


@pytest.fixture(scope="module")
def bi():
    from invariant_fixed_order_gb300 import build
    build.build()
    from invariant_fixed_order_gb300 import bi as b
    return b


def test_host_tensors_are_refused(bi):
    A = torch.zeros(4, 128, dtype=torch.bfloat16)
    W = torch.zeros(128, 128, dtype=torch.bfloat16)
    out = torch.empty(4, 128, dtype=torch.float32)
    with pytest.raises(ValueError, match="A: expected a CUDA tensor"):
        bi.gemm(A, W, out=out, c_dtype=bi.F32)
    with pytest.raises(ValueError, match="x: expected a CUDA tensor"):
        bi.rmsnorm(torch.zeros(2, 128, dtype=torch.bfloat16), torch.ones(128, dtype=torch.bfloat16),
                   out=torch.empty(2, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="logits: expected a CUDA tensor"):
        bi.argmax(torch.zeros(2, 10), out=torch.empty(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="status: expected a CUDA tensor"):
        bi.check_status(torch.zeros(1, dtype=torch.int32))


def test_missing_required_tensor_is_refused(bi):
    with pytest.raises(ValueError, match="status: a CUDA tensor is required"):
        bi.check_status(None)


def test_validation_helper_checks_layout_and_dtype(bi):
    # the helper's own rules, on host tensors standing in for device ones
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        bi._d(torch.zeros(4, 4).t(), "t")
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        bi._d("not a tensor", "t")
    assert bi._d(None, "t", optional=True) is None
