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


def test_shapes_are_checked_before_anything_else(bi):
    """The library builds its copies and stores from the sizes the binding passes; a tensor whose shape
    disagrees with them is refused by shape first (these are host tensors: the shape error comes before
    the device check)."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    A = torch.zeros(4, 128, dtype=bf)
    with pytest.raises(ValueError, match=r"W: expected shape \(\*, 128\)"):
        bi.gemm(A, torch.zeros(128, 64, dtype=bf))
    with pytest.raises(ValueError, match=r"out: expected shape \(4, 128\)"):
        bi.gemm(A, torch.zeros(128, 128, dtype=bf), out=torch.empty(3, 128, dtype=bf))
    with pytest.raises(ValueError, match=r"out: expected shape \(4, 64\)"):
        bi.gemm(A, torch.zeros(128, 128, dtype=bf), out=torch.empty(4, 128, dtype=bf), ep=bi.EP_SWIGLU)
    with pytest.raises(ValueError, match=r"residual: expected shape \(4, 128\)"):
        bi.gemm(A, torch.zeros(128, 128, dtype=bf), out=torch.empty(4, 128, dtype=bf),
                residual=torch.zeros(4, 256, dtype=bf), ep=bi.EP_RESIDUAL)
    with pytest.raises(ValueError, match=r"gamma: expected shape \(128,\)"):
        bi.rmsnorm(torch.zeros(2, 128, dtype=bf), torch.ones(64, dtype=bf))
    q = torch.zeros(3, 8, 64, dtype=bf)
    kc = torch.zeros(10, 2, 16, 64, dtype=bf)
    table = torch.zeros(3, 4, dtype=i32)
    sl = torch.ones(3, dtype=i32)
    with pytest.raises(ValueError, match=r"k_cache: expected shape \(\*, \*, 16, 64\)"):
        bi.decode_attention(q, torch.zeros(10, 2, 8, 64, dtype=bf), kc, table, sl, 16)
    with pytest.raises(ValueError, match=r"v_cache: expected shape \(10, 2, 16, 64\)"):
        bi.decode_attention(q, kc, torch.zeros(9, 2, 16, 64, dtype=bf), table, sl, 16)
    with pytest.raises(ValueError, match=r"page_table: expected shape \(3, \*\)"):
        bi.decode_attention(q, kc, kc, table[:2], sl, 16)
    with pytest.raises(ValueError, match=r"seq_lens: expected shape \(3,\)"):
        bi.decode_attention_noalloc(q, kc, kc, table, sl[:2], 16)
    with pytest.raises(ValueError, match=r"out: expected shape \(3, 8, 64\)"):
        bi.decode_attention(q, kc, kc, table, sl, 16, out=torch.empty(3, 8, 32, dtype=bf))
    cu = torch.tensor([0, 3], dtype=i32)
    with pytest.raises(ValueError, match=r"q_pos0: expected shape \(1,\)"):
        bi.prefill_attention(q, cu, torch.zeros(2, dtype=i32), kc, kc, table[:1])
    with pytest.raises(ValueError, match=r"page_table: expected shape \(1, \*\)"):
        bi.prefill_attention(q, cu, torch.zeros(1, dtype=i32), kc, kc, table)
    with pytest.raises(ValueError, match=r"out: expected shape \(2,\)"):
        bi.argmax(torch.zeros(2, 10, dtype=f32), out=torch.empty(3, dtype=i32))
    with pytest.raises(ValueError, match=r"temperatures: expected shape \(2,\)"):
        bi.sample(torch.zeros(2, 10, dtype=f32), torch.zeros(2, dtype=i32), torch.zeros(2, dtype=i32),
                  torch.ones(3, dtype=f32))
    with pytest.raises(ValueError, match=r"out: expected shape \(5, 16\)"):
        bi.embed(torch.zeros(10, 16, dtype=bf), torch.zeros(5, dtype=i32), out=torch.empty(5, 8, dtype=bf))
