"""Edge cases on the GPU: empty inputs are no-ops, a single-key context
returns its value row exactly, a step without logit rows leaves the residual
stream the same as a step with them, and degenerate logit rows."""
import numpy as np
import pytest
import torch

from invariant_fixed_order_gb300 import synth
from tests.test_gpu_kernels import make_decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from invariant_fixed_order_gb300 import bi as b
    return b


def test_empty_inputs_are_no_ops(bi):
    dev = "cuda"
    W = torch.randn(256, 128, device=dev).to(torch.bfloat16)
    assert bi.gemm(torch.empty(0, 128, dtype=torch.bfloat16, device=dev), W, c_dtype=bi.F32).shape == (0, 256)
    g = torch.ones(128, dtype=torch.bfloat16, device=dev)
    assert bi.rmsnorm(torch.empty(0, 128, dtype=torch.bfloat16, device=dev), g).shape == (0, 128)
    z = torch.empty(0, 1000, device=dev)
    assert bi.argmax(z).shape == (0,)
    assert bi.log_softmax(z).shape == (0, 1000)
    e = torch.empty(0, dtype=torch.int32, device=dev)
    assert bi.sample(z, e, e, torch.empty(0, device=dev)).shape == (0,)
    torch.cuda.synchronize()


def test_single_key_context_returns_its_value_exactly(bi):
    """Context length 1: the only weight is exp(0) = 1, so every head's output is its KV head's value row
    (the chunk's fold and the merge multiply by exactly 1)."""
    for H, Hkv, Dh in ((32, 8, 128), (4, 2, 64)):
        kv, hist, q = make_decode_case([1, 1, 1], H, Hkv, Dh, seed=21)
        sl = torch.ones(3, dtype=torch.int32, device="cuda")
        out = bi.decode_attention(q, kv.k[0], kv.v[0], kv.table_tensor(), sl, 1, out_dtype=bi.F32)
        for i in range(3):
            v = hist[i][1]  # [1, Hkv, Dh]
            for h in range(H):
                assert np.array_equal(out[i, h].cpu().numpy(), v[0, h // (H // Hkv)]), (H, i, h)


def test_step_without_logit_rows(bi):
    """A step with R = 0 (nothing needs logits, e.g. a prefill chunk that does not end its prompt) writes
    the same residual stream as the same step with logits."""
    from invariant_fixed_order_gb300.config import TINY
    from invariant_fixed_order_gb300.engine import Engine
    eng = Engine(TINY, num_pages=64, max_pages=16, max_T=128, max_B=4, max_R=128)
    ids = synth.token_ids(40, TINY.V, 77)
    t1 = np.zeros((1, 16), np.int32)
    t1[0, :3] = eng.pool.alloc(3)
    t2 = np.zeros((1, 16), np.int32)
    t2[0, :3] = eng.pool.alloc(3)
    _, _, h_with = eng.step([40], [0], ids, t1, list(range(40)), want_hidden=True)
    _, _, h_without = eng.step([40], [0], ids, t2, [], want_logits=False, want_hidden=True)
    assert torch.equal(h_with.view(torch.int16), h_without.view(torch.int16))
    eng.check()
    eng.close()


def _int_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-8, 9, shape, generator=g).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("M,N,K,skip", [(1, 128, 64, 0), (300, 4096, 4096, 5), (64, 131072, 256, 3)])
def test_gemm_bounded_wait_runs_out_and_the_stream_recovers(bi, M, N, K, skip):
    """Failure detection of the GEMM without a fault: one ring stage's copies are withheld (in every CTA of a
    pair), so the MMA issuer's bounded wait runs out after 1 ms; the kernel reports a timeout through the
    status word, drains what is in flight, frees tensor memory and returns.  The next ordinary GEMM on the
    same stream is integer-exact.  (The CTA-pair form for N <= 65536, the single-CTA form above.)"""
    A, W = _int_bf16((M, K), 1 + M), _int_bf16((N, K), 2 + N)
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    st = bi.new_status()
    bi.gemm_wait_test(A, W, out, st, wait_limit_ns=1_000_000, skip_stage=skip)
    with pytest.raises(bi.BIError) as e:
        bi.check_status(st)
    assert e.value.status == bi.BI_ERR_TIMEOUT
    bi.reset_status(st)
    A2, W2 = _int_bf16((37, 256), 3), _int_bf16((384, 256), 4)
    C = bi.gemm(A2, W2, c_dtype=bi.F32, status=st)
    bi.check_status(st)
    ref = A2.double() @ W2.double().T  # |sums| < 2^24: exact in fp32 in any order
    assert torch.equal(C.double(), ref)
