"""bi_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory where they run it.  Its split partials live in the
library's static 16 MiB device array instead of a caller workspace; it must
give exactly what bi_decode_attention gives, call after call, and turn away
batches that need more scratch than the array holds.

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

from invariant_fixed_order_gb300 import synth
from tests.helpers import PagedKV, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from invariant_fixed_order_gb300 import bi as _bi
    return _bi


def decode_case(seq_lens, H, Hkv, Dh, seed):
    B = len(seq_lens)
    max_pages = max((s + 15) // 16 for s in seq_lens) + 1
    kv = PagedKV(sum((s + 15) // 16 for s in seq_lens) + 8, Hkv, Dh, max_pages, B, seed=seed)
    for i, s in enumerate(seq_lens):
        k, v = synth.kv_history(s, Hkv, Dh, seed * 1000 + i, device="cuda")
        kv.write(i, k, v)
    q = synth.normal_bf16((B, H, Dh), 1.0, seed + 7, "cuda")
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    return kv, q, sl


@pytest.mark.parametrize("H,Hkv,Dh,mode", [(32, 8, 128, 0), (32, 8, 128, 1), (4, 2, 64, 0)])
def test_noalloc_matches_workspace_call_on_two_calls_in_a_row(bi, H, Hkv, Dh, mode):
    seq_lens = [1, 17, 256, 300, 1500, 2049]
    kv, q, sl = decode_case(seq_lens, H, Hkv, Dh, seed=11)
    table = kv.table_tensor()
    st = bi.new_status()
    ref = bi.decode_attention(q, kv.k[0], kv.v[0], table, sl, max(seq_lens), out_dtype=bi.F32, mode=mode, status=st)
    bi.check_status(st)
    for _ in range(2):
        got = bi.decode_attention_noalloc(q, kv.k[0], kv.v[0], table, sl, max(seq_lens), out_dtype=bi.F32,
                                          mode=mode, status=st)
        bi.check_status(st)
        # same kernels, same partials: the bits must agree exactly (within any tolerance)
        assert np.array_equal(bits(got), bits(ref))
    # a different batch in between leaves other contents in the shared array;
    # both calls still match the workspace entry point exactly
    sub = dict(q=q[:2].contiguous(), table=table[:2].contiguous(), sl=sl[:2].contiguous(), m=max(seq_lens[:2]))
    other = bi.decode_attention_noalloc(sub["q"], kv.k[0], kv.v[0], sub["table"], sub["sl"], sub["m"],
                                        out_dtype=bi.F32, mode=mode)
    got = bi.decode_attention_noalloc(q, kv.k[0], kv.v[0], table, sl, max(seq_lens), out_dtype=bi.F32, mode=mode)
    ref_other = bi.decode_attention(sub["q"], kv.k[0], kv.v[0], sub["table"], sub["sl"], sub["m"],
                                    out_dtype=bi.F32, mode=mode)
    torch.cuda.synchronize()
    assert np.array_equal(bits(got), bits(ref))
    assert np.array_equal(bits(other), bits(ref_other))


def test_noalloc_rejects_batches_beyond_the_static_scratch(bi):
    H, Hkv, Dh = 32, 8, 128
    kv, q, sl = decode_case([40], H, Hkv, Dh, seed=12)
    # 64 requests at up to 8192 positions need 64 * 32 * 32 * 130 * 4 bytes > 16 MiB
    B = 64
    qb = q.expand(B, -1, -1).contiguous()
    table = torch.zeros(B, 8192 // 16, dtype=torch.int32, device="cuda")
    slb = torch.full((B,), 40, dtype=torch.int32, device="cuda")
    out = torch.full((B, H, Dh), 7.0, dtype=torch.float32, device="cuda")
    need = B * H * (8192 // 256) * (Dh + 2) * 4
    assert need > bi.NOALLOC_SCRATCH_BYTES
    with pytest.raises(bi.BIError) as e:
        bi.decode_attention_noalloc(qb, kv.k[0], kv.v[0], table, slb, 8192, out_dtype=bi.F32, out=out)
    assert e.value.status == bi.BI_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # rejected before any launch: nothing written
