"""Per-kernel parity (CUDA path vs the CPU oracle, through the C ABI) and
per-kernel batch invariance (a row's bits do not depend on the other rows)."""
import numpy as np
import pytest
import torch

import oracle
from invariant_fixed_order_gb300 import synth
from tests.helpers import ATTN_MAX_ABS, PagedKV, bits, f32, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from invariant_fixed_order_gb300 import bi as _bi
    return _bi


def rand_bf16(shape, std, seed, device="cuda", mean=0.0):
    return synth.normal_bf16(shape, std, seed, device, mean=mean)


def int_bf16(shape, seed, lo=-8, hi=8, device="cuda"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16).to(device)


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,d", [(1, 256), (7, 4096), (64, 4096), (300, 256), (33, 8192)])
def test_rmsnorm_parity(bi, rows, d):
    x = rand_bf16((rows, d), 1.0, 1 + rows)
    g = rand_bf16((d,), 0.02, 2 + d, mean=1.0)
    y = bi.rmsnorm(x, g)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(f32(x), f32(g), 1e-5, round_bf16=True)
    got = f32(y)
    # equal up to one bf16 rounding flip where the fp32 values straddle a tie
    assert np.max(np.abs(got - ref) / (np.abs(ref) + 1e-30)) <= 2.0 ** -7
    assert np.mean(got == ref) > 0.99


def test_rmsnorm_row_invariance(bi):
    d = 4096
    x = rand_bf16((64, d), 1.0, 11)
    g = rand_bf16((d,), 0.02, 12, mean=1.0)
    full = bits(bi.rmsnorm(x, g))
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(3)).cuda()
    permuted = bits(bi.rmsnorm(x[perm].contiguous(), g))
    assert np.array_equal(permuted, full[perm.cpu().numpy()])
    for r in (0, 17, 63):
        assert np.array_equal(bits(bi.rmsnorm(x[r:r + 1].contiguous(), g))[0], full[r])


def test_rmsnorm_in_place(bi):
    x = rand_bf16((9, 256), 1.0, 13)
    g = rand_bf16((256,), 0.02, 14, mean=1.0)
    ref = bits(bi.rmsnorm(x, g))
    bi.rmsnorm(x, g, out=x)
    assert np.array_equal(bits(x), ref)


# ---------------------------------------------------------------------------
# GEMM (tcgen05)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (5, 128, 256), (128, 128, 4096), (129, 384, 1024),
                                   (300, 256, 14336), (64, 512, 4096), (17, 640, 1984), (600, 768, 512),
                                   (3, 25600, 128), (520, 8192, 128), (3, 65664, 128), (300, 65792, 64)])
def test_gemm_integer_valued_exact(bi, M, N, K):
    A = int_bf16((M, K), 100 + M)
    W = int_bf16((N, K), 200 + N)
    C = bi.gemm(A, W, c_dtype=bi.F32)
    torch.cuda.synchronize()
    ref = f32(A).astype(np.int64) @ f32(W).astype(np.int64).T
    assert np.array_equal(f32(C).astype(np.int64), ref)


@pytest.mark.parametrize("M,N,K", [(1, 6144, 4096), (33, 256, 1024), (200, 2048, 256)])
def test_gemm_parity_random(bi, M, N, K):
    A = rand_bf16((M, K), 1.0, 300 + M)
    W = rand_bf16((N, K), 0.02, 301 + N)
    C = bi.gemm(A, W, c_dtype=bi.F32)
    torch.cuda.synchronize()
    ref = oracle.matmul(f32(A), f32(W))
    assert rel_fro(f32(C), ref) < 1e-5
    assert np.max(np.abs(f32(C) - ref)) < 1e-4


def test_gemm_bf16_and_residual_epilogue(bi):
    M, N, K = 70, 256, 1024
    A = rand_bf16((M, K), 1.0, 400)
    W = rand_bf16((N, K), 0.02, 401)
    R = rand_bf16((M, N), 1.0, 402)
    C = bi.gemm(A, W, residual=R, ep=bi.EP_RESIDUAL)
    C32 = bi.gemm(A, W, c_dtype=bi.F32)
    torch.cuda.synchronize()
    # the epilogue is one fp32 add of the accumulator and the residual, rounded once
    expect = (C32 + R.float()).to(torch.bfloat16)
    assert np.array_equal(bits(C), bits(expect))
    ref = oracle.bf16_round(oracle.matmul(f32(A), f32(W)) + f32(R))
    assert np.mean(f32(C) == ref) > 0.98
    # every element within one bf16 rounding of the oracle's (|acc| < 2, so the two fp32 sums of 1024 products
    # differ by well under 3e-4 before the residual add and the rounding)
    assert np.all(np.abs(f32(C) - ref) <= 2.0 ** -7 * np.abs(ref) + 3e-4)
    # in place (output aliases the residual)
    Rc = R.clone()
    bi.gemm(A, W, out=Rc, residual=Rc, ep=bi.EP_RESIDUAL)
    assert np.array_equal(bits(Rc), bits(C))


@pytest.mark.parametrize("K", [4096, 14336])
def test_gemm_pair_and_single_forms_give_identical_bits(bi, K):
    """The CTA-pair MMA form (256x128x16 over two SMs) and the single-CTA form (128x128x16) give every
    element the same bits, at decode and prefill sizes: the same columns computed by a 4096-wide product
    (pair form) and by a 65792-wide one (single form).  This is what lets the form follow the tile count."""
    W = rand_bf16((65792, K), 0.02, 600 + K)
    for M in (1, 64, 300):
        A = rand_bf16((M, K), 1.0, 601 + M)
        pair = bi.gemm(A, W[:4096].contiguous(), c_dtype=bi.F32)
        single = bi.gemm(A, W, c_dtype=bi.F32)[:, :4096].contiguous()
        torch.cuda.synchronize()
        assert np.array_equal(bits(pair), bits(single)), (M, K)
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N,K", [(4096, 4096), (4096, 14336), (65792, 4096)])
def test_gemm_rows_at_every_m_match_a_300_row_product(bi, N, K):
    """How a product is laid out follows M (the A box height, the tile width, the ring), never the
    arithmetic of an element: every row at every M up to 128 has the bits of the same row in a 300-row
    product (256-wide tiles there), for fp32 output, the residual epilogue and the SwiGLU epilogue, in
    the pair form (N <= 65536) and the single-CTA form (above)."""
    A = rand_bf16((300, K), 1.0, 620 + K)
    W = rand_bf16((N, K), 0.02, 621 + N)
    R = rand_bf16((300, N), 1.0, 622)
    full = bits(bi.gemm(A, W, c_dtype=bi.F32))
    full_res = bits(bi.gemm(A, W, residual=R, ep=bi.EP_RESIDUAL))
    full_glu = bits(bi.gemm(A, W, ep=bi.EP_SWIGLU)) if N <= 8192 else None
    rng = np.random.default_rng(K + N)
    for M in (1, 2, 7, 16, 17, 33, 64, 65, 100, 128):
        rows = np.sort(rng.choice(300, size=M, replace=False))
        idx = torch.from_numpy(rows).cuda()
        sub = A[idx].contiguous()
        assert np.array_equal(bits(bi.gemm(sub, W, c_dtype=bi.F32)), full[rows]), (M, N, K)
        got = bits(bi.gemm(sub, W, residual=R[idx].contiguous(), ep=bi.EP_RESIDUAL))
        assert np.array_equal(got, full_res[rows]), (M, N, K)
        if full_glu is not None:
            assert np.array_equal(bits(bi.gemm(sub, W, ep=bi.EP_SWIGLU)), full_glu[rows]), (M, N, K)
    del A, W, R
    torch.cuda.empty_cache()


def test_gemm_swiglu_epilogue(bi):
    M, F, K = 40, 256, 512
    A = rand_bf16((M, K), 1.0, 500)
    Wg = rand_bf16((F, K), 0.05, 501)
    Wu = rand_bf16((F, K), 0.05, 502)
    Wgu = bi.pack_gate_up(Wg, Wu)
    H = bi.gemm(A, Wgu, ep=bi.EP_SWIGLU)
    torch.cuda.synchronize()
    g = oracle.matmul(f32(A), f32(Wg))
    u = oracle.matmul(f32(A), f32(Wu))
    ref = oracle.swiglu(g, u, round_bf16=True)
    got = f32(H)
    assert got.shape == (M, F)
    assert np.max(np.abs(got - ref) / (np.abs(ref) + 1e-3)) < 2.0 ** -6
    assert np.mean(got == ref) > 0.97


def test_gemm_row_invariance(bi):
    """A row's result does not depend on M, on its position in the tile, or on the other rows."""
    K, N = 4096, 256
    A = rand_bf16((300, K), 1.0, 600)
    W = rand_bf16((N, K), 0.02, 601)
    full = bits(bi.gemm(A, W, c_dtype=bi.F32))
    for rows in ([0], [5], [299], [3, 250, 7], list(range(64)), list(range(130, 300))):
        sub = A[rows].contiguous()
        got = bits(bi.gemm(sub, W, c_dtype=bi.F32))
        assert np.array_equal(got, full[rows]), rows
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(5))
    got = bits(bi.gemm(A[perm.cuda()].contiguous(), W, c_dtype=bi.F32))
    assert np.array_equal(got, full[perm.numpy()])


def test_gemm_row_invariance_across_tile_widths(bi):
    """Both MMA forms take 256-wide tiles for M > 256 and 128-wide tiles otherwise: here a vocabulary-wide
    matrix (N > 65536, single-CTA form).  Same MMA sequence per element, so the same bits."""
    K, N = 128, 65792
    A = rand_bf16((520, K), 1.0, 610)
    W = rand_bf16((N, K), 0.02, 611)
    full = bits(bi.gemm(A, W, c_dtype=bi.F32))
    for rows in ([0], [519], list(range(256, 512)), [7, 300, 2, 450]):
        got = bits(bi.gemm(A[rows].contiguous(), W, c_dtype=bi.F32))
        assert np.array_equal(got, full[rows]), rows


def test_gemm_variant_mode_splits_k(bi):
    """Variant mode: still close to the oracle, but its bits follow M (negative control)."""
    K, N = 4096, 256
    A = rand_bf16((64, K), 1.0, 700)
    W = rand_bf16((N, K), 0.02, 701)
    inv = bi.gemm(A, W, c_dtype=bi.F32, mode=bi.INVARIANT)
    var = bi.gemm(A, W, c_dtype=bi.F32, mode=bi.VARIANT)
    torch.cuda.synchronize()
    assert bi.gemm_workspace_size(64, N, K, bi.VARIANT) > 0
    ref = oracle.matmul(f32(A), f32(W))
    assert rel_fro(f32(var), ref) < 1e-5
    assert not np.array_equal(bits(inv), bits(var))
    # variant is deterministic run to run
    var2 = bi.gemm(A, W, c_dtype=bi.F32, mode=bi.VARIANT)
    assert np.array_equal(bits(var), bits(var2))


def test_gemm_rejects_bad_shapes(bi):
    A = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bi.BIError) as e:
        bi.gemm(A, W)
    assert e.value.status == bi.BI_ERR_SHAPE


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def make_decode_case(seq_lens, H, Hkv, Dh, seed):
    B = len(seq_lens)
    max_pages = max((s + 15) // 16 for s in seq_lens) + 1
    num_pages = sum((s + 15) // 16 for s in seq_lens) + 8
    kv = PagedKV(num_pages, Hkv, Dh, max_pages, B, seed=seed)
    hist = []
    for i, s in enumerate(seq_lens):
        k, v = synth.kv_history(s, Hkv, Dh, seed * 1000 + i, device="cuda")
        kv.write(i, k, v)
        hist.append((f32(k), f32(v)))
    q = synth.normal_bf16((B, H, Dh), 1.0, seed + 7, "cuda")
    return kv, hist, q


def oracle_decode(q, hist, H, Hkv):
    B = q.shape[0]
    qf = f32(q)
    out = np.zeros(qf.shape, np.float32)
    for i in range(B):
        k, v = hist[i]
        for h in range(H):
            g = h // (H // Hkv)
            out[i, h] = oracle.attention_head(qf[i, h], k[:, g], v[:, g])
    return out


@pytest.mark.parametrize("H,Hkv,Dh", [(32, 8, 128), (4, 2, 64), (8, 8, 128)])
def test_decode_attention_parity(bi, H, Hkv, Dh):
    seq_lens = [1, 15, 16, 17, 255, 256, 257, 700, 1500]
    kv, hist, q = make_decode_case(seq_lens, H, Hkv, Dh, seed=3)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    st = bi.new_status()
    out = bi.decode_attention(q, kv.k[0], kv.v[0], kv.table_tensor(), sl, max(seq_lens), out_dtype=bi.F32,
                              status=st)
    bi.check_status(st)
    ref = oracle_decode(q, hist, H, Hkv)
    err = np.max(np.abs(f32(out) - ref))
    assert err <= ATTN_MAX_ABS, err


def test_decode_attention_long_contexts(bi):
    """Contexts up to 32768 positions (128 splits): oracle parity on sampled heads,
    the same bits alone and batched, and the batch-variant plan within tolerance."""
    H, Hkv, Dh = 32, 8, 128
    seq_lens = [32768, 20001, 4097, 1]
    kv, hist, q = make_decode_case(seq_lens, H, Hkv, Dh, seed=11)
    table = kv.table_tensor()
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    st = bi.new_status()
    full = bi.decode_attention(q, kv.k[0], kv.v[0], table, sl, max(seq_lens), out_dtype=bi.F32, status=st)
    bi.check_status(st)
    qf, out = f32(q), f32(full)
    for i in range(len(seq_lens)):
        k, v = hist[i]
        for h in (0, 13, 31):
            ref = oracle.attention_head(qf[i, h], k[:, h // 4], v[:, h // 4])
            assert np.max(np.abs(out[i, h] - ref)) <= ATTN_MAX_ABS, (i, h)
    alone = bi.decode_attention(q[:1].contiguous(), kv.k[0], kv.v[0], table[:1].contiguous(), sl[:1].contiguous(),
                                seq_lens[0], out_dtype=bi.F32)
    assert np.array_equal(bits(alone)[0], bits(full)[0])
    var = bi.decode_attention(q, kv.k[0], kv.v[0], table, sl, max(seq_lens), out_dtype=bi.F32, mode=bi.VARIANT)
    assert np.max(np.abs(f32(var) - out)) <= 2 * ATTN_MAX_ABS


def test_decode_attention_batch_invariance(bi):
    H, Hkv, Dh = 32, 8, 128
    rng = np.random.default_rng(9)
    seq_lens = [int(s) for s in rng.integers(128, 3000, 24)]
    kv, hist, q = make_decode_case(seq_lens, H, Hkv, Dh, seed=4)
    table = kv.table_tensor()
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    full = bits(bi.decode_attention(q, kv.k[0], kv.v[0], table, sl, max(seq_lens)))
    for rows in ([0], [5], [23], [3, 19, 7], list(range(12))):
        r = torch.tensor(rows, device="cuda")
        # a different grid bound (max_seq_len) must not change any bits either
        got = bits(bi.decode_attention(q[r].contiguous(), kv.k[0], kv.v[0], table[r].contiguous(), sl[r].contiguous(),
                                       kv.max_pages * 16))
        assert np.array_equal(got, full[rows]), rows


def test_decode_variant_mode_differs_somewhere(bi):
    """Variant mode: within tolerance of the oracle, but a request's pieces (and
    so its bits) change with the batch; invariant mode does not."""
    H, Hkv, Dh = 32, 8, 128
    seq_lens = [300, 900, 1700, 2100]
    kv, hist, q = make_decode_case(seq_lens, H, Hkv, Dh, seed=5)
    table = kv.table_tensor()
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    ref = oracle_decode(q, hist, H, Hkv)
    one = dict(q=q[:1].contiguous(), table=table[:1].contiguous(), sl=sl[:1].contiguous())
    for mode in (bi.INVARIANT, bi.VARIANT):
        full = bi.decode_attention(q, kv.k[0], kv.v[0], table, sl, max(seq_lens), out_dtype=bi.F32, mode=mode)
        alone = bi.decode_attention(one["q"], kv.k[0], kv.v[0], one["table"], one["sl"], seq_lens[0],
                                    out_dtype=bi.F32, mode=mode)
        assert np.max(np.abs(f32(full) - ref)) <= ATTN_MAX_ABS
        same = np.array_equal(bits(alone)[0], bits(full)[0])
        assert same == (mode == bi.INVARIANT)


@pytest.mark.parametrize("H,Hkv,Dh", [(32, 8, 128), (8, 8, 128), (4, 2, 64), (16, 2, 128), (8, 1, 64)])
def test_prefill_matches_decode_bitwise(bi, H, Hkv, Dh):
    """The output at position p is the same bits from prefill (any chunking) and from decode at s = p + 1
    (GQA groups of 1, 2, 4 and 8 heads: 16, 8, 4 and 2 query tokens per prefill CTA)."""
    G = H // Hkv
    n = 600
    kv, hist, _ = make_decode_case([n], H, Hkv, Dh, seed=6)
    q = synth.normal_bf16((n, H, Dh), 1.0, 77, "cuda")
    table = kv.table_tensor()
    cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
    p0 = torch.tensor([0], dtype=torch.int32, device="cuda")
    pre = bits(bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], table, out_dtype=bi.F32))
    # the same queries as a batch of decode requests sharing the page table
    positions = np.array([0, 1, 15, 16, 255, 256, 257, 511, 512, 599])
    qd = q[torch.from_numpy(positions).cuda()].contiguous()
    td = table.expand(len(positions), -1).contiguous()
    sl = torch.from_numpy((positions + 1).astype(np.int32)).cuda()
    dec = bits(bi.decode_attention(qd, kv.k[0], kv.v[0], td, sl, n, out_dtype=bi.F32))
    assert np.array_equal(dec, pre[positions])
    # a chunked prefill: two ragged blocks [0,250) and [250,600) as two "requests"
    cu2 = torch.tensor([0, 250, n], dtype=torch.int32, device="cuda")
    p02 = torch.tensor([0, 250], dtype=torch.int32, device="cuda")
    t2 = table.expand(2, -1).contiguous()
    pre2 = bits(bi.prefill_attention(q, cu2, p02, kv.k[0], kv.v[0], t2, out_dtype=bi.F32))
    assert np.array_equal(pre2, pre)
    # parity of a few positions against the oracle
    k, v = hist[0]
    qf = f32(q)
    pre_f = pre.view(np.float32)
    for p in (0, 255, 256, 599):
        for h in (0, H // 2 + 1, H - 1):
            g = h // G
            ref = oracle.attention_head(qf[p, h], k[:p + 1, g], v[:p + 1, g])
            assert np.max(np.abs(pre_f[p, h] - ref)) <= ATTN_MAX_ABS


def test_prefill_dense_oracle_parity(bi):
    """Every position of a 600-token prompt (three chunks, the last one partial), for heads of four different
    KV groups, against the oracle's unsplit softmax attention."""
    H, Hkv, Dh = 32, 8, 128
    G = H // Hkv
    n = 600
    kv, hist, _ = make_decode_case([n], H, Hkv, Dh, seed=16)
    q = synth.normal_bf16((n, H, Dh), 1.0, 78, "cuda")
    cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
    p0 = torch.tensor([0], dtype=torch.int32, device="cuda")
    got = f32(bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], kv.table_tensor(), out_dtype=bi.F32))
    k, v = hist[0]
    qf = f32(q)
    worst = 0.0
    for h in (0, 5, 13, 31):
        g = h // G
        for p in range(n):
            ref = oracle.attention_head(qf[p, h], k[:p + 1, g], v[:p + 1, g])
            worst = max(worst, float(np.max(np.abs(got[p, h] - ref))))
    assert worst <= ATTN_MAX_ABS, worst


def ragged_prefill_case(H, Hkv, Dh, seed):
    """Five requests, each continuing a cached prefix: q_len [5, 37, 300, 1, 130] at q_pos0
    [0, 250, 17, 600, 256] (chunk boundaries inside blocks, blocks that start mid-chunk, a one-token block,
    CTAs whose 128 rows straddle requests)."""
    q_len = [5, 37, 300, 1, 130]
    q_pos0 = [0, 250, 17, 600, 256]
    ctx = [a + b for a, b in zip(q_len, q_pos0)]
    kv, hist, _ = make_decode_case(ctx, H, Hkv, Dh, seed=seed)
    T = sum(q_len)
    q = synth.normal_bf16((T, H, Dh), 1.0, seed + 5, "cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_len)]), dtype=torch.int32, device="cuda")
    p0 = torch.tensor(q_pos0, dtype=torch.int32, device="cuda")
    tok_req = np.repeat(np.arange(len(q_len)), q_len)
    tok_pos = np.concatenate([np.arange(a, a + b) for a, b in zip(q_pos0, q_len)])
    return kv, hist, q, cu, p0, tok_req, tok_pos


@pytest.mark.parametrize("H,Hkv,Dh", [(32, 8, 128), (8, 1, 64), (16, 16, 128), (4, 2, 64)])
def test_prefill_ragged_batch_equals_decode(bi, H, Hkv, Dh):
    """A ragged batch of five prompt blocks: each token's output is the bits decode gives it alone."""
    kv, hist, q, cu, p0, tok_req, tok_pos = ragged_prefill_case(H, Hkv, Dh, seed=21)
    table = kv.table_tensor()
    st = bi.new_status()
    pre = bits(bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], table, out_dtype=bi.F32, status=st))
    bi.check_status(st)
    idx = torch.from_numpy(tok_req.astype(np.int64)).cuda()
    dec = bits(bi.decode_attention(q, kv.k[0], kv.v[0], table[idx].contiguous(),
                                   torch.from_numpy((tok_pos + 1).astype(np.int32)).cuda(), int(tok_pos.max()) + 1,
                                   out_dtype=bi.F32))
    assert np.array_equal(pre, dec)
    # bf16 output: the same values rounded once
    pre16 = bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], table)
    assert np.array_equal(bits(pre16), bits(torch.from_numpy(pre.view(np.float32)).to(torch.bfloat16)))


def test_prefill_variant_mode_negative_control(bi):
    """Batch-variant prefill cuts every query's keys by the occupancy rule of its batch: within the parity
    tolerance of the invariant result, the same bits on a repeat, and different bits somewhere (the split
    follows the batch)."""
    H, Hkv, Dh = 32, 8, 128
    kv, hist, q, cu, p0, tok_req, tok_pos = ragged_prefill_case(H, Hkv, Dh, seed=22)
    table = kv.table_tensor()
    inv = bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], table, out_dtype=bi.F32)
    var = bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], table, out_dtype=bi.F32, mode=bi.VARIANT)
    again = bi.prefill_attention(q, cu, p0, kv.k[0], kv.v[0], table, out_dtype=bi.F32, mode=bi.VARIANT)
    assert np.array_equal(bits(var), bits(again))
    assert float((var - inv).abs().max()) <= ATTN_MAX_ABS
    assert not np.array_equal(bits(var), bits(inv))
    # one query checked against the oracle directly
    t = int(np.argmax(tok_pos))
    r, p = int(tok_req[t]), int(tok_pos[t])
    k, v = hist[r]
    ref = oracle.attention_head(f32(q)[t, 3], k[:p + 1, 0], v[:p + 1, 0])
    assert np.max(np.abs(f32(var)[t, 3] - ref)) <= ATTN_MAX_ABS


def test_attention_bad_page_reports_status(bi):
    H, Hkv, Dh = 4, 2, 64
    kv, hist, q = make_decode_case([40], H, Hkv, Dh, seed=8)
    table = kv.table_tensor().clone()
    table[0, 1] = 10 ** 6  # outside the pool
    sl = torch.tensor([40], dtype=torch.int32, device="cuda")
    st = bi.new_status()
    bi.decode_attention(q, kv.k[0], kv.v[0], table, sl, 40, status=st)
    with pytest.raises(bi.BIError) as e:
        bi.check_status(st)
    assert e.value.status == bi.BI_ERR_DEVICE


# ---------------------------------------------------------------------------
# RoPE + KV append, argmax, embedding
# ---------------------------------------------------------------------------

def test_rope_kv_append_matches_oracle(bi):
    H, Hkv, Dh, T = 32, 8, 128, 9
    qkv = synth.normal_bf16((T, (H + 2 * Hkv) * Dh), 1.0, 90, "cuda").float()
    pos = np.array([0, 1, 2, 17, 100, 4095, 4096, 30000, 33000], np.int32)
    req = np.zeros(T, np.int32)
    kv = PagedKV(3000, Hkv, Dh, 2100, 1, seed=1)
    kv.ensure(0, 33001)
    c, s = bi.rope_table(33001, Dh, 500000.0)
    q_out = torch.empty(T, H, Dh, dtype=torch.bfloat16, device="cuda")
    st = bi.new_status()
    bi.rope_kv_append(qkv, torch.from_numpy(req).cuda(), torch.from_numpy(pos).cuda(), c.cuda(), s.cuda(), q_out,
                      kv.k[0], kv.v[0], kv.table_tensor(), H, Hkv, Dh, st)
    bi.check_status(st)
    x = f32(qkv).reshape(T, H + 2 * Hkv, Dh)
    ref_q = oracle.bf16_round(oracle.rope_apply(x[:, :H], pos[:, None], 500000.0))
    ref_k = oracle.bf16_round(oracle.rope_apply(x[:, H:H + Hkv], pos[:, None], 500000.0))
    ref_v = oracle.bf16_round(x[:, H + Hkv:])
    assert np.array_equal(f32(q_out), ref_q)
    table = kv.table
    for t in range(T):
        pg, sl = table[0, pos[t] // 16], pos[t] % 16
        assert np.array_equal(f32(kv.k[0][pg, :, sl]), ref_k[t])
        assert np.array_equal(f32(kv.v[0][pg, :, sl]), ref_v[t])


def test_rope_table_matches_oracle(bi):
    c, s = bi.rope_table(5000, 128, 500000.0)
    oc, os_ = oracle.rope_table(5000, 128, 500000.0)
    assert np.array_equal(c.numpy(), oc) and np.array_equal(s.numpy(), os_)


def test_argmax_ties_nan_and_random(bi):
    rng = np.random.default_rng(21)
    x = rng.integers(-3, 4, (37, 128256)).astype(np.float32)
    x[3, :] = -np.inf
    x[4, 1000] = np.nan
    x[4, 5] = np.nan
    x[5, 128255] = 100.0
    x[6, 0] = 100.0
    x[6, 7] = 100.0
    got = bi.argmax(torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.array_equal(got, oracle.argmax_rows(x))
    assert got[4] == 5 and got[5] == 128255 and got[6] == 0 and got[3] == 0


def test_embed(bi):
    E = synth.normal_bf16((2048, 256), 1.0, 31, "cuda")
    ids = torch.tensor([5, 0, 2047, 5], dtype=torch.int32, device="cuda")
    x = bi.embed(E, ids)
    assert np.array_equal(bits(x), bits(E[ids.long()]))
    st = bi.new_status()
    bi.embed(E, torch.tensor([3, 9999], dtype=torch.int32, device="cuda"), status=st)
    with pytest.raises(bi.BIError):
        bi.check_status(st)
