"""Pins for the CPU oracle: each test checks it against something other than
itself — values the pages print, closed forms, invariants, library routines in
float64, or brute force on tiny inputs.  A plausible mistake in the oracle (a
dropped term, a wrong sign or index, a transposed operand) fails at least one.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f32_bits(x) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def bf16_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 with torch's conversion (library RNE)."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def rand_bf16(rng, shape, std=1.0, mean=0.0):
    return bf16_f64(rng.standard_normal(shape) * std + mean).astype(np.float32)


# ---------------------------------------------------------------------------
# "Non-associativity, concretely" (Figure 1): the printed witness
# ---------------------------------------------------------------------------

def test_witness_serial_and_pairwise_bits(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "witness_nonassoc.json")))
    p = np.array([int(b, 16) for b in g["inputs_bits"]], np.uint32).view(np.float32)
    pr = g["printed"]
    serial = oracle.sum_serial(p)
    pairwise = oracle.sum_pairwise(p)
    assert f32_bits(serial) == int(pr["serial_result_bits"], 16)
    assert f32_bits(pairwise) == int(pr["pairwise_result_bits"], 16)
    assert f32_bits(pairwise) - f32_bits(serial) == pr["ulp_distance"]
    # printed intermediates
    s01 = oracle.sum_serial(p[:2])
    assert s01 == np.float32(pr["serial_after_p0_p1"])
    s012 = oracle.sum_serial(p[:3])
    assert abs(float(s012) - pr["serial_after_p2"]) < 5e-9
    assert oracle.sum_serial(p[2:]) == np.float32(pr["pairwise_p2_plus_p3"])
    exact = sum(Fraction(float(x)) for x in p)
    # the page's summands are not printed; the reconstruction's exact sum agrees
    # with the printed 0.00066451075 to within 2 units of its last digit
    assert abs(float(exact) - pr["exact_sum"]) < 2e-11
    # both answers exceed the exact sum, errors of the same sign
    assert Fraction(float(serial)) > exact and Fraction(float(pairwise)) > exact


def test_sum_orders_agree_with_fraction_on_exact_cases():
    # integers below 2^24 add exactly in any order
    x = np.arange(1, 1000, dtype=np.float32)
    assert oracle.sum_serial(x) == np.float32(sum(range(1, 1000)))
    assert oracle.sum_pairwise(x) == np.float32(sum(range(1, 1000)))


def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8],
                                 np.float32)]).astype(np.float32)
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))
    assert np.isnan(oracle.bf16_round(np.array([np.nan], np.float32)))[0]


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("c", [0.5, -3.0, 1e-3, 7.25])
def test_rmsnorm_constant_closed_form(c):
    d, eps = 256, 1e-5
    gamma = rand_bf16(np.random.default_rng(1), d, 0.02, 1.0)
    x = np.full((3, d), c, np.float32)
    y = oracle.rmsnorm(x, gamma, eps, round_bf16=False)
    closed = c / np.sqrt(c * c + eps) * gamma.astype(np.float64)
    np.testing.assert_allclose(y, np.broadcast_to(closed, y.shape), rtol=2e-6)
    yb = oracle.rmsnorm(x, gamma, eps, round_bf16=True)
    assert np.array_equal(yb, np.broadcast_to(bf16_f64(closed), y.shape).astype(np.float32))


def test_rmsnorm_matches_float64_library():
    rng = np.random.default_rng(2)
    x = rand_bf16(rng, (17, 4096))
    gamma = rand_bf16(rng, 4096, 0.02, 1.0)
    y = oracle.rmsnorm(x, gamma, 1e-5, round_bf16=False)
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt(np.mean(x64 ** 2, axis=1, keepdims=True) + 1e-5) * gamma
    np.testing.assert_allclose(y, ref, rtol=2e-6, atol=1e-7)


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 8, 14336), (5, 33, 4096), (13, 17, 64)])
def test_matmul_integer_valued_is_exact(M, N, K):
    rng = np.random.default_rng(3)
    A = rng.integers(-8, 9, (M, K)).astype(np.float32)
    W = rng.integers(-8, 9, (N, K)).astype(np.float32)
    C = oracle.matmul(A, W)
    ref = A.astype(np.int64) @ W.astype(np.int64).T
    assert np.array_equal(C.astype(np.int64), ref)


def test_matmul_orientation_and_float64():
    rng = np.random.default_rng(4)
    A = rand_bf16(rng, (7, 96))
    W = rand_bf16(rng, (40, 96), 0.02)
    C = oracle.matmul(A, W)
    np.testing.assert_allclose(C, A.astype(np.float64) @ W.astype(np.float64).T, rtol=1e-5, atol=1e-6)
    # a non-square case that would fail if the operand were transposed
    assert C.shape == (7, 40)


# ---------------------------------------------------------------------------
# Softmax and attention
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 255, 256, 257, 4096])
def test_softmax_rows_sum_to_one(n):
    rng = np.random.default_rng(5)
    s = (rng.standard_normal(n) * 4).astype(np.float32)
    p = oracle.softmax(s)
    assert abs(float(np.sum(p.astype(np.float64))) - 1.0) <= n * 2.0 ** -24 + 1e-7
    np.testing.assert_allclose(p, scipy.special.softmax(s.astype(np.float64)), rtol=1e-5, atol=1e-9)


def test_softmax_is_shift_invariant_beyond_the_exp_range():
    """softmax(s + c) = softmax(s): with s on a 2^-10 grid the shift by 512 is exact in binary32, so the
    values must agree bit for bit although e^512 is far beyond binary32's range."""
    rng = np.random.default_rng(15)
    s = (np.round(rng.standard_normal(300) * 4 * 1024) / 1024).astype(np.float32)
    p = oracle.softmax(s)
    assert np.array_equal(oracle.softmax(s + np.float32(512.0)), p)
    assert np.array_equal(oracle.softmax(s - np.float32(512.0)), p)
    # two logits 100 apart: the larger takes all the mass to binary32 precision
    p2 = oracle.softmax(np.float32([0.0, 100.0]))
    assert p2[1] == np.float32(1.0) and 0.0 <= p2[0] < 1e-40


@pytest.mark.parametrize("n", [1, 3, 256, 700])
def test_attention_identical_keys_returns_mean_of_v(n):
    rng = np.random.default_rng(6)
    Dh = 128
    q = rand_bf16(rng, Dh)
    k = np.broadcast_to(rand_bf16(rng, Dh), (n, Dh)).copy()
    v = rand_bf16(rng, (n, Dh))
    out = oracle.attention_head(q, k, v)
    np.testing.assert_allclose(out, v.astype(np.float64).mean(axis=0), rtol=1e-6, atol=1e-6 * n ** 0.5)


def test_attention_one_key_returns_v_exactly():
    rng = np.random.default_rng(7)
    q, k, v = rand_bf16(rng, 64), rand_bf16(rng, (1, 64)), rand_bf16(rng, (1, 64))
    assert np.array_equal(oracle.attention_head(q, k, v), v[0])


def test_attention_matches_float64_softmax():
    rng = np.random.default_rng(8)
    n, Dh = 300, 128
    q, k, v = rand_bf16(rng, Dh), rand_bf16(rng, (n, Dh)), rand_bf16(rng, (n, Dh))
    out = oracle.attention_head(q, k, v)
    s = (k.astype(np.float64) @ q.astype(np.float64)) / np.sqrt(Dh)
    ref = scipy.special.softmax(s) @ v.astype(np.float64)
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("n,chunk", [(1, 256), (256, 256), (257, 256), (1000, 256), (5000, 256), (77, 16)])
def test_split_merge_equals_unsplit_within_rounding(n, chunk):
    rng = np.random.default_rng(9)
    Dh = 128
    q, k, v = rand_bf16(rng, Dh, 2.0), rand_bf16(rng, (n, Dh)), rand_bf16(rng, (n, Dh))
    a = oracle.attention_head(q, k, v)
    b = oracle.attention_head_split(q, k, v, chunk)
    s = (k.astype(np.float64) @ q.astype(np.float64)) / np.sqrt(Dh)
    ref = scipy.special.softmax(s) @ v.astype(np.float64)
    np.testing.assert_allclose(a, ref, rtol=2e-5, atol=2e-6)
    np.testing.assert_allclose(b, ref, rtol=2e-5, atol=2e-6)


# ---------------------------------------------------------------------------
# SwiGLU, argmax
# ---------------------------------------------------------------------------

def test_swiglu_matches_expit_and_special_values():
    rng = np.random.default_rng(10)
    g = (rng.standard_normal(4000) * 3).astype(np.float32)
    u = rng.standard_normal(4000).astype(np.float32)
    h = oracle.swiglu(g, u, round_bf16=False)
    ref = g.astype(np.float64) * scipy.special.expit(g.astype(np.float64)) * u
    np.testing.assert_allclose(h, ref, rtol=2e-6, atol=1e-7)
    # silu(0) = 0; silu(large) = g; gate and up are not interchangeable
    assert oracle.swiglu(np.float32([0.0]), np.float32([5.0]))[0] == 0.0
    assert oracle.swiglu(np.float32([40.0]), np.float32([2.0]), round_bf16=False)[0] == np.float32(80.0)
    assert oracle.swiglu(np.float32([-2.0]), np.float32([1.0]))[0] != oracle.swiglu(np.float32([1.0]),
                                                                                    np.float32([-2.0]))[0]


def test_argmax_brute_force_and_ties():
    rng = np.random.default_rng(11)
    for _ in range(200):
        n = int(rng.integers(1, 300))
        x = rng.integers(-3, 4, n).astype(np.float32)  # many ties
        assert oracle.argmax(x) == int(np.argmax(x))  # numpy returns the first maximum
    x = np.array([1.0, 5.0, 5.0, -np.inf, 5.0], np.float32)
    assert oracle.argmax(x) == 1
    assert oracle.argmax(np.array([1.0, np.nan, 9.0, np.nan], np.float32)) == 1
    assert oracle.argmax(np.array([np.nan, 1.0], np.float32)) == 0
    assert oracle.argmax(np.array([-np.inf, -np.inf], np.float32)) == 0
    assert oracle.argmax(np.array([-0.0, 0.0], np.float32)) == 0  # -0 == +0: lowest index
    rows = rng.standard_normal((9, 50)).astype(np.float32)
    assert np.array_equal(oracle.argmax_rows(rows), np.argmax(rows, axis=1))


# ---------------------------------------------------------------------------
# Rotary embedding
# ---------------------------------------------------------------------------

def rope_complex_f64(x, pos, theta):
    """Rotate-half RoPE as a complex rotation: (x_i + j x_{i+D/2}) * e^{j pos theta^(-2i/D)}."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    inv = theta ** (-np.arange(half) * 2.0 / D)
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * np.asarray(pos, np.float64)[..., None] * inv)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(12)
    x = rand_bf16(rng, (5, 128))
    assert np.array_equal(oracle.rope_apply(x, np.zeros(5, np.int32), 500000.0), x)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(13)
    x = rand_bf16(rng, (40, 128))
    pos = rng.integers(0, 40000, 40).astype(np.int32)
    out = oracle.rope_apply(x, pos, 500000.0)
    np.testing.assert_allclose(out, rope_complex_f64(x, pos, 500000.0), rtol=0, atol=2e-5)


def test_rope_relative_position_property():
    rng = np.random.default_rng(14)
    q, k = rand_bf16(rng, 64), rand_bf16(rng, 64)
    d1 = float(np.dot(oracle.rope_apply(q[None], [100], 500000.0)[0].astype(np.float64),
                      oracle.rope_apply(k[None], [37], 500000.0)[0].astype(np.float64)))
    d2 = float(np.dot(oracle.rope_apply(q[None], [1163], 500000.0)[0].astype(np.float64),
                      oracle.rope_apply(k[None], [1100], 500000.0)[0].astype(np.float64)))
    assert abs(d1 - d2) < 1e-4 * (1 + abs(d1))
    # and the dot product does change with the offset
    d3 = float(np.dot(oracle.rope_apply(q[None], [101], 500000.0)[0].astype(np.float64),
                      oracle.rope_apply(k[None], [37], 500000.0)[0].astype(np.float64)))
    assert abs(d3 - d1) > 1e-3


# ---------------------------------------------------------------------------
# Whole layer: float64 brute force from library routines
# ---------------------------------------------------------------------------

def layer_f64(dims, w, q_lens, pos0, k_hist, v_hist, x, round_fn):
    d, H, Hkv, Dh = dims.d, dims.H, dims.Hkv, dims.Dh
    W = {k: np.asarray(v, np.float64) for k, v in w.items()}
    x = np.asarray(x, np.float64)
    T = x.shape[0]

    def rms(a, g):
        return a / np.sqrt(np.mean(a * a, axis=-1, keepdims=True) + dims.eps) * g

    y = round_fn(rms(x, W["gamma_attn"]))
    qkv = y @ W["w_qkv"].T
    q = qkv[:, :H * Dh].reshape(T, H, Dh)
    k = qkv[:, H * Dh:(H + Hkv) * Dh].reshape(T, Hkv, Dh)
    v = qkv[:, (H + Hkv) * Dh:].reshape(T, Hkv, Dh)
    pos = np.concatenate([np.arange(p, p + n) for p, n in zip(pos0, q_lens)])
    q = round_fn(rope_complex_f64(q, pos[:, None], dims.rope_theta))
    k = round_fn(rope_complex_f64(k, pos[:, None], dims.rope_theta))
    v = round_fn(v)
    att = np.zeros((T, H, Dh))
    t0 = 0
    for i, (p0, n) in enumerate(zip(pos0, q_lens)):
        K = np.concatenate([np.asarray(k_hist[i][:p0], np.float64), k[t0:t0 + n]], axis=0)
        Vv = np.concatenate([np.asarray(v_hist[i][:p0], np.float64), v[t0:t0 + n]], axis=0)
        for t in range(n):
            p = p0 + t
            for h in range(H):
                g = h // (H // Hkv)
                s = K[:p + 1, g] @ q[t0 + t, h] / np.sqrt(Dh)
                att[t0 + t, h] = scipy.special.softmax(s) @ Vv[:p + 1, g]
        t0 += n
    att = att.reshape(T, H * Dh)
    x1 = round_fn(x + round_fn(att) @ W["w_o"].T)
    y2 = round_fn(rms(x1, W["gamma_ffn"]))
    gt = y2 @ W["w_gate"].T
    up = y2 @ W["w_up"].T
    hdn = round_fn(gt * scipy.special.expit(gt) * up)
    x2 = round_fn(x1 + hdn @ W["w_down"].T)
    return x2, att


def tiny_case(seed=20):
    rng = np.random.default_rng(seed)
    dims = oracle.Dims(d=256, H=4, Hkv=2, Dh=64, F=1024)
    w = {
        "gamma_attn": rand_bf16(rng, 256, 0.02, 1.0),
        "w_qkv": rand_bf16(rng, (512, 256), 0.02),
        "w_o": rand_bf16(rng, (256, 256), 0.02),
        "gamma_ffn": rand_bf16(rng, 256, 0.02, 1.0),
        "w_gate": rand_bf16(rng, (1024, 256), 0.02),
        "w_up": rand_bf16(rng, (1024, 256), 0.02),
        "w_down": rand_bf16(rng, (256, 1024), 0.02),
    }
    q_lens, pos0 = [3, 1, 5], [0, 40, 7]
    k_hist = [rand_bf16(rng, (max(p, 1), 2, 64)) for p in pos0]
    v_hist = [rand_bf16(rng, (max(p, 1), 2, 64)) for p in pos0]
    x = rand_bf16(rng, (sum(q_lens), 256))
    return dims, w, q_lens, pos0, k_hist, v_hist, x


def rel_fro(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_layer_pure_fp32_matches_float64_brute_force():
    dims, w, q_lens, pos0, kh, vh, x = tiny_case()
    dims.round_bf16 = False
    x_out, attn, _, _ = oracle.layer_forward(dims, w, q_lens, pos0, kh, vh, x)
    ref_x, ref_att = layer_f64(dims, w, q_lens, pos0, kh, vh, x, lambda a: a)
    assert rel_fro(attn, ref_att) < 1e-5
    assert rel_fro(x_out - x, ref_x - x) < 1e-5


def test_layer_bf16_storage_matches_float64_with_same_rounding():
    dims, w, q_lens, pos0, kh, vh, x = tiny_case(21)
    x_out, attn, _, _ = oracle.layer_forward(dims, w, q_lens, pos0, kh, vh, x)
    ref_x, ref_att = layer_f64(dims, w, q_lens, pos0, kh, vh, x, bf16_f64)
    assert rel_fro(attn, ref_att) < 5e-3
    assert rel_fro(x_out - x, ref_x - x) < 5e-3
    # most stored elements agree exactly
    assert np.mean(x_out == ref_x) > 0.97


def test_layer_gqa_mapping():
    """Heads h read kv head h // (H/Hkv): make every key identical so each head's
    output is the mean of its kv head's V, and give kv heads distinct constant V."""
    dims = oracle.Dims(d=64, H=4, Hkv=2, Dh=32, F=64, round_bf16=False)
    rng = np.random.default_rng(22)
    w = {"gamma_attn": np.ones(64, np.float32), "w_qkv": np.zeros((256, 64), np.float32),
         "w_o": np.zeros((64, 128), np.float32),
         "gamma_ffn": np.ones(64, np.float32), "w_gate": np.zeros((64, 64), np.float32),
         "w_up": np.zeros((64, 64), np.float32), "w_down": np.zeros((64, 64), np.float32)}
    n = 6
    kh = np.zeros((n, 2, 32), np.float32)
    vh = np.zeros((n, 2, 32), np.float32)
    vh[:, 0, :] = 1.0
    vh[:, 1, :] = 2.0
    x = rand_bf16(rng, (1, 64))
    # new token's v is zero (w_qkv = 0): each head sees n history values and one zero
    _, attn, _, _ = oracle.layer_forward(dims, w, [1], [n], [kh], [vh], x)
    per_head = attn.reshape(4, 32)
    expect = np.array([1.0, 1.0, 2.0, 2.0]) * n / (n + 1)
    np.testing.assert_allclose(per_head, np.broadcast_to(expect[:, None], (4, 32)), rtol=1e-6)


def test_layer_is_causal_and_chunking_free():
    """Outputs at earlier positions do not change when later tokens are appended,
    and prefilling a prompt in two chunks equals prefilling it at once."""
    dims, w, _, _, _, _, _ = tiny_case(23)
    rng = np.random.default_rng(23)
    n = 9
    x = rand_bf16(rng, (n, 256))
    empty = [np.zeros((1, 2, 64), np.float32)]
    full, _, k_all, v_all = oracle.layer_forward(dims, w, [n], [0], empty, empty, x)
    head, _, k1, v1 = oracle.layer_forward(dims, w, [4], [0], empty, empty, x[:4])
    assert np.array_equal(full[:4], head)
    tail, _, _, _ = oracle.layer_forward(dims, w, [n - 4], [4], [k1[0]], [v1[0]], x[4:])
    assert np.array_equal(full[4:], tail)


def test_lm_head_matches_float64_and_argmax():
    rng = np.random.default_rng(24)
    dims = oracle.Dims(d=256, H=4, Hkv=2, Dh=64, F=1024, round_bf16=False)
    g = rand_bf16(rng, 256, 0.02, 1.0)
    W = rand_bf16(rng, (2048, 256), 0.02)
    x = rand_bf16(rng, (6, 256))
    rows = np.array([5, 0, 3], np.int32)
    logits, toks = oracle.lm_head(dims, g, W, x, rows)
    xr = x[rows].astype(np.float64)
    y = xr / np.sqrt(np.mean(xr * xr, axis=1, keepdims=True) + 1e-5) * g
    ref = y @ W.astype(np.float64).T
    np.testing.assert_allclose(logits, ref, rtol=1e-5, atol=1e-5)
    assert np.array_equal(toks, np.argmax(logits, axis=1))


def test_embed_gathers_rows():
    E = np.arange(40, dtype=np.float32).reshape(10, 4)
    assert np.array_equal(oracle.embed(E, [3, 0, 9]), E[[3, 0, 9]])


# ---------------------------------------------------------------------------
# "Mathematically equivalent is not bitwise equivalent": logprobs are the
# log_softmax of the logits
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 7, 128256])
def test_log_softmax_uniform_row_is_minus_log_n(n):
    lp = oracle.log_softmax_rows(np.full((1, n), 3.25, np.float32))
    assert np.allclose(lp, -np.log(n), rtol=0, atol=1e-12)


def test_log_softmax_two_columns_closed_form():
    a, b = np.float32(1.5), np.float32(-2.25)
    lp = oracle.log_softmax_rows(np.array([[a, b]], np.float32))[0]
    d = float(b) - float(a)
    assert abs(lp[0] - (-np.log1p(np.exp(d)))) < 1e-14
    assert abs(lp[1] - (d - np.log1p(np.exp(d)))) < 1e-14


def test_log_softmax_beyond_the_float64_exp_range():
    """Logits 1000 apart: e^1000 overflows float64, but the logprobs are [-1000 - log1p(e^-1000), -log1p(...)]
    = [-1000, 0] exactly (e^-1000 underflows to 0)."""
    lp = oracle.log_softmax_rows(np.float32([[0.0, 1000.0], [1000.0, 0.0], [-1000.0, 1000.0]]))
    assert np.array_equal(lp, [[-1000.0, 0.0], [0.0, -1000.0], [-2000.0, 0.0]])


def test_log_softmax_matches_library_and_invariants():
    rng = np.random.default_rng(11)
    # multiples of 2^-10 below 32 in magnitude: adding 64 below is exact in binary32
    x = np.clip(np.round(rng.standard_normal((5, 3000)) * 4 * 1024) / 1024, -31, 31).astype(np.float32)
    lp = oracle.log_softmax_rows(x)
    ref = scipy.special.log_softmax(x.astype(np.float64), axis=1)
    assert np.max(np.abs(lp - ref)) < 1e-10
    assert np.allclose(np.exp(lp).sum(axis=1), 1.0, atol=1e-12)
    assert np.all(lp <= 0)
    assert np.array_equal(np.argmax(lp, axis=1), np.argmax(x, axis=1))
    # shifting a row by a constant (exact in binary32 here) leaves its logprobs unchanged
    lp2 = oracle.log_softmax_rows(x + np.float32(64.0))
    assert np.max(np.abs(lp2 - lp)) < 1e-12
    # each row on its own gives the same values as in the batch
    assert np.array_equal(oracle.log_softmax_rows(x[2:3]), lp[2:3])


# ---------------------------------------------------------------------------
# "The weaker guarantees, which are usually enough": seeded Gumbel sampling
# ---------------------------------------------------------------------------

# MurmurHash3 x86_32 verification values published with the reference
# implementation of the hash (key, seed, hash).
MURMUR3_VECTORS = [(b"", 0, 0x00000000), (b"", 1, 0x514E28B7), (b"", 0xFFFFFFFF, 0x81F16F39),
                   (b"\0\0\0\0", 0, 0x2362F9DE), (b"aaaa", 0x9747B28C, 0x5A97808A), (b"abc", 0, 0xB3DD93FA),
                   (b"Hello, world!", 0x9747B28C, 0x24884CBA),
                   (b"The quick brown fox jumps over the lazy dog", 0x9747B28C, 0x2FA826CD)]


@pytest.mark.parametrize("key,seed,expect", MURMUR3_VECTORS)
def test_murmur3_published_vectors(key, seed, expect):
    assert oracle.murmur3_32(key, seed) == expect


@pytest.mark.parametrize("t", [0.5, 1.0, 2.0])
def test_gumbel_sampling_frequencies_follow_softmax(t):
    """Over many positions the draws follow softmax(x / t) (chi-square, 3 degrees of freedom): pins the
    sign of the Gumbel transform, the temperature's use and the uniform mapping."""
    x = np.array([0.0, 1.0, 2.0, 0.5], np.float32)
    n = 20000
    rows = np.tile(x, (n, 1))
    tok = oracle.sample_gumbel_rows(rows, np.full(n, 7), np.arange(n), np.full(n, t))
    counts = np.bincount(tok, minlength=4)
    p = scipy.special.softmax(x.astype(np.float64) / t)
    chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
    assert chi2 < 30.0, (counts, n * p)


def test_gumbel_sampling_depends_on_seed_position_and_logits_only():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(500).astype(np.float32)
    a = [oracle.sample_gumbel(x, 11, p, 1.0) for p in range(64)]
    assert a == [oracle.sample_gumbel(x, 11, p, 1.0) for p in range(64)]   # reproducible
    assert a != [oracle.sample_gumbel(x, 12, p, 1.0) for p in range(64)]   # the seed matters
    assert len(set(a)) > 20                                                  # positions draw afresh
    # a column far above the rest always wins (Gumbel noise lies within [-3.2, 23.2])
    y = x.copy()
    y[123] = 60.0
    assert all(oracle.sample_gumbel(y, 5, p, 1.0) == 123 for p in range(32))
    # lowering a column that did not win leaves the winner (the draws are per column)
    for p in range(16):
        w = oracle.sample_gumbel(x, 9, p, 1.0)
        z = x.copy()
        z[(w + 1) % x.size] = -1e30
        assert oracle.sample_gumbel(z, 9, p, 1.0) == w


def test_gumbel_sampling_special_rows():
    x = np.array([0.5, np.nan, 3.0, np.nan], np.float32)
    assert oracle.sample_gumbel(x, 1, 0, 1.0) == 1          # a NaN beats every number, first NaN wins
    y = np.array([1.0, 4.0, 4.0, -2.0], np.float32)
    assert oracle.sample_gumbel(y, 1, 0, 0.0) == 1          # temperature 0: greedy, lowest index of ties
    assert oracle.sample_gumbel(y, 1, 0, -1.0) == 1
