"""CPU oracle for the batch-invariant forward step (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  The product path
(``invariant_fixed_order_gb300``) never imports it, and it never imports the
product package: the two share no code.

The C source is the plain definition of a Llama-style decoder step in binary32
with no fused multiply-add, plus logprobs and seeded Gumbel-max sampling in
float64; see ``oracle.h`` for the page and section each function follows
("Lockstep"; "Batch invariance and reproducible inference").
All tensors cross this wrapper as float32 numpy arrays; bf16 tensors are passed
as float32 arrays holding bf16-representable values.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP when available) into _build/liboracle.so."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler found")
    base = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class _Dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("Dh", ctypes.c_int32), ("F", ctypes.c_int32), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_double), ("round_bf16", ctypes.c_int32)]


_FP = ctypes.POINTER(ctypes.c_float)


class _LayerW(ctypes.Structure):
    _fields_ = [("gamma_attn", _FP), ("w_qkv", _FP), ("w_o", _FP), ("gamma_ffn", _FP),
                ("w_gate", _FP), ("w_up", _FP), ("w_down", _FP)]


def bind(path: str) -> ctypes.CDLL:
    """Load a compiled oracle library from ``path`` and declare its functions'
    argument types (the functions of oracle.h)."""
    L = ctypes.CDLL(path)
    f32p, i32p, i64p = _FP, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    L.orc_bf16_round.restype = ctypes.c_float
    L.orc_bf16_round.argtypes = [ctypes.c_float]
    L.orc_bf16_round_array.argtypes = [f32p, f32p, i64]
    L.orc_sum_serial.restype = ctypes.c_float
    L.orc_sum_serial.argtypes = [f32p, i64]
    L.orc_sum_pairwise.restype = ctypes.c_float
    L.orc_sum_pairwise.argtypes = [f32p, i64]
    L.orc_rmsnorm.argtypes = [f32p, f32p, f32p, i64, i32, ctypes.c_float, ctypes.c_int]
    L.orc_matmul.argtypes = [f32p, f32p, f32p, i64, i32, i32]
    L.orc_softmax.argtypes = [f32p, f32p, i32]
    L.orc_swiglu.argtypes = [f32p, f32p, f32p, i64, ctypes.c_int]
    L.orc_argmax.restype = i32
    L.orc_argmax.argtypes = [f32p, i32]
    L.orc_argmax_rows.argtypes = [f32p, i32p, i64, i32]
    f64p, u32p, u8p = (ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint32),
                       ctypes.POINTER(ctypes.c_uint8))
    L.orc_log_softmax_rows.argtypes = [f32p, f64p, i64, i32]
    L.orc_murmur3_32.restype = ctypes.c_uint32
    L.orc_murmur3_32.argtypes = [u8p, i32, ctypes.c_uint32]
    L.orc_sample_gumbel.restype = ctypes.c_int32
    L.orc_sample_gumbel.argtypes = [f32p, i32, ctypes.c_uint32, i32, ctypes.c_float]
    L.orc_sample_gumbel_rows.argtypes = [f32p, u32p, i32p, f32p, i32p, i64, i32]
    L.orc_rope_table.argtypes = [f32p, f32p, i32, i32, ctypes.c_double]
    L.orc_rope_apply.argtypes = [f32p, i32p, i64, i32, f32p, f32p, i32]
    L.orc_attention_head.argtypes = [f32p, f32p, f32p, i32, i64, i32, ctypes.c_float, f32p]
    L.orc_attention_head_split.argtypes = [f32p, f32p, f32p, i32, i64, i32,
                                           ctypes.c_float, i32, f32p]
    L.orc_layer_forward.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_LayerW), i32,
                                    i32p, i32p, i64p, f32p, f32p, f32p, f32p, f32p]
    L.orc_lm_head.argtypes = [ctypes.POINTER(_Dims), f32p, f32p, i32, f32p, i32p, i32,
                              f32p, i32p]
    L.orc_embed.argtypes = [f32p, i32, i32, i32p, i64, f32p]
    L.orc_num_threads.restype = ctypes.c_int
    L.orc_set_num_threads.argtypes = [ctypes.c_int]
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray, ty=ctypes.c_float):
    return a.ctypes.data_as(ctypes.POINTER(ty))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---- primitives -------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    x = _f32(x)
    out = np.empty_like(x)
    lib().orc_bf16_round_array(_ptr(x), _ptr(out), x.size)
    return out


def sum_serial(x) -> np.float32:
    x = _f32(x)
    return np.float32(lib().orc_sum_serial(_ptr(x), x.size))


def sum_pairwise(x) -> np.float32:
    x = _f32(x)
    return np.float32(lib().orc_sum_pairwise(_ptr(x), x.size))


def rmsnorm(x, gamma, eps: float = 1e-5, round_bf16: bool = True) -> np.ndarray:
    x, gamma = _f32(x), _f32(gamma)
    d = x.shape[-1]
    rows = x.size // d
    y = np.empty_like(x)
    _check(lib().orc_rmsnorm(_ptr(x), _ptr(gamma), _ptr(y), rows, d, eps, int(round_bf16)), "rmsnorm")
    return y


def matmul(A, W) -> np.ndarray:
    """C = A @ W.T with one serial fp32 loop over K per element."""
    A, W = _f32(A), _f32(W)
    M, K = A.shape
    N, K2 = W.shape
    assert K == K2
    C = np.empty((M, N), np.float32)
    _check(lib().orc_matmul(_ptr(A), _ptr(W), _ptr(C), M, N, K), "matmul")
    return C


def softmax(s) -> np.ndarray:
    s = _f32(s)
    p = np.empty_like(s)
    _check(lib().orc_softmax(_ptr(s), _ptr(p), s.size), "softmax")
    return p


def swiglu(g, u, round_bf16: bool = True) -> np.ndarray:
    g, u = _f32(g), _f32(u)
    h = np.empty_like(g)
    _check(lib().orc_swiglu(_ptr(g), _ptr(u), _ptr(h), g.size, int(round_bf16)), "swiglu")
    return h


def argmax(x) -> int:
    x = _f32(x)
    return int(lib().orc_argmax(_ptr(x), x.size))


def argmax_rows(x) -> np.ndarray:
    x = _f32(x)
    rows, n = x.shape
    out = np.empty(rows, np.int32)
    _check(lib().orc_argmax_rows(_ptr(x), _ptr(out, ctypes.c_int32), rows, n), "argmax_rows")
    return out


def log_softmax_rows(x) -> np.ndarray:
    """float64 logprobs of each row of fp32 logits (the definition)."""
    x = _f32(np.atleast_2d(x))
    rows, n = x.shape
    out = np.empty((rows, n), np.float64)
    _check(lib().orc_log_softmax_rows(_ptr(x), _ptr(out, ctypes.c_double), rows, n), "log_softmax_rows")
    return out


def murmur3_32(key: bytes, seed: int) -> int:
    buf = np.frombuffer(key, np.uint8).copy() if key else np.zeros(1, np.uint8)
    return int(lib().orc_murmur3_32(_ptr(buf, ctypes.c_uint8), len(key), seed & 0xffffffff))


def sample_gumbel(x, seed: int, pos: int, t: float) -> int:
    x = _f32(np.ravel(x))
    r = int(lib().orc_sample_gumbel(_ptr(x), x.size, seed & 0xffffffff, pos, t))
    if r < 0:
        raise ValueError("oracle sample_gumbel: bad arguments")
    return r


def sample_gumbel_rows(x, seeds, pos, t) -> np.ndarray:
    x = _f32(np.atleast_2d(x))
    rows, n = x.shape
    seeds = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint32).reshape(rows))
    pos = _i32(np.asarray(pos).reshape(rows))
    t = _f32(np.asarray(t).reshape(rows))
    out = np.empty(rows, np.int32)
    _check(lib().orc_sample_gumbel_rows(_ptr(x), _ptr(seeds, ctypes.c_uint32), _ptr(pos, ctypes.c_int32), _ptr(t),
                                        _ptr(out, ctypes.c_int32), rows, n), "sample_gumbel_rows")
    return out


def rope_table(n_pos: int, Dh: int, theta: float):
    c = np.empty((n_pos, Dh // 2), np.float32)
    s = np.empty((n_pos, Dh // 2), np.float32)
    _check(lib().orc_rope_table(_ptr(c), _ptr(s), n_pos, Dh, theta), "rope_table")
    return c, s


def rope_apply(x, pos, theta: float) -> np.ndarray:
    """Rotate vectors x[..., Dh] at positions pos (broadcast over leading dims)."""
    x = _f32(x).copy()
    Dh = x.shape[-1]
    pos = _i32(np.broadcast_to(np.asarray(pos, np.int32)[..., None], x.shape[:-1] + (1,))[..., 0])
    n_pos = int(pos.max()) + 1 if pos.size else 1
    c, s = rope_table(n_pos, Dh, theta)
    _check(lib().orc_rope_apply(_ptr(x), _ptr(pos, ctypes.c_int32), x.size // Dh, Dh,
                                _ptr(c), _ptr(s), n_pos), "rope_apply")
    return x


def attention_head(q, k, v, scale: float | None = None) -> np.ndarray:
    """q [Dh]; k, v [n, Dh]."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    n, Dh = k.shape
    scale = np.float32(1.0) / np.sqrt(np.float32(Dh)) if scale is None else scale
    out = np.empty(Dh, np.float32)
    _check(lib().orc_attention_head(_ptr(q), _ptr(k), _ptr(v), n, Dh, Dh, float(scale), _ptr(out)),
           "attention_head")
    return out


def attention_head_split(q, k, v, chunk: int, scale: float | None = None) -> np.ndarray:
    q, k, v = _f32(q), _f32(k), _f32(v)
    n, Dh = k.shape
    scale = np.float32(1.0) / np.sqrt(np.float32(Dh)) if scale is None else scale
    out = np.empty(Dh, np.float32)
    _check(lib().orc_attention_head_split(_ptr(q), _ptr(k), _ptr(v), n, Dh, Dh, float(scale),
                                          chunk, _ptr(out)), "attention_head_split")
    return out


# ---- decoder layer / model ---------------------------------------------------

class Dims:
    def __init__(self, d, H, Hkv, Dh, F, eps=1e-5, rope_theta=500000.0, round_bf16=True):
        self.d, self.H, self.Hkv, self.Dh, self.F = d, H, Hkv, Dh, F
        self.eps, self.rope_theta, self.round_bf16 = eps, rope_theta, round_bf16

    def c(self) -> _Dims:
        return _Dims(self.d, self.H, self.Hkv, self.Dh, self.F, self.eps, self.rope_theta,
                     int(self.round_bf16))


def layer_forward(dims: Dims, w: dict, q_lens, pos0, k_hist, v_hist, x_in):
    """One decoder layer over a ragged batch.

    w: dict of float32 arrays gamma_attn, w_qkv, w_o, gamma_ffn, w_gate, w_up, w_down.
    k_hist / v_hist: list over requests of arrays [>= pos0[i], Hkv, Dh] holding the
    history (positions < pos0[i]).
    Returns (x_out [T, d], attn_fp32 [T, H*Dh], k_new, v_new) where k_new[i] / v_new[i]
    are [pos0[i] + q_len[i], Hkv, Dh] including the appended tokens.
    """
    q_lens = [int(q) for q in q_lens]
    pos0 = [int(p) for p in pos0]
    B = len(q_lens)
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(q_lens)
    rows = [p + q for p, q in zip(pos0, q_lens)]
    row0 = np.zeros(B, np.int64)
    if B:
        row0[1:] = np.cumsum(rows)[:-1]
    total = int(sum(rows))
    kv_shape = (max(total, 1), dims.Hkv, dims.Dh)
    k_pool = np.zeros(kv_shape, np.float32)
    v_pool = np.zeros(kv_shape, np.float32)
    for i in range(B):
        if pos0[i]:
            k_pool[row0[i]:row0[i] + pos0[i]] = k_hist[i][:pos0[i]]
            v_pool[row0[i]:row0[i] + pos0[i]] = v_hist[i][:pos0[i]]
    x_in = _f32(x_in)
    T = int(cu[-1])
    x_out = np.empty((T, dims.d), np.float32)
    attn = np.empty((T, dims.H * dims.Dh), np.float32)
    keep = {k: _f32(w[k]) for k in ("gamma_attn", "w_qkv", "w_o", "gamma_ffn", "w_gate", "w_up", "w_down")}
    lw = _LayerW(*[_ptr(keep[k]) for k in ("gamma_attn", "w_qkv", "w_o", "gamma_ffn", "w_gate",
                                            "w_up", "w_down")])
    pos0_a = _i32(pos0)
    cd = dims.c()
    _check(lib().orc_layer_forward(ctypes.byref(cd), ctypes.byref(lw), B,
                                   _ptr(cu, ctypes.c_int32), _ptr(pos0_a, ctypes.c_int32),
                                   _ptr(row0, ctypes.c_int64), _ptr(k_pool), _ptr(v_pool),
                                   _ptr(x_in), _ptr(x_out), _ptr(attn)), "layer_forward")
    k_new = [k_pool[row0[i]:row0[i] + rows[i]] for i in range(B)]
    v_new = [v_pool[row0[i]:row0[i] + rows[i]] for i in range(B)]
    return x_out, attn, k_new, v_new


def lm_head(dims: Dims, gamma_final, w_lm, x, rows):
    gamma_final, w_lm, x = _f32(gamma_final), _f32(w_lm), _f32(x)
    rows = _i32(rows)
    V = w_lm.shape[0]
    R = rows.size
    logits = np.empty((R, V), np.float32)
    tokens = np.empty(R, np.int32)
    cd = dims.c()
    _check(lib().orc_lm_head(ctypes.byref(cd), _ptr(gamma_final), _ptr(w_lm), V, _ptr(x),
                             _ptr(rows, ctypes.c_int32), R, _ptr(logits),
                             _ptr(tokens, ctypes.c_int32)), "lm_head")
    return logits, tokens


def embed(E, ids) -> np.ndarray:
    E = _f32(E)
    ids = _i32(ids)
    V, d = E.shape
    x = np.empty((ids.size, d), np.float32)
    _check(lib().orc_embed(_ptr(E), V, d, _ptr(ids, ctypes.c_int32), ids.size, _ptr(x)), "embed")
    return x


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))
