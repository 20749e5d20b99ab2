"""Thin ctypes binding of libbi (include/bi.h).

Argument marshalling only: every step of the forward path runs in the CUDA
library.  PyTorch provides device memory and streams.  Importing this module
loads ``_build/libbi.so`` and raises if it has not been built — there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

BI_OK, BI_ERR_INVALID, BI_ERR_SHAPE, BI_ERR_UNSUPPORTED, BI_ERR_CUDA, BI_ERR_TIMEOUT, BI_ERR_DEVICE, \
    BI_ERR_WORKSPACE = range(8)
INVARIANT, VARIANT = 0, 1
BF16, F32 = 0, 1
EP_NONE, EP_RESIDUAL, EP_SWIGLU = 0, 1, 2
KV_CHUNK, PAGE = 256, 16

_STATUS_NAMES = {0: "BI_OK", 1: "BI_ERR_INVALID", 2: "BI_ERR_SHAPE", 3: "BI_ERR_UNSUPPORTED", 4: "BI_ERR_CUDA",
                 5: "BI_ERR_TIMEOUT", 6: "BI_ERR_DEVICE", 7: "BI_ERR_WORKSPACE"}


class BIError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libbi.so is not built ({path}); run invariant_fixed_order_gb300.build.build()")
    return ctypes.CDLL(path)


_lib = _load()
LIB_PATH = _build.LIB

_vp, _i32, _i64, _f32, _f64, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                    ctypes.c_double, ctypes.c_size_t)
_i32p = ctypes.POINTER(ctypes.c_int32)


class ModelConfigC(ctypes.Structure):
    _fields_ = [("d", _i32), ("H", _i32), ("Hkv", _i32), ("Dh", _i32), ("F", _i32), ("V", _i32),
                ("n_layers", _i32), ("eps", _f32), ("rope_theta", _f64), ("max_pos", _i32)]


class ModelWeightsC(ctypes.Structure):
    _fields_ = [("embed", _vp), ("gamma_final", _vp), ("w_lm", _vp), ("gamma_attn", ctypes.POINTER(_vp)),
                ("w_qkv", ctypes.POINTER(_vp)), ("w_o", ctypes.POINTER(_vp)), ("gamma_ffn", ctypes.POINTER(_vp)),
                ("w_gu", ctypes.POINTER(_vp)), ("w_down", ctypes.POINTER(_vp))]


class KVCacheC(ctypes.Structure):
    _fields_ = [("k", ctypes.POINTER(_vp)), ("v", ctypes.POINTER(_vp)), ("num_pages", _i32)]


class BatchC(ctypes.Structure):
    _fields_ = [("B", _i32), ("q_len", _i32p), ("pos0", _i32p), ("token_ids", _vp), ("page_table", _vp),
                ("max_pages", _i32), ("R", _i32), ("logit_rows", _i32p), ("meta", _vp)]


def _proto(name, restype, *args):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(args)
    return f


_proto("bi_last_error", ctypes.c_char_p)
_proto("bi_version", _i32)
_proto("bi_check_status", _i32, _vp, _vp)
_proto("bi_reset_status", _i32, _vp, _vp)
_proto("bi_rmsnorm", _i32, _vp, _vp, _vp, _i64, _i32, _f32, _vp)
_proto("bi_gemm_workspace_size", _sz, _i64, _i32, _i32, _i32)
_proto("bi_gemm", _i32, _vp, _vp, _vp, _i32, _vp, _i32, _i64, _i32, _i32, _i32, _vp, _sz, _vp, _vp)
_proto("bi_pack_gate_up", _i32, _vp, _vp, _vp, _i32, _i32, _vp)
_proto("bi_gemm_wait_test", _i32, _vp, _vp, _vp, _i32, _i64, _i32, _i32, ctypes.c_uint64, _i32, _vp, _vp)
_proto("bi_rope_kv_append", _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
       _i32, _vp, _vp)
_proto("bi_rope_table", _i32, _vp, _vp, _i32, _i32, _f64)
_proto("bi_decode_attention_workspace_size", _sz, _i32, _i32, _i32, _i32, _i32)
_proto("bi_decode_attention", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
       _f32, _i32, _vp, _sz, _vp, _vp)
_proto("bi_decode_attention_noalloc", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
       _i32, _f32, _i32, _vp, _vp)
_proto("bi_prefill_attention_workspace_size", _sz, _i32, _i32, _i32, _i32, _i32)
_proto("bi_prefill_attention", _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
       _i32, _i32, _f32, _i32, _vp, _sz, _vp, _vp)
_proto("bi_argmax", _i32, _vp, _vp, _i32, _i32, _vp)
_proto("bi_log_softmax_workspace_size", _sz, _i32, _i32)
_proto("bi_log_softmax", _i32, _vp, _vp, _i32, _i32, _vp, _sz, _vp)
_proto("bi_sample_workspace_size", _sz, _i32, _i32)
_proto("bi_sample", _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _sz, _vp)
_proto("bi_embed", _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp)
_proto("bi_model_create", _i32, ctypes.POINTER(ModelConfigC), ctypes.POINTER(ModelWeightsC),
       ctypes.POINTER(_vp))
_proto("bi_model_destroy", None, _vp)
_proto("bi_forward_workspace_size", _sz, ctypes.POINTER(ModelConfigC), _i32, _i32, _i32, _i32)
_proto("bi_forward_step", _i32, _vp, ctypes.POINTER(BatchC), ctypes.POINTER(KVCacheC), _vp, _vp, _vp, _i32, _vp,
       _sz, _vp, _vp)


def _check(rc: int) -> None:
    if rc != BI_OK:
        raise BIError(rc, _lib.bi_last_error().decode(errors="replace"))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def version() -> int:
    return int(_lib.bi_version())


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor, stream=None) -> None:
    _check(_lib.bi_check_status(_d(status, "status", _I32), _stream(stream)))


def reset_status(status: torch.Tensor, stream=None) -> None:
    _check(_lib.bi_reset_status(_d(status, "status", _I32), _stream(stream)))


_BF16, _F32, _I32 = (torch.bfloat16,), (torch.float32,), (torch.int32,)
_U32 = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _d(t, name: str, dtypes=None, optional: bool = False):
    """The device pointer of a dense CUDA tensor (the C ABI reads it as a flat
    row-major array), after checking that it is one; None stays NULL when the
    argument is optional."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name}: a CUDA tensor is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor (the library reads it as a dense row-major array)")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name}: expected dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    return _p(t)


def _shape(t, name: str, *dims, optional: bool = False, min_rows: bool = False):
    """Checks t's shape against the sizes passed to the C ABI (None: any), before any pointer is taken: the
    library builds its copies and stores from those sizes, so a tensor of another shape would be read or
    written out of bounds.  min_rows: the first dimension may be larger (rows past it are never touched)."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name}: a CUDA tensor is required")
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name}: expected a CUDA tensor")
    got = tuple(int(x) for x in t.shape)
    want = tuple(dims)
    ok = len(got) == len(want) and all(w is None or g == w or (min_rows and i == 0 and g >= w)
                                       for i, (g, w) in enumerate(zip(got, want)))
    if not ok:
        shown = "(" + ", ".join("*" if w is None else str(w) for w in want) + ("," if len(want) == 1 else "") + ")"
        raise ValueError(f"{name}: expected shape {shown}{' (or more rows)' if min_rows else ''}, got {got}")


def _out_dt(c_dtype: int):
    return _F32 if c_dtype == F32 else _BF16


# ---- kernels ------------------------------------------------------------------

def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-5, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    d = x.shape[-1]
    out = torch.empty_like(x) if out is None else out
    _shape(gamma, "gamma", d)
    _shape(out, "out", *x.shape)
    _check(_lib.bi_rmsnorm(_d(x, "x", _BF16), _d(gamma, "gamma", _BF16), _d(out, "out", _BF16), x.numel() // d, d,
                           eps, _stream(stream)))
    return out


def gemm_workspace_size(M: int, N: int, K: int, mode: int = INVARIANT) -> int:
    return int(_lib.bi_gemm_workspace_size(M, N, K, mode))


def gemm(A: torch.Tensor, W: torch.Tensor, out: torch.Tensor | None = None, c_dtype: int = BF16,
         residual: torch.Tensor | None = None, ep: int = EP_NONE, mode: int = INVARIANT,
         ws: torch.Tensor | None = None, status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _shape(A, "A", None, None)
    M, K = A.shape
    _shape(W, "W", None, K)
    N = W.shape[0]
    ncol = N // 2 if ep == EP_SWIGLU else N
    if out is None:
        out = torch.empty(M, ncol, device=A.device, dtype=torch.float32 if c_dtype == F32 else torch.bfloat16)
    _shape(out, "out", M, ncol)
    _shape(residual, "residual", M, N, optional=True)
    need = gemm_workspace_size(M, N, K, mode)
    if need and (ws is None or ws.numel() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=A.device)
    _check(_lib.bi_gemm(_d(A, "A", _BF16), _d(W, "W", _BF16), _d(out, "out", _out_dt(c_dtype)), c_dtype,
                        _d(residual, "residual", _BF16, optional=True), ep, M, N, K, mode,
                        _d(ws, "ws", optional=True), 0 if ws is None else ws.numel() * ws.element_size(),
                        _d(status, "status", _I32, optional=True), _stream(stream)))
    return out


def gemm_wait_test(A: torch.Tensor, W: torch.Tensor, out: torch.Tensor, status: torch.Tensor,
                   wait_limit_ns: int = 1_000_000, skip_stage: int = 0, stream=None) -> None:
    """bi_gemm_wait_test: the GEMM with a short wait limit and one ring stage's copies withheld (its bounded
    wait runs out and the kernel reports through status)."""
    _shape(A, "A", None, None)
    M, K = A.shape
    _shape(W, "W", None, K)
    N = W.shape[0]
    _shape(out, "out", M, N)
    _check(_lib.bi_gemm_wait_test(_d(A, "A", _BF16), _d(W, "W", _BF16), _d(out, "out", _F32), F32, M, N, K,
                                  wait_limit_ns, skip_stage, _d(status, "status", _I32), _stream(stream)))


def pack_gate_up(w_gate: torch.Tensor, w_up: torch.Tensor, stream=None) -> torch.Tensor:
    _shape(w_gate, "w_gate", None, None)
    F, d = w_gate.shape
    _shape(w_up, "w_up", F, d)
    out = torch.empty(2 * F, d, dtype=torch.bfloat16, device=w_gate.device)
    _check(_lib.bi_pack_gate_up(_d(w_gate, "w_gate", _BF16), _d(w_up, "w_up", _BF16), _d(out, "out", _BF16), F, d,
                                _stream(stream)))
    return out


def rope_table(n_pos: int, Dh: int, theta: float):
    c = torch.empty(n_pos, Dh // 2, dtype=torch.float32)
    s = torch.empty(n_pos, Dh // 2, dtype=torch.float32)
    _check(_lib.bi_rope_table(_p(c), _p(s), n_pos, Dh, theta))
    return c, s


def rope_kv_append(qkv, tok_req, tok_pos, rope_cos, rope_sin, q_out, k_cache, v_cache, page_table, H, Hkv, Dh,
                   status, stream=None):
    _shape(qkv, "qkv", None, (H + 2 * Hkv) * Dh)
    T = qkv.shape[0]
    _shape(tok_req, "tok_req", T)
    _shape(tok_pos, "tok_pos", T)
    _shape(rope_cos, "rope_cos", None, Dh // 2)
    _shape(rope_sin, "rope_sin", rope_cos.shape[0], Dh // 2)
    _shape(q_out, "q_out", T, H, Dh)
    _shape(k_cache, "k_cache", None, Hkv, PAGE, Dh)
    _shape(v_cache, "v_cache", *k_cache.shape)
    _shape(page_table, "page_table", None, None)
    _check(_lib.bi_rope_kv_append(_d(qkv, "qkv", _F32), _d(tok_req, "tok_req", _I32), _d(tok_pos, "tok_pos", _I32),
                                  _d(rope_cos, "rope_cos", _F32), _d(rope_sin, "rope_sin", _F32),
                                  rope_cos.shape[0], _d(q_out, "q_out", _BF16), _d(k_cache, "k_cache", _BF16),
                                  _d(v_cache, "v_cache", _BF16), _d(page_table, "page_table", _I32),
                                  page_table.shape[-1], k_cache.shape[0], T, H, Hkv, Dh,
                                  _d(status, "status", _I32, optional=True),
                                  _stream(stream)))


def decode_attention_workspace_size(B: int, H: int, Dh: int, max_seq_len: int, mode: int = INVARIANT) -> int:
    return int(_lib.bi_decode_attention_workspace_size(B, H, Dh, max_seq_len, mode))


def _attn_shapes(q, k_cache, v_cache, page_table, rows: int):
    _shape(q, "q", rows, None, None)
    _, H, Dh = q.shape
    _shape(k_cache, "k_cache", None, None, PAGE, Dh)
    _shape(v_cache, "v_cache", *k_cache.shape)
    _shape(page_table, "page_table", None, None)
    return H, k_cache.shape[1]


def decode_attention(q, k_cache, v_cache, page_table, seq_lens, max_seq_len: int, out_dtype: int = BF16,
                     mode: int = INVARIANT, scale: float | None = None, ws=None, status=None, out=None,
                     stream=None) -> torch.Tensor:
    """scale None: the library's default fl32(1 / fl32(sqrt(Dh)))."""
    _shape(q, "q", None, None, None)
    B, H, Dh = q.shape
    _attn_shapes(q, k_cache, v_cache, page_table, B)
    Hkv = k_cache.shape[1]
    _shape(page_table, "page_table", B, None)
    _shape(seq_lens, "seq_lens", B)
    if out is None:
        out = torch.empty(B, H, Dh, device=q.device, dtype=torch.float32 if out_dtype == F32 else torch.bfloat16)
    _shape(out, "out", B, H, Dh)
    need = decode_attention_workspace_size(B, H, Dh, max_seq_len, mode)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(_lib.bi_decode_attention(_d(q, "q", _BF16), _d(k_cache, "k_cache", _BF16), _d(v_cache, "v_cache", _BF16),
                                    _d(page_table, "page_table", _I32), _d(seq_lens, "seq_lens", _I32),
                                    _d(out, "out", _out_dt(out_dtype)), out_dtype, B, H, Hkv, Dh,
                                    page_table.shape[-1], k_cache.shape[0], max_seq_len,
                                    0.0 if scale is None else scale, mode,
                                    _d(ws, "ws"), ws.numel() * ws.element_size(),
                                    _d(status, "status", _I32, optional=True), _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def decode_attention_noalloc(q, k_cache, v_cache, page_table, seq_lens, max_seq_len: int, out_dtype: int = BF16,
                             mode: int = INVARIANT, scale: float | None = None, status=None, out=None,
                             stream=None) -> torch.Tensor:
    """decode_attention without a workspace: the library's static device
    scratch holds the split partials (for callers that cannot allocate)."""
    _shape(q, "q", None, None, None)
    B, H, Dh = q.shape
    _attn_shapes(q, k_cache, v_cache, page_table, B)
    Hkv = k_cache.shape[1]
    _shape(page_table, "page_table", B, None)
    _shape(seq_lens, "seq_lens", B)
    if out is None:
        out = torch.empty(B, H, Dh, device=q.device, dtype=torch.float32 if out_dtype == F32 else torch.bfloat16)
    _shape(out, "out", B, H, Dh)
    _check(_lib.bi_decode_attention_noalloc(_d(q, "q", _BF16), _d(k_cache, "k_cache", _BF16),
                                            _d(v_cache, "v_cache", _BF16), _d(page_table, "page_table", _I32),
                                            _d(seq_lens, "seq_lens", _I32), _d(out, "out", _out_dt(out_dtype)),
                                            out_dtype, B, H, Hkv, Dh, page_table.shape[-1], k_cache.shape[0],
                                            max_seq_len, 0.0 if scale is None else scale, mode,
                                            _d(status, "status", _I32, optional=True), _stream(stream)))
    return out


def prefill_attention_workspace_size(T: int, H: int, Dh: int, max_seq_len: int, mode: int = INVARIANT) -> int:
    return int(_lib.bi_prefill_attention_workspace_size(T, H, Dh, max_seq_len, mode))


def prefill_attention(q, cu_q, q_pos0, k_cache, v_cache, page_table, out_dtype: int = BF16,
                      scale: float | None = None, status=None, out=None, stream=None, mode: int = INVARIANT,
                      max_seq_len: int | None = None, ws=None) -> torch.Tensor:
    """Causal attention of ragged query blocks.  max_seq_len None: the page table's capacity (a bound the
    caller need not compute); scale None: the library's default."""
    _shape(q, "q", None, None, None)
    T, H, Dh = q.shape
    _shape(cu_q, "cu_q", None)
    B = cu_q.shape[0] - 1
    _attn_shapes(q, k_cache, v_cache, page_table, T)
    Hkv = k_cache.shape[1]
    _shape(q_pos0, "q_pos0", B)
    _shape(page_table, "page_table", B, None)
    if max_seq_len is None:
        max_seq_len = page_table.shape[-1] * PAGE
    if out is None:
        out = torch.empty(T, H, Dh, device=q.device, dtype=torch.float32 if out_dtype == F32 else torch.bfloat16)
    _shape(out, "out", T, H, Dh)
    need = prefill_attention_workspace_size(T, H, Dh, max_seq_len, mode)
    if need and (ws is None or ws.numel() < need):
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(_lib.bi_prefill_attention(_d(q, "q", _BF16), _d(cu_q, "cu_q", _I32), _d(q_pos0, "q_pos0", _I32),
                                     _d(k_cache, "k_cache", _BF16), _d(v_cache, "v_cache", _BF16),
                                     _d(page_table, "page_table", _I32), _d(out, "out", _out_dt(out_dtype)), out_dtype,
                                     B, T, H, Hkv, Dh, page_table.shape[-1], k_cache.shape[0], max_seq_len,
                                     0.0 if scale is None else scale, mode, _d(ws, "ws", optional=True),
                                     0 if ws is None else ws.numel() * ws.element_size(),
                                     _d(status, "status", _I32, optional=True), _stream(stream)))
    return out


def argmax(logits: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _shape(logits, "logits", None, None)
    R, V = logits.shape
    out = torch.empty(R, dtype=torch.int32, device=logits.device) if out is None else out
    _shape(out, "out", R)
    _check(_lib.bi_argmax(_d(logits, "logits", _F32), _d(out, "out", _I32), R, V, _stream(stream)))
    return out


def log_softmax_workspace_size(R: int, V: int) -> int:
    return int(_lib.bi_log_softmax_workspace_size(R, V))


def log_softmax(logits: torch.Tensor, out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    _shape(logits, "logits", None, None)
    R, V = logits.shape
    out = torch.empty(R, V, dtype=torch.float32, device=logits.device) if out is None else out
    _shape(out, "out", R, V)
    need = log_softmax_workspace_size(R, V)
    if ws is None or ws.numel() < need:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=logits.device)
    _check(_lib.bi_log_softmax(_d(logits, "logits", _F32), _d(out, "out", _F32), R, V, _d(ws, "ws"),
                               ws.numel() * ws.element_size(), _stream(stream)))
    return out


def sample_workspace_size(R: int, V: int) -> int:
    return int(_lib.bi_sample_workspace_size(R, V))


def sample(logits: torch.Tensor, seeds: torch.Tensor, positions: torch.Tensor, temperatures: torch.Tensor,
           out: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Seeded Gumbel-max tokens; seeds uint32 (or int32 holding the same bits), positions int32,
    temperatures fp32, all DEVICE [R]."""
    _shape(logits, "logits", None, None)
    R, V = logits.shape
    out = torch.empty(R, dtype=torch.int32, device=logits.device) if out is None else out
    for name, t in (("seeds", seeds), ("positions", positions), ("temperatures", temperatures), ("out", out)):
        _shape(t, name, R)
    need = sample_workspace_size(R, V)
    if ws is None or ws.numel() < need:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=logits.device)
    _check(_lib.bi_sample(_d(logits, "logits", _F32), _d(seeds, "seeds", _U32), _d(positions, "positions", _I32),
                          _d(temperatures, "temperatures", _F32), _d(out, "out", _I32), R, V, _d(ws, "ws"),
                          ws.numel() * ws.element_size(), _stream(stream)))
    return out


def embed(E: torch.Tensor, ids: torch.Tensor, status=None, out=None, stream=None) -> torch.Tensor:
    _shape(E, "E", None, None)
    V, d = E.shape
    _shape(ids, "ids", None)
    T = ids.shape[0]
    out = torch.empty(T, d, dtype=torch.bfloat16, device=E.device) if out is None else out
    _shape(out, "out", T, d)
    _check(_lib.bi_embed(_d(E, "E", _BF16), _d(ids, "ids", _I32), _d(out, "out", _BF16), T, V, d,
                         _d(status, "status", _I32, optional=True), _stream(stream)))
    return out


# ---- model ----------------------------------------------------------------------

def _ptr_array(tensors):
    arr = (_vp * len(tensors))(*[t.data_ptr() for t in tensors])
    return arr


class Model:
    """Owns nothing but the library's model handle; the weight tensors are
    borrowed (kept referenced here so they outlive the handle)."""

    def __init__(self, cfg, layers: list, head: dict, max_pos: int):
        self.cfg = cfg
        self.layers = layers
        self.head = head
        self.max_pos = max_pos
        self._c = ModelConfigC(cfg.d, cfg.H, cfg.Hkv, cfg.Dh, cfg.F, cfg.V, cfg.n_layers, cfg.eps, cfg.rope_theta,
                               max_pos)
        if len(layers) != cfg.n_layers:
            raise ValueError(f"layers: expected {cfg.n_layers}, got {len(layers)}")
        qkv = (cfg.H + 2 * cfg.Hkv) * cfg.Dh
        want = {"gamma_attn": (cfg.d,), "w_qkv": (qkv, cfg.d), "w_o": (cfg.d, cfg.H * cfg.Dh), "gamma_ffn": (cfg.d,),
                "w_gu": (2 * cfg.F, cfg.d), "w_down": (cfg.d, cfg.F)}
        for i, L in enumerate(layers):
            for k in ("gamma_attn", "w_qkv", "w_o", "gamma_ffn", "w_gu", "w_down"):
                _shape(L[k], f"layers[{i}][{k}]", *want[k])
                _d(L[k], f"layers[{i}][{k}]", _BF16)
        for k, shp in (("embed", (cfg.V, cfg.d)), ("gamma_final", (cfg.d,)), ("w_lm", (cfg.V, cfg.d))):
            _shape(head[k], f"head[{k}]", *shp)
            _d(head[k], f"head[{k}]", _BF16)
        self._arrays = {k: _ptr_array([L[k] for L in layers])
                        for k in ("gamma_attn", "w_qkv", "w_o", "gamma_ffn", "w_gu", "w_down")}
        w = ModelWeightsC(head["embed"].data_ptr(), head["gamma_final"].data_ptr(), head["w_lm"].data_ptr(),
                          self._arrays["gamma_attn"], self._arrays["w_qkv"], self._arrays["w_o"],
                          self._arrays["gamma_ffn"], self._arrays["w_gu"], self._arrays["w_down"])
        h = ctypes.c_void_p()
        _check(_lib.bi_model_create(ctypes.byref(self._c), ctypes.byref(w), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.bi_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_size(self, max_T: int, max_B: int, max_R: int, max_seq: int) -> int:
        return int(_lib.bi_forward_workspace_size(ctypes.byref(self._c), max_T, max_B, max_R, max_seq))

    def forward_step(self, q_len, pos0, token_ids: torch.Tensor, page_table: torch.Tensor, kv_k: list, kv_v: list,
                     logit_rows, ws: torch.Tensor, status: torch.Tensor, logits_out=None, tokens_out=None,
                     hidden_out=None, mode: int = INVARIANT, stream=None, meta: torch.Tensor | None = None):
        """One ragged step.  q_len / pos0 / logit_rows are host int sequences; meta (optional) is the
        step's per-token metadata already on the device (the layout bi_batch documents)."""
        B = len(q_len)
        if len(pos0) != B:
            raise ValueError(f"pos0: expected {B} entries, got {len(pos0)}")
        ql = (ctypes.c_int32 * B)(*[int(v) for v in q_len])
        p0 = (ctypes.c_int32 * B)(*[int(v) for v in pos0])
        R = len(logit_rows)
        rows = (ctypes.c_int32 * max(R, 1))(*[int(v) for v in logit_rows])
        T = sum(int(v) for v in q_len)
        c = self.cfg
        _shape(token_ids, "token_ids", T)
        _shape(page_table, "page_table", B, None, min_rows=True)
        _shape(meta, "meta", 3 * T + R, optional=True)
        _shape(logits_out, "logits_out", R, c.V, optional=True, min_rows=True)
        _shape(tokens_out, "tokens_out", R, optional=True, min_rows=True)
        _shape(hidden_out, "hidden_out", T, c.d, optional=True, min_rows=True)
        if len(kv_k) != c.n_layers or len(kv_v) != c.n_layers:
            raise ValueError(f"kv_k / kv_v: expected {c.n_layers} layers")
        for name, caches in (("kv_k", kv_k), ("kv_v", kv_v)):
            for i, t in enumerate(caches):
                _shape(t, f"{name}[{i}]", kv_k[0].shape[0], c.Hkv, PAGE, c.Dh)
        batch = BatchC(B, ql, p0, _d(token_ids, "token_ids", _I32).value, _d(page_table, "page_table", _I32).value,
                       page_table.shape[-1], R, rows,
                       None if meta is None else _d(meta, "meta", _I32).value)
        for name, caches in (("kv_k", kv_k), ("kv_v", kv_v)):
            for i, t in enumerate(caches):
                _d(t, f"{name}[{i}]", _BF16)
        ka, va = _ptr_array(kv_k), _ptr_array(kv_v)
        kv = KVCacheC(ka, va, kv_k[0].shape[0])
        _check(_lib.bi_forward_step(self._h, ctypes.byref(batch), ctypes.byref(kv),
                                    _d(logits_out, "logits_out", _F32, optional=True),
                                    _d(tokens_out, "tokens_out", _I32, optional=True),
                                    _d(hidden_out, "hidden_out", _BF16, optional=True), mode, _d(ws, "ws"),
                                    ws.numel() * ws.element_size(), _d(status, "status", _I32), _stream(stream)))
