"""The C ABI's error behaviour (include/bi.h): every call validates its
arguments before it launches anything and returns a status with a message.
These calls fail validation, so no device memory is touched and no GPU is
needed; the pointers passed are never dereferenced.  Each group of cases runs
in a child process that sees no GPU (CUDA_VISIBLE_DEVICES empty): should a
check ever let one of these calls through, it fails with a CUDA error instead
of launching a kernel on a fake address."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BI_OK, BI_ERR_INVALID, BI_ERR_SHAPE, BI_ERR_UNSUPPORTED, BI_ERR_CUDA, BI_ERR_TIMEOUT, BI_ERR_DEVICE, \
    BI_ERR_WORKSPACE = range(8)

P = ctypes.c_void_p
FAKE = P(0x10000)    # a pointer value that validation sees as non-null (never dereferenced)
FAKE2 = P(0x90000)
i32, i64, f32, f64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_size_t


def load_lib():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from invariant_fixed_order_gb300 import build
    L = ctypes.CDLL(build.build())
    L.bi_last_error.restype = ctypes.c_char_p
    return L


def call(lib, name, *args):
    f = getattr(lib, name)
    f.restype = ctypes.c_int32
    return f(*args)


def case_gemm_validation(lib):
    # K not a multiple of 64
    assert call(lib, "bi_gemm", FAKE, FAKE, FAKE, i32(1), None, i32(0), i64(4), i32(128), i32(100), i32(0),
                None, sz(0), None, None) == BI_ERR_SHAPE
    assert b"K % 64" in lib.bi_last_error()
    # N not a multiple of 128
    assert call(lib, "bi_gemm", FAKE, FAKE, FAKE, i32(1), None, i32(0), i64(4), i32(100), i32(128), i32(0),
                None, sz(0), None, None) == BI_ERR_SHAPE
    # null operand
    assert call(lib, "bi_gemm", None, FAKE, FAKE, i32(1), None, i32(0), i64(4), i32(128), i32(128), i32(0),
                None, sz(0), None, None) == BI_ERR_INVALID
    # residual epilogue without a residual, fused epilogue with fp32 output, bad mode
    assert call(lib, "bi_gemm", FAKE, FAKE, FAKE, i32(0), None, i32(1), i64(4), i32(128), i32(128), i32(0),
                None, sz(0), None, None) == BI_ERR_INVALID
    assert call(lib, "bi_gemm", FAKE, FAKE, FAKE, i32(1), FAKE2, i32(1), i64(4), i32(128), i32(128), i32(0),
                None, sz(0), None, None) == BI_ERR_UNSUPPORTED
    assert call(lib, "bi_gemm", FAKE, FAKE, FAKE, i32(1), None, i32(0), i64(4), i32(128), i32(128), i32(7),
                None, sz(0), None, None) == BI_ERR_INVALID
    # misaligned pointer
    assert call(lib, "bi_gemm", P(0x10004), FAKE, FAKE, i32(1), None, i32(0), i64(4), i32(128), i32(128), i32(0),
                None, sz(0), None, None) == BI_ERR_INVALID
    # the wait test: a limit outside [1 ms, 2 s], no status word
    assert call(lib, "bi_gemm_wait_test", FAKE, FAKE, FAKE, i32(1), i64(1), i32(128), i32(64),
                ctypes.c_uint64(1000), i32(0), FAKE, None) == BI_ERR_INVALID
    assert call(lib, "bi_gemm_wait_test", FAKE, FAKE, FAKE, i32(1), i64(1), i32(128), i32(64),
                ctypes.c_uint64(1000000), i32(0), None, None) == BI_ERR_INVALID
    # M = 0 is a valid no-op
    assert call(lib, "bi_gemm", None, None, None, i32(1), None, i32(0), i64(0), i32(128), i32(128), i32(0),
                None, sz(0), None, None) == BI_OK


def case_row_kernels_validation(lib):
    assert call(lib, "bi_rmsnorm", FAKE, FAKE, FAKE, i64(4), i32(100), f32(1e-5), None) == BI_ERR_SHAPE
    assert call(lib, "bi_rmsnorm", None, FAKE, FAKE, i64(4), i32(128), f32(1e-5), None) == BI_ERR_INVALID
    assert call(lib, "bi_rmsnorm", P(0x10008), FAKE, FAKE, i64(4), i32(128), f32(1e-5), None) == BI_ERR_INVALID
    assert call(lib, "bi_argmax", FAKE, FAKE, i32(2), i32(0), None) == BI_ERR_SHAPE
    assert call(lib, "bi_argmax", None, FAKE, i32(2), i32(10), None) == BI_ERR_INVALID
    assert call(lib, "bi_embed", FAKE, FAKE, FAKE, i32(3), i32(10), i32(12), None, None) == BI_ERR_SHAPE
    assert call(lib, "bi_pack_gate_up", FAKE, FAKE, FAKE, i32(30), i32(64), None) == BI_ERR_SHAPE


def case_logits_ops_validation(lib):
    n = 2 * 1000 * 4
    # logprobs written over the logits
    assert call(lib, "bi_log_softmax", FAKE, P(0x10000 + n // 2), i32(2), i32(1000), FAKE2, sz(1 << 20),
                None) == BI_ERR_INVALID
    assert b"overlap" in lib.bi_last_error()
    # workspace too small or missing
    lib.bi_log_softmax_workspace_size.restype = sz
    need = lib.bi_log_softmax_workspace_size(i32(2), i32(1000))
    assert need > 0
    assert call(lib, "bi_log_softmax", FAKE, P(0x800000), i32(2), i32(1000), FAKE2, sz(need - 16),
                None) == BI_ERR_WORKSPACE
    assert call(lib, "bi_sample", FAKE, FAKE, FAKE, FAKE, FAKE, i32(2), i32(1000), None, sz(0),
                None) == BI_ERR_WORKSPACE
    assert call(lib, "bi_sample", FAKE, FAKE, FAKE, None, FAKE, i32(2), i32(1000), FAKE2, sz(1 << 20),
                None) == BI_ERR_INVALID
    assert call(lib, "bi_sample", FAKE, FAKE, FAKE, FAKE, FAKE, i32(2), i32(0), FAKE2, sz(1 << 20),
                None) == BI_ERR_SHAPE
    # zero rows: no-ops
    assert call(lib, "bi_log_softmax", None, None, i32(0), i32(1000), None, sz(0), None) == BI_OK
    assert call(lib, "bi_sample", None, None, None, None, None, i32(0), i32(1000), None, sz(0), None) == BI_OK


class Cfg(ctypes.Structure):
    _fields_ = [("d", i32), ("H", i32), ("Hkv", i32), ("Dh", i32), ("F", i32), ("V", i32), ("n_layers", i32),
                ("eps", f32), ("rope_theta", f64), ("max_pos", i32)]


def case_model_and_step_validation(lib):
    out = P()
    bad = Cfg(d=100, H=4, Hkv=2, Dh=64, F=1024, V=2048, n_layers=1, eps=1e-5, rope_theta=5e5, max_pos=64)
    assert call(lib, "bi_model_create", ctypes.byref(bad), FAKE, ctypes.byref(out)) == BI_ERR_SHAPE
    assert "multiples" in lib.bi_last_error().decode()
    zero = Cfg(d=0, H=4, Hkv=2, Dh=64, F=1024, V=2048, n_layers=1, eps=1e-5, rope_theta=5e5, max_pos=64)
    assert call(lib, "bi_model_create", ctypes.byref(zero), FAKE, ctypes.byref(out)) == BI_ERR_SHAPE
    assert call(lib, "bi_model_create", None, FAKE, ctypes.byref(out)) == BI_ERR_INVALID
    lib.bi_forward_workspace_size.restype = sz
    good = Cfg(d=256, H=4, Hkv=2, Dh=64, F=1024, V=2048, n_layers=1, eps=1e-5, rope_theta=5e5, max_pos=64)
    assert lib.bi_forward_workspace_size(ctypes.byref(good), i32(0), i32(1), i32(1), i32(64)) == 0
    assert lib.bi_forward_workspace_size(ctypes.byref(good), i32(16), i32(4), i32(4), i32(64)) > 0
    assert call(lib, "bi_forward_step", None, FAKE, FAKE, None, None, None, i32(0), FAKE, sz(0), FAKE,
                None) == BI_ERR_INVALID
    assert call(lib, "bi_check_status", None, None) == BI_ERR_INVALID


def _decode(lib, H=32, Hkv=8, Dh=128, B=4, max_pages=64, max_seq=1000, mode=0, ws=FAKE2, ws_bytes=1 << 30):
    return call(lib, "bi_decode_attention", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, i32(1), i32(B), i32(H), i32(Hkv),
                i32(Dh), i32(max_pages), i32(100), i32(max_seq), f32(0.08), i32(mode), ws, sz(ws_bytes), FAKE,
                None)


def _prefill(lib, B=2, T=8, H=32, Hkv=8, Dh=128, max_pages=64, max_seq=1000, mode=0, ws=None, ws_bytes=0,
             cu_q=FAKE):
    return call(lib, "bi_prefill_attention", FAKE, cu_q, FAKE, FAKE, FAKE, FAKE, FAKE, i32(1), i32(B), i32(T),
                i32(H), i32(Hkv), i32(Dh), i32(max_pages), i32(100), i32(max_seq), f32(0.0), i32(mode), ws,
                sz(ws_bytes), FAKE, None)


def case_attention_validation(lib):
    assert _decode(lib, H=6, Hkv=4) == BI_ERR_UNSUPPORTED      # group 1.5
    assert _decode(lib, H=32, Hkv=2) == BI_ERR_UNSUPPORTED     # group 16
    assert _decode(lib, Dh=96) == BI_ERR_UNSUPPORTED
    assert _decode(lib, max_seq=64 * 16 + 1) == BI_ERR_SHAPE   # beyond the page table
    assert _decode(lib, max_seq=0) == BI_ERR_SHAPE
    assert _decode(lib, mode=3) == BI_ERR_INVALID
    assert _decode(lib, B=-1) == BI_ERR_SHAPE
    assert _decode(lib, B=0, ws=None, ws_bytes=0) == BI_OK
    # the invariant split plan is ceil(max_seq / 256) chunks of 256 keys for every request: the workspace
    # holds B * H * splits partial rows of Dh + 2 floats, whatever else shares the batch
    lib.bi_decode_attention_workspace_size.restype = sz
    need = lib.bi_decode_attention_workspace_size(i32(4), i32(32), i32(128), i32(1000), i32(0))
    assert need >= 4 * 32 * 4 * 130 * 4
    assert need == lib.bi_decode_attention_workspace_size(i32(4), i32(32), i32(128), i32(1024), i32(0))
    assert need < lib.bi_decode_attention_workspace_size(i32(4), i32(32), i32(128), i32(1025), i32(0))
    assert _decode(lib, ws_bytes=need - 1) == BI_ERR_WORKSPACE
    assert _decode(lib, ws=None, ws_bytes=0) == BI_ERR_WORKSPACE
    assert _decode(lib, ws=P(0x90008), ws_bytes=need) == BI_ERR_INVALID   # misaligned workspace
    # the no-alloc form rejects what does not fit its static partials array before any launch
    big = call(lib, "bi_decode_attention_noalloc", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, i32(1), i32(256), i32(64),
               i32(8), i32(128), i32(2048), i32(100), i32(32768), f32(0.08), i32(0), FAKE, None)
    assert big == BI_ERR_WORKSPACE
    # prefill: null metadata, negative sizes, an out-of-range context bound, a bad mode
    assert _prefill(lib, cu_q=None) == BI_ERR_INVALID
    assert _prefill(lib, T=-1) == BI_ERR_SHAPE
    assert _prefill(lib, max_seq=0) == BI_ERR_SHAPE
    assert _prefill(lib, max_seq=64 * 16 + 1) == BI_ERR_SHAPE
    assert _prefill(lib, mode=2) == BI_ERR_INVALID
    assert _prefill(lib, B=0) == BI_OK
    # invariant prefill needs no workspace; the batch-variant split keeps (Dh + 2) floats per query, head and
    # piece, at most max(ceil(s / 256), 16) pieces
    lib.bi_prefill_attention_workspace_size.restype = sz
    assert lib.bi_prefill_attention_workspace_size(i32(600), i32(32), i32(128), i32(1000), i32(0)) == 0
    vneed = lib.bi_prefill_attention_workspace_size(i32(600), i32(32), i32(128), i32(1000), i32(1))
    assert vneed >= 600 * 32 * 16 * 130 * 4
    assert _prefill(lib, mode=1, ws=None, ws_bytes=0) == BI_ERR_WORKSPACE
    assert _prefill(lib, mode=1, ws_bytes=64) == BI_ERR_WORKSPACE
    assert _prefill(lib, mode=1, ws=P(0x90008), ws_bytes=vneed) == BI_ERR_INVALID


CASES = sorted(n[len("case_"):] for n in list(globals()) if n.startswith("case_"))


@pytest.fixture(scope="module", autouse=True)
def built():
    load_lib()  # builds once here, so the child processes only load it


@pytest.mark.parametrize("case", CASES)
def test_validation_without_a_visible_gpu(case):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), case], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr


if __name__ == "__main__":
    globals()["case_" + sys.argv[1]](load_lib())
