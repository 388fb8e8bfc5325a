"""C-ABI checks that need no GPU: the library loads, exports every declared entry point,
reports workspace sizes, and rejects bad arguments on the host before any launch.

The pointers used below are never dereferenced on the host: every call here fails
validation before it reaches CUDA.
"""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def capi():
    from entropy_gated_kv_gb300 import build as B

    B.build()
    from entropy_gated_kv_gb300 import _capi as C

    C.load()
    return C


def header_functions() -> list[str]:
    text = (ROOT / "include" / "entropycache.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ec_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(capi):
    names = header_functions()
    assert len(names) >= 10
    lib = capi.load()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(capi.SIGNATURES), "binding and header disagree"


def test_status_strings(capi):
    lib = capi.load()
    assert lib.ec_status_string(0) == b"EC_OK"
    assert lib.ec_status_string(capi.EC_ERR_INVALID_ARG) == b"EC_ERR_INVALID_ARG"
    assert lib.ec_status_string(capi.EC_ERR_TIMEOUT) == b"EC_ERR_TIMEOUT"
    assert lib.ec_status_string(999) == b"EC_ERR_UNKNOWN"
    assert lib.ec_version() >= 100


def _params(C, **kw):
    base = dict(B=1, L=1024, Hq=32, Hkv=32, D=128, V=126464, C_max=32, k=64, n_dec=1, tau=1.0, logits_dtype=C.EC_BF16)
    base.update(kw)
    return C.EcParams(**base)


def test_workspace_sizes(capi):
    lib = capi.load()
    # one vocabulary chunk per CTA: 8192 bf16 / 4096 fp32 elements
    assert lib.ec_entropy_decode_workspace_size(32, 126464, capi.EC_BF16) >= 32 * 16 * 16
    assert lib.ec_entropy_decode_workspace_size(32, 32000, capi.EC_F32) >= 32 * 8 * 16
    assert lib.ec_entropy_decode_workspace_size(-1, 10, capi.EC_F32) == 0
    assert lib.ec_entropy_decode_workspace_size(1, 10, 7) == 0
    p = _params(capi)
    a = lib.ec_partial_attention_workspace_size(ctypes.byref(p))
    s = lib.ec_step_workspace_size(ctypes.byref(p))
    assert a > 0 and s > a + 1024 * 32 * 128 * 2
    bad = _params(capi, D=96)
    assert lib.ec_partial_attention_workspace_size(ctypes.byref(bad)) == 0
    assert lib.ec_step_workspace_size(ctypes.byref(bad)) == 0


FAKE = 0x100000  # an aligned address that is never dereferenced


def test_entropy_decode_rejects_bad_args(capi):
    lib = capi.load()
    f = lib.ec_entropy_decode
    p = ctypes.c_void_p(FAKE)
    INV = capi.EC_ERR_INVALID_ARG
    assert f(p, 32000, 4, 32000, 7, p, p, p, p, 1 << 20, None) == INV  # dtype
    assert f(p, 100, 4, 200, capi.EC_F32, p, p, p, p, 1 << 20, None) == INV  # stride < V
    assert f(p, 32001, 4, 32000, capi.EC_F32, p, p, p, p, 1 << 20, None) == INV  # stride*4 % 16
    assert f(p, 50257, 4, 50257, capi.EC_BF16, p, p, p, p, 1 << 20, None) == INV  # stride*2 % 16
    assert f(None, 32000, 4, 32000, capi.EC_F32, p, p, p, p, 1 << 20, None) == INV
    assert f(ctypes.c_void_p(FAKE + 4), 32000, 4, 32000, capi.EC_F32, p, p, p, p, 1 << 20, None) == INV
    assert f(p, 32000, 4, 32000, capi.EC_F32, p, p, p, None, 0, None) == INV  # workspace
    assert f(p, 32000, 4, 32000, capi.EC_F32, p, p, p, p, 16, None) == INV  # workspace too small
    assert f(p, 32000, -1, 32000, capi.EC_F32, p, p, p, p, 1 << 20, None) == INV
    assert f(p, 32000, 0, 32000, capi.EC_F32, None, None, None, None, 0, None) == capi.EC_OK  # empty: no-op


def test_partial_attention_rejects_bad_args(capi):
    lib = capi.load()
    f = lib.ec_partial_attention
    p = ctypes.c_void_p(FAKE)
    big = 1 << 30
    good = _params(capi)
    for bad, want in [
        (_params(capi, Hkv=5), capi.EC_ERR_INVALID_ARG),  # Hq % Hkv
        (_params(capi, D=96), capi.EC_ERR_UNSUPPORTED),
        (_params(capi, Hq=256, Hkv=1), capi.EC_ERR_UNSUPPORTED),  # g > 128
        (_params(capi, B=0), capi.EC_ERR_INVALID_ARG),
        (_params(capi, L=0), capi.EC_ERR_INVALID_ARG),
    ]:
        assert f(ctypes.byref(bad), p, p, p, p, 0.1, p, p, big, None, None) == want
    assert f(None, p, p, p, p, 0.1, p, p, big, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), None, p, p, p, 0.1, p, p, big, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), ctypes.c_void_p(FAKE + 8), p, p, p, 0.1, p, p, big, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), p, p, p, p, 0.1, p, p, 64, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), p, p, p, p, float("nan"), p, p, big, None, None) == capi.EC_ERR_INVALID_ARG


def test_dense_attention_rejects_bad_args(capi):
    lib = capi.load()
    f = lib.ec_dense_attention
    p = ctypes.c_void_p(FAKE)
    good = _params(capi, D=128)
    for bad, want in [
        (_params(capi, D=128, Hkv=5), capi.EC_ERR_INVALID_ARG),  # Hq % Hkv
        (_params(capi, D=64), capi.EC_ERR_UNSUPPORTED),  # the dense kernel is built for D = 128
        (_params(capi, D=96), capi.EC_ERR_UNSUPPORTED),
        (_params(capi, D=128, B=0), capi.EC_ERR_INVALID_ARG),
        (_params(capi, D=128, L=0), capi.EC_ERR_INVALID_ARG),
    ]:
        assert f(ctypes.byref(bad), p, p, p, 0.1, p, None, None) == want
    assert f(None, p, p, p, 0.1, p, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), None, p, p, 0.1, p, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), p, p, p, 0.1, None, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), p, ctypes.c_void_p(FAKE + 8), p, 0.1, p, None, None) == capi.EC_ERR_INVALID_ARG
    assert f(ctypes.byref(good), p, p, p, float("nan"), p, None, None) == capi.EC_ERR_INVALID_ARG


def test_select_and_scatter_reject_bad_args(capi):
    lib = capi.load()
    p = ctypes.c_void_p(FAKE)
    st = capi.EcState(*([p] * 11))
    INV = capi.EC_ERR_INVALID_ARG
    for bad in [dict(k=0), dict(k=2000), dict(n_dec=0), dict(n_dec=33), dict(C_max=0), dict(C_max=2048),
                dict(tau=float("nan"))]:
        pp = _params(capi, **bad)
        assert lib.ec_select_recompute(ctypes.byref(pp), ctypes.byref(st), p, p, p, p, p, None) == INV, bad
    good = _params(capi)
    st_missing = capi.EcState(*([p] * 10 + [None]))  # dev_err may be NULL ...
    st_bad = capi.EcState(*([None] + [p] * 10))  # ... tokens may not
    assert lib.ec_select_recompute(ctypes.byref(good), ctypes.byref(st_bad), p, p, p, p, p, None) == INV
    assert lib.ec_select_recompute(ctypes.byref(good), None, p, p, p, p, p, None) == INV
    assert lib.ec_select_recompute(ctypes.byref(good), ctypes.byref(st_missing), None, p, p, p, p, None) == INV
    sc = lib.ec_kv_scatter
    assert sc(ctypes.byref(_params(capi, D=80)), p, p, p, p, 0, p, p, None, None) == capi.EC_ERR_UNSUPPORTED
    assert sc(ctypes.byref(good), p, p, p, p, 2, p, p, None, None) == INV
    assert sc(ctypes.byref(good), p, ctypes.c_void_p(FAKE + 2), p, p, 0, p, p, None, None) == INV
    assert sc(ctypes.byref(good), p, p, p, p, 0, None, p, None, None) == INV


GIB = 1 << 30  # fake buffers this far apart never overlap at the shapes used here


def test_step_rejects_bad_args(capi):
    lib = capi.load()
    p = ctypes.c_void_p(FAKE)
    st = capi.EcState(*([p] * 11))
    # k_cache, v_cache, k_src, v_src, q_src, out: six distinct buffers
    arrs = [(ctypes.c_void_p * 1)(FAKE + (i + 1) * GIB) for i in range(6)]
    good = _params(capi)
    big = 1 << 34
    f = lib.ec_step
    args = lambda pp, n=1, ws=p, wsb=big: (ctypes.byref(pp), ctypes.byref(st), p, p, p, n, *arrs,  # noqa: E731
                                           0.088, ws, wsb, None)
    assert f(*args(_params(capi, V=50257))) == capi.EC_ERR_INVALID_ARG  # V*2 % 16 for the packed logits
    assert f(*args(good, n=-1)) == capi.EC_ERR_INVALID_ARG
    assert f(*args(good, wsb=1024)) == capi.EC_ERR_INVALID_ARG
    assert f(*args(good, ws=None)) == capi.EC_ERR_INVALID_ARG
    null_arr = (ctypes.c_void_p * 1)(0)
    a = list(args(good))
    a[6] = null_arr
    assert f(*a) == capi.EC_ERR_INVALID_ARG


def test_overlapping_buffers_are_rejected(capi):
    # a buffer that is written while another is read must not share bytes with it: out against
    # the queries and caches of the attention, the caches against each other and against the
    # fresh rows of the scatter (8 MB queries and outputs, 8 MB caches at these shapes)
    lib = capi.load()
    INV = capi.EC_ERR_INVALID_ARG
    good = _params(capi)
    big = 1 << 34
    buf = [ctypes.c_void_p(FAKE + (i + 1) * GIB) for i in range(6)]
    ws = ctypes.c_void_p(FAKE)
    inside = lambda b: ctypes.c_void_p(b.value + (4 << 20))  # noqa: E731  (4 MB into a buffer)
    q, k, v, out = buf[0], buf[1], buf[2], buf[3]
    for o in (q, k, v, inside(q), inside(k)):
        assert lib.ec_partial_attention(ctypes.byref(good), q, k, v, ws, 0.088, o, ws, big, None, None) == INV
        assert lib.ec_dense_attention(ctypes.byref(good), q, k, v, 0.088, o, None, None) == INV
    # the scatter: caches against each other and against the fresh rows
    kc, vc, kn, vn = buf[0], buf[1], buf[2], buf[3]
    for args in [(kc, kc, kn, vn), (kc, inside(kc), kn, vn), (kc, vc, kc, vn), (kc, vc, kn, inside(vc))]:
        assert lib.ec_kv_scatter(ctypes.byref(good), *args, 1, ws, ws, None, None) == INV
    # the step checks every layer
    st = capi.EcState(*([ws] * 11))
    arrs = [(ctypes.c_void_p * 1)(b.value) for b in buf]  # k_cache, v_cache, k_src, v_src, q_src, out
    for i, j in [(5, 4), (5, 0), (2, 0), (1, 0)]:  # out = q_src, out = k_cache, k_src = k_cache, v_cache = k_cache
        a = list(arrs)
        a[i] = arrs[j]
        assert lib.ec_step(ctypes.byref(good), ctypes.byref(st), ws, ws, ws, 1, *a, 0.088, ws, big, None) == INV


def test_read_device_error_rejects_null(capi):
    lib = capi.load()
    assert lib.ec_read_device_error(None, None, None) == capi.EC_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(capi):
    import torch

    import entropy_gated_kv_gb300 as E

    with pytest.raises(ValueError):
        E.entropy_decode(torch.zeros(2, 64))


def test_lm_head_entropy_validation(capi):
    lib = capi.load()
    INV = capi.EC_ERR_INVALID_ARG
    assert lib.ec_lm_head_entropy_workspace_size(0) == 0
    assert lib.ec_lm_head_entropy_workspace_size(257) == 0
    assert lib.ec_lm_head_entropy_workspace_size(32) >= 32 * 16
    p = 1 << 20  # never dereferenced: every call below fails validation first
    ws = lib.ec_lm_head_entropy_workspace_size(32)
    ok = dict(hidden=p, weight=p, n_rows=32, d_model=4096, V=126464, ids=p, ent=p, conf=p, ws=p, ws_bytes=ws)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.ec_lm_head_entropy(a["hidden"], a["weight"], a["n_rows"], a["d_model"], a["V"], a["ids"],
                                      a["ent"], a["conf"], a["ws"], a["ws_bytes"], None)

    assert call(n_rows=0) == INV
    assert call(n_rows=257) == INV
    assert call(d_model=100) == INV  # not a multiple of 64
    assert call(d_model=0) == INV
    assert call(V=0) == INV
    assert call(hidden=None) == INV
    assert call(weight=p + 8) == INV  # not 16-byte aligned
    assert call(ws_bytes=ws - 1) == INV


def test_selftest_bounded_wait_validation(capi):
    lib = capi.load()
    INV = capi.EC_ERR_INVALID_ARG
    assert lib.ec_selftest_bounded_wait(None, 1000, None) == INV
    assert lib.ec_selftest_bounded_wait(1 << 20, 0, None) == INV
    assert lib.ec_selftest_bounded_wait(1 << 20, 10 ** 10 + 1, None) == INV


def test_conf_threshold_validation(capi):
    import math

    lib = capi.load()
    # the step's workspace query validates every parameter: 0 marks a rejected set
    for ok in (0.0, -1.0, 0.5, 1.0):
        p = _params(capi, conf_threshold=ok)
        assert lib.ec_step_workspace_size(ctypes.byref(p)) > 0, ok
    for bad in (math.nan, 1.5):
        p = _params(capi, conf_threshold=bad)
        assert lib.ec_step_workspace_size(ctypes.byref(p)) == 0, bad


def test_scope_validation(capi):
    lib = capi.load()
    # both 0: the whole sequence; otherwise 0 <= lo < hi <= L
    for lo, hi in ((0, 0), (0, 1024), (992, 1024), (0, 32), (5, 6)):
        p = _params(capi, scope_lo=lo, scope_hi=hi)
        assert lib.ec_step_workspace_size(ctypes.byref(p)) > 0, (lo, hi)
    for lo, hi in ((-1, 32), (32, 32), (40, 32), (0, 1025), (1024, 1025), (7, 0)):
        p = _params(capi, scope_lo=lo, scope_hi=hi)
        assert lib.ec_step_workspace_size(ctypes.byref(p)) == 0, (lo, hi)


def test_candidates_validation(capi):
    lib = capi.load()
    INV = capi.EC_ERR_INVALID_ARG
    p = _params(capi)
    st = capi.EcState(*([1 << 20] * 11))  # never dereferenced: validation fails first
    buf = ctypes.c_void_p(1 << 20)
    assert lib.ec_candidates(ctypes.byref(p), ctypes.byref(st), 2, 0, 32, buf, buf, None) == INV  # bad mode
    assert lib.ec_candidates(ctypes.byref(p), ctypes.byref(st), 0, -1, 32, buf, buf, None) == INV  # start < 0
    assert lib.ec_candidates(ctypes.byref(p), ctypes.byref(st), 0, 1024, 32, buf, buf, None) == INV  # start >= L
    assert lib.ec_candidates(ctypes.byref(p), ctypes.byref(st), 1, 0, 0, buf, buf, None) == INV  # width < 1
    assert lib.ec_candidates(ctypes.byref(p), ctypes.byref(st), 1, 0, 33, buf, buf, None) == INV  # width > C_max
    assert lib.ec_candidates(ctypes.byref(p), None, 0, 0, 32, buf, buf, None) == INV
    assert lib.ec_candidates(ctypes.byref(p), ctypes.byref(st), 0, 0, 32, None, buf, None) == INV
    bad = _params(capi, scope_lo=3, scope_hi=2)
    assert lib.ec_candidates(ctypes.byref(bad), ctypes.byref(st), 0, 0, 32, buf, buf, None) == INV


def test_read_floor_validation(capi):
    lib = capi.load()
    INV = capi.EC_ERR_INVALID_ARG
    buf = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    assert lib.ec_read_floor(None, 1024, buf, None) == INV
    assert lib.ec_read_floor(buf, 1024, None, None) == INV
    assert lib.ec_read_floor(ctypes.c_void_p((1 << 20) + 8), 1024, buf, None) == INV  # misaligned
    assert lib.ec_read_floor(buf, 1000, buf, None) == INV  # not a multiple of 16 bytes


def test_missing_library_fails_loudly(capi, tmp_path):
    # no fallback: loading a library that is not there raises
    with pytest.raises(ImportError, match="no CPU fallback"):
        capi.load(tmp_path / "libentropycache.so")


def test_product_path_never_touches_the_oracle():
    # the package and the input generators import nothing from oracle/, and the oracle nothing
    # from the package (checked on the sources and in a fresh interpreter)
    import subprocess
    import sys

    pat = re.compile(r"^\s*(import\s+oracle\b|from\s+oracle\b)", re.M)
    for d in ("entropy_gated_kv_gb300", "workloads"):
        for f in (ROOT / d).rglob("*.py"):
            assert not pat.search(f.read_text()), f"{f} imports the oracle"
    pkg = re.compile(r"^\s*(import|from)\s+entropy_gated_kv_gb300\b", re.M)
    for f in (ROOT / "oracle").rglob("*.py"):
        assert not pkg.search(f.read_text()), f"{f} imports the CUDA package"
    code = "import sys, entropy_gated_kv_gb300, workloads; sys.exit(1 if 'oracle' in sys.modules else 0)"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
