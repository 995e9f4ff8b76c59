"""Host-side checks of libqlinear.so that need no GPU: the library builds, loads,
exports every entry point that include/qlinear.h declares, and rejects bad
arguments before touching the device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlinear.h")


@pytest.fixture(scope="module")
def q():
    from weight_only_bit_mlx_gb300 import build
    build.build_library()
    from weight_only_bit_mlx_gb300 import qlinear
    return qlinear


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(q\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_paths():
    names = declared_functions()
    for f in ("qlinear_mv", "qlinear_mv_rows", "qffn_swiglu_mv", "qattn_proj_mv", "qlinear_pgemm"):
        assert f in names


def test_library_exports_every_declared_symbol(q):
    lib = ctypes.CDLL(q.LIB_PATH)
    out = subprocess.run(["nm", "-D", "--defined-only", q.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s+(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in exported, name


def test_strerror_and_version(q):
    assert q.qlinear_strerror(0) == "ok"
    assert "wait" in q.qlinear_strerror(q.QL_ERR_TIMEOUT)
    assert q.qlinear_strerror(12345).startswith("unknown")
    assert q.qlinear_version() >= 1


def _w(q, **kw):
    d = dict(wq=0x10000, scales=0x20000, biases=0x30000, n=64, k=128, bits=4, group=64)
    d.update(kw)
    return q.ql_weight(d["wq"], d["scales"], d["biases"], d["n"], d["k"], d["bits"], d["group"])


@pytest.mark.parametrize("kw,code", [
    (dict(wq=0), "QL_ERR_NULL"),
    (dict(group=32), "QL_ERR_GROUP"),
    (dict(bits=5), "QL_ERR_BITS"),
    (dict(bits=2), "QL_ERR_BITS"),
    (dict(k=96), "QL_ERR_SHAPE"),
    (dict(k=0), "QL_ERR_SHAPE"),
    (dict(n=0), "QL_ERR_SHAPE"),
    (dict(wq=0x10004), "QL_ERR_ALIGN"),
])
def test_bad_weight_rejected_on_host(q, kw, code):
    w = _w(q, **kw)
    x, y = 0x40000, 0x50000
    assert q.LIB.qlinear_mv_rows(ctypes.byref(w), x, 1, 128, y, 64, None) == getattr(q, code)
    assert q.LIB.qlinear_pgemm(ctypes.byref(w), x, 8, 128, y, 64, None) == getattr(q, code)


def test_bad_rows_and_layout_rejected_on_host(q):
    w = _w(q)
    L = q.LIB
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40000, 0, 128, 0x50000, 64, None) == q.QL_ERR_ROWS
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40000, 17, 128, 0x50000, 64, None) == q.QL_ERR_ROWS
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40008, 2, 128, 0x50000, 64, None) == q.QL_ERR_ALIGN
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40000, 2, 124, 0x50000, 64, None) == q.QL_ERR_ALIGN
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40000, 2, 64, 0x50000, 64, None) == q.QL_ERR_ALIGN
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40000, 2, 128, 0x50000, 32, None) == q.QL_ERR_ALIGN
    assert L.qlinear_mv_rows(ctypes.byref(w), 0, 1, 128, 0x50000, 64, None) == q.QL_ERR_NULL
    assert L.qlinear_mv_rows(ctypes.byref(w), 0x40000, 1, 128, 0, 64, None) == q.QL_ERR_NULL
    assert L.qlinear_pgemm(ctypes.byref(w), 0x40000, -1, 128, 0x50000, 64, None) == q.QL_ERR_SHAPE
    assert L.qlinear_pgemm(ctypes.byref(w), 0x40000, 4, 120, 0x50000, 64, None) == q.QL_ERR_ALIGN
    w3 = _w(q, n=32)
    assert L.qffn_swiglu_mv(ctypes.byref(w), ctypes.byref(w3), 0x40000, 1, 128, 0x50000, 64,
                            None) == q.QL_ERR_SHAPE
    w6 = _w(q, bits=6)
    assert L.qffn_swiglu_mv(ctypes.byref(w), ctypes.byref(w6), 0x40000, 1, 128, 0x50000, 64,
                            None) == q.QL_ERR_BITS
    wk = _w(q, k=256)
    assert L.qattn_proj_mv(ctypes.byref(w), ctypes.byref(wk), ctypes.byref(w), ctypes.byref(w), 0x40000, 1,
                           128, 0x50000, 0x50000, 0x50000, 0x50000, None) == q.QL_ERR_SHAPE
    assert L.qswiglu(0x40000, 0x50000, 0, 8, 8, 0x60000, 8, None) == q.QL_ERR_SHAPE
    assert L.qswiglu(0, 0x50000, 1, 8, 8, 0x60000, 8, None) == q.QL_ERR_NULL


def test_wait_budget_setter(q):
    old = q.qlinear_set_wait_budget_ns(12345)
    assert q.qlinear_set_wait_budget_ns(old) == 12345


def test_post_ops_reject_bad_arguments_on_host(q):
    L = q.LIB
    P = 0x40000
    args = dict(q=P, ldq=2048, k=P, ldk=512, v=P, ldv=512, rows=1, nq=32, nkv=8, hd=64, rot=64, base=1e4, eps=1e-5,
                qw=P, kw=P, pos=P, qo=P, ldqo=2048, kr=P, vr=P, L=16)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.qattn_qknorm_rope_kv(a["q"], a["ldq"], a["k"], a["ldk"], a["v"], a["ldv"], a["rows"], a["nq"],
                                      a["nkv"], a["hd"], a["rot"], a["base"], a["eps"], a["qw"], a["kw"], a["pos"],
                                      a["qo"], a["ldqo"], a["kr"], a["vr"], a["L"], None)

    assert call(q=0) == q.QL_ERR_NULL
    assert call(pos=0) == q.QL_ERR_NULL
    assert call(rows=0) == q.QL_ERR_ROWS
    assert call(rows=17) == q.QL_ERR_ROWS
    assert call(hd=48) == q.QL_ERR_SHAPE
    assert call(hd=288) == q.QL_ERR_SHAPE
    assert call(rot=66) == q.QL_ERR_SHAPE
    assert call(rot=63) == q.QL_ERR_SHAPE
    assert call(L=0) == q.QL_ERR_SHAPE
    assert call(base=0.0) == q.QL_ERR_SHAPE
    assert call(eps=-1.0) == q.QL_ERR_SHAPE
    assert call(ldq=2047) == q.QL_ERR_ALIGN
    assert call(ldqo=100) == q.QL_ERR_ALIGN
    assert call(k=P + 2) == q.QL_ERR_ALIGN
    assert L.qresid_rmsnorm(0, 8, P, 8, 1, 8, P, 1e-5, P, 8, None) == q.QL_ERR_NULL
    assert L.qresid_rmsnorm(P, 8, P, 8, 0, 8, P, 1e-5, P, 8, None) == q.QL_ERR_ROWS
    assert L.qresid_rmsnorm(P, 8, P, 8, 1, 0, P, 1e-5, P, 8, None) == q.QL_ERR_SHAPE
    assert L.qresid_rmsnorm(P, 8, P, 8, 1, 8, P, -1.0, P, 8, None) == q.QL_ERR_SHAPE
    assert L.qresid_rmsnorm(P, 7, P, 8, 1, 8, P, 1e-5, P, 8, None) == q.QL_ERR_ALIGN
    assert L.qresid_rmsnorm(P + 1, 8, P, 8, 1, 8, P, 1e-5, P, 8, None) == q.QL_ERR_ALIGN


def test_fused_resid_norm_rejects_bad_arguments_on_host(q):
    w = _w(q)
    L = q.LIB
    P = 0x40000
    assert L.qlinear_mv_resid_norm(ctypes.byref(w), P, 1, 128, 0, 64, P, 1e-5, P, 64, None) == q.QL_ERR_NULL
    assert L.qlinear_mv_resid_norm(ctypes.byref(w), P, 1, 128, P, 64, P, -1.0, P, 64, None) == q.QL_ERR_SHAPE
    assert L.qlinear_mv_resid_norm(ctypes.byref(w), P, 17, 128, P, 64, P, 1e-5, P, 64, None) == q.QL_ERR_ROWS
    assert L.qlinear_mv_resid_norm(ctypes.byref(w), P, 2, 128, P, 32, P, 1e-5, P, 64, None) == q.QL_ERR_ALIGN
    assert L.qlinear_mv_resid_norm(ctypes.byref(w), P + 8, 1, 128, P, 64, P, 1e-5, P, 64, None) == q.QL_ERR_ALIGN


def test_binding_fails_loudly_without_the_library(tmp_path):
    """A copy of the Python package with no libqlinear.so beside it must refuse to
    import: there is no CPU or eager fallback behind the binding."""
    import shutil
    import sys
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "weight_only_bit_mlx_gb300")
    dst = tmp_path / "weight_only_bit_mlx_gb300"
    dst.mkdir()
    for name in os.listdir(src):
        if name.endswith(".py"):
            shutil.copy(os.path.join(src, name), dst / name)
    assert not (dst / "libqlinear.so").exists()
    r = subprocess.run([sys.executable, "-c", "import weight_only_bit_mlx_gb300.qlinear"], cwd=tmp_path,
                       env={**os.environ, "PYTHONPATH": str(tmp_path)}, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "is not built" in r.stderr


def test_fused_prompt_gemm_epilogues_reject_bad_arguments_on_host(q):
    w = _w(q)
    L = q.LIB
    P = 0x40000
    sw = L.qlinear_pgemm_swiglu
    assert sw(ctypes.byref(w), P, 0, 128, 0, 64, 0, 64, None) == q.QL_OK  # an empty window enqueues nothing
    assert sw(ctypes.byref(w), P, -1, 128, P, 64, P, 64, None) == q.QL_ERR_SHAPE
    assert sw(ctypes.byref(w), P, 4, 128, 0, 64, P, 64, None) == q.QL_ERR_NULL
    assert sw(ctypes.byref(w), P, 4, 128, P, 64, 0, 64, None) == q.QL_ERR_NULL
    assert sw(ctypes.byref(w), P, 4, 128, P, 32, P, 64, None) == q.QL_ERR_ALIGN
    assert sw(ctypes.byref(w), P, 4, 128, P, 64, P + 1, 64, None) == q.QL_ERR_ALIGN
    assert sw(ctypes.byref(w), P + 8, 4, 128, P, 64, P, 64, None) == q.QL_ERR_ALIGN
    rn = L.qlinear_pgemm_resid_norm
    assert rn(ctypes.byref(w), P, 0, 128, 0, 64, 0, 1e-5, 0, 64, None) == q.QL_OK
    assert rn(ctypes.byref(w), P, 4, 128, 0, 64, P, 1e-5, P, 64, None) == q.QL_ERR_NULL
    assert rn(ctypes.byref(w), P, 4, 128, P, 64, P, -1.0, P, 64, None) == q.QL_ERR_SHAPE
    assert rn(ctypes.byref(w), P, 4, 128, P, 32, P, 1e-5, P, 64, None) == q.QL_ERR_ALIGN
    assert rn(ctypes.byref(w), P, 4, 120, P, 64, P, 1e-5, P, 64, None) == q.QL_ERR_ALIGN
    w5 = _w(q, bits=5)
    assert rn(ctypes.byref(w5), P, 4, 128, P, 64, P, 1e-5, P, 64, None) == q.QL_ERR_BITS


def test_pgemm_multi_rejects_bad_arguments_on_host(q):
    # qlinear_pgemm_multi: every weight checked as qlinear_pgemm checks it, the k equal,
    # 1 <= nw <= 16, outputs and their pitches checked per weight, all before the device
    L = q.LIB
    W = ctypes.POINTER(q.ql_weight)
    w, w2, wk, wbad = _w(q), _w(q, n=32), _w(q, k=256), _w(q, bits=5)

    def call(ws, nw, x=0x40000, m=8, ldx=128, ys=None, lds=None):
        wp = (W * max(1, len(ws)))(*[ctypes.pointer(v) for v in ws])
        n = max(1, len(ws))
        yp = (ctypes.c_void_p * n)(*(ys or [0x50000 + 0x10000 * i for i in range(n)]))
        ld = (ctypes.c_int64 * n)(*(lds or [64] * n))
        return L.qlinear_pgemm_multi(wp, nw, x, m, ldx, yp, ld, None)

    assert call([w, w2], 0) == q.QL_ERR_SHAPE
    assert call([w] * 16, 17) == q.QL_ERR_SHAPE
    assert call([w, wk], 2) == q.QL_ERR_SHAPE              # the k differ
    assert call([w, wbad], 2) == q.QL_ERR_BITS             # a bad weight
    assert call([w, w2], 2, m=-1) == q.QL_ERR_SHAPE
    assert call([w, w2], 2, m=0) == q.QL_OK               # an empty window: nothing enqueued
    assert call([w, w2], 2, x=0) == q.QL_ERR_NULL
    assert call([w, w2], 2, x=0x40008) == q.QL_ERR_ALIGN
    assert call([w, w2], 2, ldx=120) == q.QL_ERR_ALIGN
    assert call([w, w2], 2, ys=[0x50000, 0]) == q.QL_ERR_NULL
    assert call([w, w2], 2, lds=[64, 16]) == q.QL_ERR_ALIGN  # w2 has n = 32 > 16
    assert L.qlinear_pgemm_multi(None, 1, 0x40000, 8, 128, None, None, None) == q.QL_ERR_NULL
