"""Python binding of libqlinear.so (argument marshalling only).

Every function here has the name of the C entry point it calls (include/qlinear.h)
and does nothing but check tensor placement, allocate outputs with PyTorch and pass
device pointers and the current CUDA stream.  All arithmetic runs in the library's
sm_103a kernels; if the library is missing this module raises on import - there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqlinear.so")

QL_OK = 0
QL_ERR_NULL = -1
QL_ERR_SHAPE = -2
QL_ERR_BITS = -3
QL_ERR_GROUP = -4
QL_ERR_ROWS = -5
QL_ERR_ALIGN = -6
QL_ERR_ARCH = -7
QL_ERR_LAUNCH = -8
QL_ERR_TIMEOUT = -9
QL_ERR_CUDA = -10
QL_ERR_NOMEM = -11
QL_ERR_TOO_LARGE = -12


class QlinearError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({qlinear_strerror(code)})")


class ql_weight(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("n", ctypes.c_int32), ("k", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("group", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m weight_only_bit_mlx_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, U64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    W = ctypes.POINTER(ql_weight)
    sig = {
        "qlinear_mv": (ctypes.c_int, [W, P, P, P]),
        "qlinear_mv_rows": (ctypes.c_int, [W, P, I32, I64, P, I64, P]),
        "qffn_swiglu_mv": (ctypes.c_int, [W, W, P, I32, I64, P, I64, P]),
        "qattn_proj_mv": (ctypes.c_int, [W, W, W, W, P, I32, I64, P, P, P, P, P]),
        "qlinear_pgemm": (ctypes.c_int, [W, P, I32, I64, P, I64, P]),
        "qlinear_pgemm_noalloc": (ctypes.c_int, [W, P, I32, I64, P, I64, P]),
        "qlinear_pgemm_multi": (ctypes.c_int, [ctypes.POINTER(W), I32, P, I32, I64, ctypes.POINTER(P),
                                               ctypes.POINTER(I64), P]),
        "qlinear_pgemm_swiglu": (ctypes.c_int, [W, P, I32, I64, P, I64, P, I64, P]),
        "qlinear_pgemm_resid_norm": (ctypes.c_int, [W, P, I32, I64, P, I64, P, ctypes.c_float, P, I64, P]),
        "qswiglu": (ctypes.c_int, [P, P, I32, I32, I64, P, I64, P]),
        "qattn_qknorm_rope_kv": (ctypes.c_int, [P, I64, P, I64, P, I64, I32, I32, I32, I32, I32, ctypes.c_float,
                                                ctypes.c_float, P, P, P, P, I64, P, P, I32, P]),
        "qresid_rmsnorm": (ctypes.c_int, [P, I64, P, I64, I32, I32, P, ctypes.c_float, P, I64, P]),
        "qlinear_mv_resid_norm": (ctypes.c_int, [W, P, I32, I64, P, I64, P, ctypes.c_float, P, I64, P]),
        "qlinear_last_error": (ctypes.c_int, [P]),
        "qlinear_set_wait_budget_ns": (U64, [U64]),
        "qlinear_wait_probe": (ctypes.c_int, [U64, P]),
        "qlinear_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "qlinear_version": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()


# ----------------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------------
class QWeight:
    """A quantized weight on the device, as stored.

    ``wq``: int32 tensor [n, k*bits/32] (the uint32 words' bits); ``scales`` and
    ``biases``: bfloat16 tensors [n, k/64].
    """

    def __init__(self, wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, k: int, bits: int,
                 group: int = 64):
        self.wq, self.scales, self.biases = wq, scales, biases
        self.n, self.k, self.bits, self.group = int(wq.shape[0]), int(k), int(bits), int(group)
        for t in (wq, scales, biases):
            if not t.is_contiguous():
                raise ValueError("weight tensors must be contiguous")
        self.c = ql_weight(wq.data_ptr(), scales.data_ptr(), biases.data_ptr(), self.n, self.k, self.bits,
                           self.group)

    @classmethod
    def from_numpy(cls, d: dict, device="cuda") -> "QWeight":
        """From a dict with uint32 ``wq``, uint16 (bf16 bits) ``scales``/``biases``, ``k``, ``bits``."""
        wq = torch.from_numpy(np.ascontiguousarray(d["wq"]).view(np.int32)).to(device)
        sc = torch.from_numpy(np.ascontiguousarray(d["scales"]).view(np.int16)).to(device).view(torch.bfloat16)
        bi = torch.from_numpy(np.ascontiguousarray(d["biases"]).view(np.int16)).to(device).view(torch.bfloat16)
        return cls(wq, sc, bi, d["k"], d["bits"])

    def rows(self, lo: int, hi: int) -> "QWeight":
        """Rows lo..hi-1 of the weight (views, no copy)."""
        return QWeight(self.wq[lo:hi], self.scales[lo:hi], self.biases[lo:hi], self.k, self.bits, self.group)


def bf16_from_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    """A bfloat16 device tensor with the given uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bfloat16 tensor (copied to the host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int, where: str):
    if code != QL_OK:
        raise QlinearError(code, where)


def _act(x: torch.Tensor, k: int) -> tuple[torch.Tensor, int, int]:
    if x.dtype != torch.bfloat16 or not x.is_cuda:
        raise ValueError("activations must be a CUDA bfloat16 tensor")
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.shape[1] != k or x.stride(1) != 1:
        raise ValueError(f"activations must be [rows, {k}] with unit column stride")
    return x, int(x.shape[0]), int(x.stride(0))


# ----------------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------------
def qlinear_mv(w: QWeight, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    x, rows, _ = _act(x, w.k)
    if rows != 1:
        raise ValueError("qlinear_mv takes one activation row")
    if y is None:
        y = torch.empty(w.n, dtype=torch.float32, device=x.device)
    _check(LIB.qlinear_mv(ctypes.byref(w.c), x.data_ptr(), y.data_ptr(), _stream(stream)), "qlinear_mv")
    return y


def qlinear_mv_rows(w: QWeight, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    x, rows, ldx = _act(x, w.k)
    if y is None:
        y = torch.empty(rows, w.n, dtype=torch.float32, device=x.device)
    _check(LIB.qlinear_mv_rows(ctypes.byref(w.c), x.data_ptr(), rows, ldx, y.data_ptr(), y.stride(0),
                               _stream(stream)), "qlinear_mv_rows")
    return y


def qffn_swiglu_mv(w1: QWeight, w3: QWeight, x: torch.Tensor, h: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    x, rows, ldx = _act(x, w1.k)
    if h is None:
        h = torch.empty(rows, w1.n, dtype=torch.bfloat16, device=x.device)
    _check(LIB.qffn_swiglu_mv(ctypes.byref(w1.c), ctypes.byref(w3.c), x.data_ptr(), rows, ldx, h.data_ptr(),
                              h.stride(0), _stream(stream)), "qffn_swiglu_mv")
    return h


def qattn_proj_mv(wq: QWeight, wk: QWeight, wv: QWeight, wg: QWeight, x: torch.Tensor, outs=None,
                  stream=None):
    x, rows, ldx = _act(x, wq.k)
    if outs is None:
        outs = [torch.empty(rows, w.n, dtype=torch.float32, device=x.device) for w in (wq, wk, wv, wg)]
    q, k, v, g = outs
    _check(LIB.qattn_proj_mv(ctypes.byref(wq.c), ctypes.byref(wk.c), ctypes.byref(wv.c), ctypes.byref(wg.c),
                             x.data_ptr(), rows, ldx, q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                             _stream(stream)), "qattn_proj_mv")
    return q, k, v, g


def qlinear_pgemm(w: QWeight, X: torch.Tensor, Y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if X.dtype != torch.bfloat16 or not X.is_cuda or X.dim() != 2 or X.shape[1] != w.k or X.stride(1) != 1:
        raise ValueError(f"X must be a CUDA bfloat16 [m, {w.k}] tensor with unit column stride")
    m = int(X.shape[0])
    if Y is None:
        Y = torch.empty(m, w.n, dtype=torch.float32, device=X.device)
    _check(LIB.qlinear_pgemm(ctypes.byref(w.c), X.data_ptr(), m, X.stride(0), Y.data_ptr(), Y.stride(0),
                             _stream(stream)), "qlinear_pgemm")
    return Y


def qlinear_pgemm_multi(ws, X: torch.Tensor, Ys=None, stream=None) -> list:
    """qlinear_pgemm for several weights that read the same X (the split row sums of X are
    formed once); returns the outputs, each bit-equal to its own qlinear_pgemm call."""
    ws = list(ws)
    if not ws:
        raise ValueError("at least one weight")
    k = ws[0].k
    if X.dtype != torch.bfloat16 or not X.is_cuda or X.dim() != 2 or X.shape[1] != k or X.stride(1) != 1:
        raise ValueError(f"X must be a CUDA bfloat16 [m, {k}] tensor with unit column stride")
    m = int(X.shape[0])
    if Ys is None:
        Ys = [torch.empty(m, w.n, dtype=torch.float32, device=X.device) for w in ws]
    if len(Ys) != len(ws):
        raise ValueError("one output per weight")
    nw = len(ws)
    wp = (ctypes.POINTER(ql_weight) * nw)(*[ctypes.pointer(w.c) for w in ws])
    yp = (ctypes.c_void_p * nw)(*[Y.data_ptr() for Y in Ys])
    ld = (ctypes.c_int64 * nw)(*[Y.stride(0) for Y in Ys])
    _check(LIB.qlinear_pgemm_multi(wp, nw, X.data_ptr(), m, X.stride(0), yp, ld, _stream(stream)),
           "qlinear_pgemm_multi")
    return Ys


def qlinear_pgemm_noalloc(w: QWeight, X: torch.Tensor, Y: torch.Tensor, stream=None) -> torch.Tensor:
    """qlinear_pgemm with the library's fixed static scratch: the library allocates
    nothing, so the caller passes the output buffer too."""
    if X.dtype != torch.bfloat16 or not X.is_cuda or X.dim() != 2 or X.shape[1] != w.k or X.stride(1) != 1:
        raise ValueError(f"X must be a CUDA bfloat16 [m, {w.k}] tensor with unit column stride")
    _check(LIB.qlinear_pgemm_noalloc(ctypes.byref(w.c), X.data_ptr(), int(X.shape[0]), X.stride(0), Y.data_ptr(),
                                     Y.stride(0), _stream(stream)), "qlinear_pgemm_noalloc")
    return Y


def _prompt(X: torch.Tensor, k: int) -> int:
    if X.dtype != torch.bfloat16 or not X.is_cuda or X.dim() != 2 or X.shape[1] != k or X.stride(1) != 1:
        raise ValueError(f"X must be a CUDA bfloat16 [m, {k}] tensor with unit column stride")
    return int(X.shape[0])


def qlinear_pgemm_swiglu(w3: QWeight, X: torch.Tensor, A: torch.Tensor, H: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """H = bf16(silu(A) * (X w3^T)): the up-projection prompt GEMM with the SwiGLU as its
    epilogue.  A: float32 [m, n] (the gate projection's output)."""
    m = _prompt(X, w3.k)
    A = _rows2d(A, torch.float32, "A")
    if tuple(A.shape) != (m, w3.n):
        raise ValueError("A must be [m, n]")
    if H is None:
        H = torch.empty(m, w3.n, dtype=torch.bfloat16, device=X.device)
    _check(LIB.qlinear_pgemm_swiglu(ctypes.byref(w3.c), X.data_ptr(), m, X.stride(0), A.data_ptr(), A.stride(0),
                                    H.data_ptr(), H.stride(0), _stream(stream)), "qlinear_pgemm_swiglu")
    return H


def qlinear_pgemm_resid_norm(w: QWeight, X: torch.Tensor, resid: torch.Tensor, gamma: torch.Tensor, eps: float,
                             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """resid <- bf16(resid + X w^T) in the prompt GEMM's epilogue; returns
    out = bf16(rmsnorm(resid) * gamma).  resid: bfloat16 [m, n]; gamma: bfloat16 [n]."""
    m = _prompt(X, w.k)
    r = _rows2d(resid, torch.bfloat16, "resid")
    if tuple(r.shape) != (m, w.n) or gamma.dtype != torch.bfloat16 or gamma.numel() != w.n or \
            not gamma.is_contiguous():
        raise ValueError("resid must be [m, n] and gamma a contiguous bfloat16 [n]")
    if out is None:
        out = torch.empty(m, w.n, dtype=torch.bfloat16, device=X.device)
    _check(LIB.qlinear_pgemm_resid_norm(ctypes.byref(w.c), X.data_ptr(), m, X.stride(0), r.data_ptr(), r.stride(0),
                                        gamma.data_ptr(), float(eps), out.data_ptr(), out.stride(0),
                                        _stream(stream)), "qlinear_pgemm_resid_norm")
    return out


def qswiglu(a: torch.Tensor, c: torch.Tensor, h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if a.shape != c.shape or a.dtype != torch.float32 or c.dtype != torch.float32 or a.stride() != c.stride():
        raise ValueError("a and c must be float32 tensors of one shape and layout")
    a2 = a.view(1, -1) if a.dim() == 1 else a
    c2 = c.view(1, -1) if c.dim() == 1 else c
    rows, n = int(a2.shape[0]), int(a2.shape[1])
    if h is None:
        h = torch.empty(rows, n, dtype=torch.bfloat16, device=a.device)
    _check(LIB.qswiglu(a2.data_ptr(), c2.data_ptr(), rows, n, a2.stride(0), h.data_ptr(), h.stride(0),
                       _stream(stream)), "qswiglu")
    return h


def _rows2d(t: torch.Tensor, dtype, what: str) -> torch.Tensor:
    if t.dtype != dtype or not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA {dtype} tensor")
    t = t.view(1, -1) if t.dim() == 1 else t
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{what} must be [rows, n] with unit column stride")
    return t


def qattn_qknorm_rope_kv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_q_heads: int, n_kv_heads: int,
                         head_dim: int, rot_dim: int, rope_base: float, eps: float, q_norm_w: torch.Tensor,
                         k_norm_w: torch.Tensor, pos: torch.Tensor, k_ring: torch.Tensor, v_ring: torch.Tensor,
                         q_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """QK norm + partial RoPE of q and k, k/v into slot pos % ring_len of each stream's
    rings.  q, k, v: float32 [rows, *]; q_norm_w, k_norm_w: bfloat16 [head_dim];
    pos: int32 [rows]; k_ring, v_ring: bfloat16 [rows, ring_len, n_kv_heads*head_dim]
    (contiguous).  Returns q_out (bfloat16 [rows, n_q_heads*head_dim])."""
    q, k, v = (_rows2d(t, torch.float32, nm) for t, nm in ((q, "q"), (k, "k"), (v, "v")))
    rows = int(q.shape[0])
    if k.shape[0] != rows or v.shape[0] != rows or pos.numel() != rows or pos.dtype != torch.int32:
        raise ValueError("q, k, v and pos must have one row / entry per stream (pos int32)")
    for t, nm in ((q_norm_w, "q_norm_w"), (k_norm_w, "k_norm_w")):
        if t.dtype != torch.bfloat16 or t.numel() != head_dim or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous bfloat16 [head_dim] tensor")
    width = n_kv_heads * head_dim
    for t, nm in ((k_ring, "k_ring"), (v_ring, "v_ring")):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or t.shape[0] != rows or t.shape[2] != width or \
                not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous bfloat16 [rows, ring_len, {width}] tensor")
    if k_ring.shape != v_ring.shape:
        raise ValueError("k_ring and v_ring must have one shape")
    if q_out is None:
        q_out = torch.empty(rows, n_q_heads * head_dim, dtype=torch.bfloat16, device=q.device)
    _check(LIB.qattn_qknorm_rope_kv(q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0), v.data_ptr(), v.stride(0),
                                    rows, n_q_heads, n_kv_heads, head_dim, rot_dim, float(rope_base), float(eps),
                                    q_norm_w.data_ptr(), k_norm_w.data_ptr(), pos.data_ptr(), q_out.data_ptr(),
                                    q_out.stride(0), k_ring.data_ptr(), v_ring.data_ptr(), int(k_ring.shape[1]),
                                    _stream(stream)), "qattn_qknorm_rope_kv")
    return q_out


def qresid_rmsnorm(y: torch.Tensor, resid: torch.Tensor, gamma: torch.Tensor, eps: float,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """resid <- bf16(resid + y) in place; returns out = bf16(rmsnorm(resid) * gamma).
    y: float32 [rows, n]; resid: bfloat16 [rows, n]; gamma: bfloat16 [n]."""
    y = _rows2d(y, torch.float32, "y")
    r = _rows2d(resid, torch.bfloat16, "resid")
    rows, n = int(y.shape[0]), int(y.shape[1])
    if tuple(r.shape) != (rows, n) or gamma.dtype != torch.bfloat16 or gamma.numel() != n or \
            not gamma.is_contiguous():
        raise ValueError("resid must be [rows, n] like y and gamma a contiguous bfloat16 [n]")
    if out is None:
        out = torch.empty(rows, n, dtype=torch.bfloat16, device=y.device)
    _check(LIB.qresid_rmsnorm(y.data_ptr(), y.stride(0), r.data_ptr(), r.stride(0), rows, n, gamma.data_ptr(),
                              float(eps), out.data_ptr(), out.stride(0), _stream(stream)), "qresid_rmsnorm")
    return out


def qlinear_mv_resid_norm(w: QWeight, x: torch.Tensor, resid: torch.Tensor, gamma: torch.Tensor, eps: float,
                          out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = W x; resid <- bf16(resid + y) in place; returns out = bf16(rmsnorm(resid) * gamma),
    in one launch.  x: bfloat16 [rows, k]; resid: bfloat16 [rows, n]; gamma: bfloat16 [n]."""
    x, rows, ldx = _act(x, w.k)
    r = _rows2d(resid, torch.bfloat16, "resid")
    if tuple(r.shape) != (rows, w.n) or gamma.dtype != torch.bfloat16 or gamma.numel() != w.n or \
            not gamma.is_contiguous():
        raise ValueError("resid must be [rows, n] and gamma a contiguous bfloat16 [n]")
    if out is None:
        out = torch.empty(rows, w.n, dtype=torch.bfloat16, device=x.device)
    _check(LIB.qlinear_mv_resid_norm(ctypes.byref(w.c), x.data_ptr(), rows, ldx, r.data_ptr(), r.stride(0),
                                     gamma.data_ptr(), float(eps), out.data_ptr(), out.stride(0), _stream(stream)),
           "qlinear_mv_resid_norm")
    return out


def qlinear_last_error(stream=None) -> int:
    return int(LIB.qlinear_last_error(_stream(stream)))


def qlinear_set_wait_budget_ns(ns: int) -> int:
    return int(LIB.qlinear_set_wait_budget_ns(int(ns)))


def qlinear_wait_probe(budget_ns: int, stream=None):
    _check(LIB.qlinear_wait_probe(int(budget_ns), _stream(stream)), "qlinear_wait_probe")


def qlinear_strerror(code: int) -> str:
    return LIB.qlinear_strerror(int(code)).decode()


def qlinear_version() -> int:
    return int(LIB.qlinear_version())
