"""ORACLE — test infrastructure, not product code.

ctypes wrapper around ``attn_oracle.c``, the plain fp64 CPU restatement of
multi-head scaled dot-product attention, of the post-norm MHA and feed-forward
sublayers and of the sinusoidal positional encoding.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
it; the CUDA path never imports it and shares no code with it.

All arrays passed in are fp64 (inputs already rounded to the kernel dtype and
widened back), laid out [B, n, h, d] for activations and [d_in, d_out] for
projection matrices.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

OK, EINVAL, EEMPTY, ENOMEM = 0, -1, -2, -3
MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: it runs on x86 and Arm hosts)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        u8p = ctypes.POINTER(ctypes.c_ubyte)
        c_int, c_double = ctypes.c_int, ctypes.c_double
        lib.oracle_softmax.argtypes = [dp, u8p, c_int, dp]
        lib.oracle_softmax.restype = c_int
        lib.oracle_attn.argtypes = [dp, dp, dp, dp] + [c_int] * 6 + [c_double, c_int, ip, c_int]
        lib.oracle_attn.restype = c_int
        lib.oracle_attn_rows.argtypes = ([dp, dp, dp] + [c_int] * 6 + [c_double, c_int, ip, ip,
                                                                        c_int, dp, dp, c_int])
        lib.oracle_attn_rows.restype = c_int
        lib.oracle_matmul.argtypes = [dp, dp, dp, c_int, c_int, c_int, c_int]
        lib.oracle_matmul.restype = None
        lib.oracle_layernorm_row.argtypes = [dp, dp, dp, c_double, c_int, dp]
        lib.oracle_layernorm_row.restype = None
        lib.oracle_mha.argtypes = ([dp] * 8 + [c_double, dp] + [c_int] * 8 + [ip, c_int]
                                   + [dp] * 4)
        lib.oracle_mha.restype = c_int
        lib.oracle_mha_rows.argtypes = ([dp] * 8 + [c_double] + [c_int] * 8 + [ip, ip, c_int, dp,
                                                                               c_int])
        lib.oracle_mha_rows.restype = c_int
        lib.oracle_pos_encoding.argtypes = [dp, dp, c_int, c_int, c_int, c_double, c_int]
        lib.oracle_pos_encoding.restype = c_int
        lib.oracle_ffn.argtypes = [dp] * 7 + [c_double, dp, c_int, c_int, c_int, c_int]
        lib.oracle_ffn.restype = c_int
        lib.oracle_attn_bwd.argtypes = [dp] * 4 + [c_int] * 6 + [c_double, c_int, ip] + [dp] * 4
        lib.oracle_attn_bwd.restype = c_int
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _dp(x: np.ndarray):
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what} returned {rc}")


def _keylens(key_lens, mask_kind):
    if key_lens is None:
        return None
    return np.ascontiguousarray(key_lens, dtype=np.int32)


def softmax(s, visible=None) -> np.ndarray:
    """Row softmax over the visible entries of a 1-D score vector."""
    lib = _load()
    s = _f64(s).ravel()
    w = np.empty_like(s)
    vis = None
    vis_p = None
    if visible is not None:
        vis = np.ascontiguousarray(visible, dtype=np.uint8).ravel()
        vis_p = vis.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))
    _check(lib.oracle_softmax(_dp(s), vis_p, s.size, _dp(w)), "oracle_softmax")
    return w


def attn(q, k, v, scale, mask_kind=MASK_NONE, key_lens=None, nthreads=0) -> np.ndarray:
    """Multi-head attention on [B, n, h, d] fp64 arrays -> [B, n_q, h, d_v]."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, n_q, h, d_k = q.shape
    n_k, d_v = k.shape[1], v.shape[3]
    out = np.empty((B, n_q, h, d_v), dtype=np.float64)
    kl = _keylens(key_lens, mask_kind)
    rc = lib.oracle_attn(_dp(q), _dp(k), _dp(v), _dp(out), B, h, n_q, n_k, d_k, d_v,
                         float(scale), int(mask_kind), _ip(kl), int(nthreads))
    _check(rc, "oracle_attn")
    return out


def attn_rows(q, k, v, scale, sel, mask_kind=MASK_NONE, key_lens=None, weights=False,
              nthreads=0):
    """Selected rows (b, t, head) of multi-head attention.

    Returns out_rows [n_sel, d_v] (and the weight rows [n_sel, n_k] when asked).
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, n_q, h, d_k = q.shape
    n_k, d_v = k.shape[1], v.shape[3]
    sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 3)
    out = np.empty((sel.shape[0], d_v), dtype=np.float64)
    w = np.empty((sel.shape[0], n_k), dtype=np.float64) if weights else None
    kl = _keylens(key_lens, mask_kind)
    rc = lib.oracle_attn_rows(_dp(q), _dp(k), _dp(v), B, h, n_q, n_k, d_k, d_v, float(scale),
                              int(mask_kind), _ip(kl), _ip(sel), sel.shape[0], _dp(out),
                              _dp(w) if weights else None, int(nthreads))
    _check(rc, "oracle_attn_rows")
    return (out, w) if weights else out


def matmul(a, w, nthreads=0) -> np.ndarray:
    lib = _load()
    a, w = _f64(a), _f64(w)
    M, K = a.shape
    N = w.shape[1]
    c = np.empty((M, N), dtype=np.float64)
    lib.oracle_matmul(_dp(a), _dp(w), _dp(c), M, K, N, int(nthreads))
    return c


def layernorm(z, gamma, beta, eps) -> np.ndarray:
    """LayerNorm over the last axis of a 2-D array (row by row)."""
    lib = _load()
    z = _f64(z)
    z2 = z.reshape(-1, z.shape[-1])
    g, b = _f64(gamma), _f64(beta)
    y = np.empty_like(z2)
    for r in range(z2.shape[0]):
        row = np.ascontiguousarray(z2[r])
        yr = np.empty_like(row)
        lib.oracle_layernorm_row(_dp(row), _dp(g), _dp(b), float(eps), row.size, _dp(yr))
        y[r] = yr
    return y.reshape(z.shape)


def mha(x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, h, mask_kind=MASK_NONE, key_lens=None,
        nthreads=0, intermediates=False):
    """Post-norm MHA sublayer: y = LN(X_q + Concat_i Attn(X_q W^Q_i, X_kv W^K_i, X_kv W^V_i) W^O).

    x_q [B, n_q, d_model], x_kv [B, n_k, d_model]; returns y [B, n_q, d_model]
    (and the dict of fp64 intermediates Q, K, V, A when asked).
    """
    lib = _load()
    x_q, x_kv = _f64(x_q), _f64(x_kv)
    wq, wk, wv, wo = _f64(wq), _f64(wk), _f64(wv), _f64(wo)
    gamma, beta = _f64(gamma), _f64(beta)
    B, n_q, d_model = x_q.shape
    n_k = x_kv.shape[1]
    d_k = wq.shape[1] // h
    d_v = wv.shape[1] // h
    y = np.empty_like(x_q)
    inter = None
    ptrs = [None] * 4
    if intermediates:
        inter = {
            "q": np.empty((B, n_q, h, d_k)), "k": np.empty((B, n_k, h, d_k)),
            "v": np.empty((B, n_k, h, d_v)), "a": np.empty((B, n_q, h, d_v)),
        }
        ptrs = [_dp(inter[n]) for n in ("q", "k", "v", "a")]
    kl = _keylens(key_lens, mask_kind)
    rc = lib.oracle_mha(_dp(x_q), _dp(x_kv), _dp(wq), _dp(wk), _dp(wv), _dp(wo), _dp(gamma),
                        _dp(beta), float(eps), _dp(y), B, n_q, n_k, d_model, h, d_k, d_v,
                        int(mask_kind), _ip(kl), int(nthreads), *ptrs)
    _check(rc, "oracle_mha")
    return (y, inter) if intermediates else y


def mha_rows(x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, h, sel, mask_kind=MASK_NONE,
             key_lens=None, nthreads=0) -> np.ndarray:
    """Selected output rows (b, t) of the sublayer -> [n_sel, d_model]."""
    lib = _load()
    x_q, x_kv = _f64(x_q), _f64(x_kv)
    wq, wk, wv, wo = _f64(wq), _f64(wk), _f64(wv), _f64(wo)
    gamma, beta = _f64(gamma), _f64(beta)
    B, n_q, d_model = x_q.shape
    n_k = x_kv.shape[1]
    d_k = wq.shape[1] // h
    d_v = wv.shape[1] // h
    sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
    y = np.empty((sel.shape[0], d_model), dtype=np.float64)
    kl = _keylens(key_lens, mask_kind)
    rc = lib.oracle_mha_rows(_dp(x_q), _dp(x_kv), _dp(wq), _dp(wk), _dp(wv), _dp(wo), _dp(gamma),
                             _dp(beta), float(eps), B, n_q, n_k, d_model, h, d_k, d_v,
                             int(mask_kind), _ip(kl), _ip(sel), sel.shape[0], _dp(y),
                             int(nthreads))
    _check(rc, "oracle_mha_rows")
    return y


def pos_encoding(B, n, d_model, emb=None, emb_scale=1.0, pos0=0) -> np.ndarray:
    """Sinusoidal encoding of positions pos0 .. pos0+n-1 added to emb * emb_scale
    (emb [B, n, d_model] fp64, or None for the encoding alone) -> [B, n, d_model]."""
    lib = _load()
    out = np.empty((B, n, d_model), dtype=np.float64)
    e = None if emb is None else _f64(emb)
    rc = lib.oracle_pos_encoding(None if e is None else _dp(e), _dp(out), int(B), int(n),
                                 int(d_model), float(emb_scale), int(pos0))
    _check(rc, "oracle_pos_encoding")
    return out


def ffn(x, w1, b1, w2, b2, gamma, beta, eps, nthreads=0) -> np.ndarray:
    """Post-norm feed-forward sublayer y = LayerNorm(x + max(0, x W1 + b1) W2 + b2) on the
    rows of x [..., d_model] (W1 [d_model, d_ff], W2 [d_ff, d_model])."""
    lib = _load()
    x = _f64(x)
    shape = x.shape
    d_model = shape[-1]
    x2 = x.reshape(-1, d_model)
    w1, b1, w2, b2 = _f64(w1), _f64(b1), _f64(w2), _f64(b2)
    gamma, beta = _f64(gamma), _f64(beta)
    d_ff = w1.shape[1]
    y = np.empty_like(x2)
    rc = lib.oracle_ffn(_dp(x2), _dp(w1), _dp(b1), _dp(w2), _dp(b2), _dp(gamma), _dp(beta),
                        float(eps), _dp(y), x2.shape[0], d_model, d_ff, int(nthreads))
    _check(rc, "oracle_ffn")
    return y.reshape(shape)


def attn_bwd(q, k, v, dout, scale, mask_kind=MASK_NONE, key_lens=None):
    """Gradients (dq, dk, dv) of sum(dout * attn(q, k, v)) and the forward's per-row
    log-sum-exp lse [B, h, n_q] (natural log of sum_j exp(scale q.k_j) over visible keys)."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, n_q, h, d_k = q.shape
    n_k, d_v = k.shape[1], v.shape[3]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    lse = np.empty((B, h, n_q), dtype=np.float64)
    kl = _keylens(key_lens, mask_kind)
    rc = lib.oracle_attn_bwd(_dp(q), _dp(k), _dp(v), _dp(dout), B, h, n_q, n_k, d_k, d_v,
                             float(scale), int(mask_kind), _ip(kl), _dp(dq), _dp(dk), _dp(dv),
                             _dp(lse))
    _check(rc, "oracle_attn_bwd")
    return dq, dk, dv, lse
