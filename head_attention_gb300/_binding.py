"""ctypes binding of libhattn.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
turns torch tensors into raw device pointers and sizes, calls the C ABI and
turns status codes into exceptions. There is no fallback path: if the library
is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import builder as _build

HATTN_F32, HATTN_BF16 = 0, 1
MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2
OK, EINVAL, EUNSUPPORTED, ECUDA, ETIMEOUT, EKEYLEN, EWORKSPACE, ESCRATCH = 0, -1, -2, -3, -4, -5, -6, -7
NOALLOC_SCRATCH_BYTES = 32 << 20

# Every symbol include/hattn.h declares.
EXPORTED = ("attn_fwd", "attn_fwd_lse", "attn_bwd", "attn_bwd_workspace_bytes", "attn_decode_fwd", "attn_decode_workspace_bytes", "mha_fwd",
            "mha_fwd_noalloc", "mha_workspace_bytes", "pos_encoding_fwd", "ffn_fwd",
            "ffn_workspace_bytes", "encoder_layer_fwd", "encoder_layer_workspace_bytes",
            "decoder_layer_fwd", "decoder_layer_workspace_bytes", "hattn_status_str",
            "hattn_check_device_error", "hattn_version", "hattn_selftest_wait_timeout")


class MhaWeights(ctypes.Structure):
    """hattn_mha_weights: device pointers of one MHA sublayer's weights."""
    _fields_ = [("Wq", ctypes.c_void_p), ("Wk", ctypes.c_void_p), ("Wv", ctypes.c_void_p),
                ("Wo", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p)]


class FfnWeights(ctypes.Structure):
    """hattn_ffn_weights: device pointers of one feed-forward sublayer's weights."""
    _fields_ = [("W1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("W2", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p)]

_lock = threading.Lock()
_lib = None


class HattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Loads libhattn.so (built in-tree by head_attention_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with head_attention_gb300.build()")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, vp]
        lib.attn_fwd.restype = i
        lib.mha_fwd.argtypes = [vp] * 8 + [f, vp, i, i, i, i, i, i, i, i, i, vp, vp, sz, vp]
        lib.mha_fwd.restype = i
        lib.mha_fwd_noalloc.argtypes = [vp] * 8 + [f, vp, i, i, i, i, i, i, i, i, i, vp, vp]
        lib.mha_fwd_noalloc.restype = i
        lib.attn_decode_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, sz, vp]
        lib.attn_decode_fwd.restype = i
        lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i]
        lib.attn_decode_workspace_bytes.restype = sz
        lib.pos_encoding_fwd.argtypes = [vp, vp, i, i, i, i, f, i, vp]
        lib.pos_encoding_fwd.restype = i
        lib.attn_fwd_lse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, vp]
        lib.attn_fwd_lse.restype = i
        lib.attn_bwd.argtypes = [vp] * 9 + [i] * 7 + [f, i, vp, vp, sz, vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_workspace_bytes.argtypes = [i, i, i]
        lib.attn_bwd_workspace_bytes.restype = sz
        lib.mha_workspace_bytes.argtypes = [i] * 8
        lib.mha_workspace_bytes.restype = sz
        lib.ffn_fwd.argtypes = [vp] * 7 + [f, vp, i, i, i, i, vp, sz, vp]
        lib.ffn_fwd.restype = i
        lib.ffn_workspace_bytes.argtypes = [i] * 4
        lib.ffn_workspace_bytes.restype = sz
        mw, fw = ctypes.POINTER(MhaWeights), ctypes.POINTER(FfnWeights)
        lib.encoder_layer_fwd.argtypes = [vp, mw, fw, f, vp, i, i, i, i, i, i, i, vp, vp, sz, vp]
        lib.encoder_layer_fwd.restype = i
        lib.encoder_layer_workspace_bytes.argtypes = [i] * 7
        lib.encoder_layer_workspace_bytes.restype = sz
        lib.decoder_layer_fwd.argtypes = ([vp, vp, mw, mw, fw, f, vp] + [i] * 8
                                          + [vp, vp, sz, vp])
        lib.decoder_layer_fwd.restype = i
        lib.decoder_layer_workspace_bytes.argtypes = [i] * 8
        lib.decoder_layer_workspace_bytes.restype = sz
        lib.hattn_status_str.argtypes = [i]
        lib.hattn_status_str.restype = ctypes.c_char_p
        lib.hattn_check_device_error.argtypes = [vp]
        lib.hattn_check_device_error.restype = i
        lib.hattn_version.argtypes = []
        lib.hattn_version.restype = i
        lib.hattn_selftest_wait_timeout.argtypes = [vp]
        lib.hattn_selftest_wait_timeout.restype = i
        _lib = lib
        return lib


def status_str(status: int) -> str:
    return load().hattn_status_str(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return HATTN_F32
    if t.dtype == torch.bfloat16:
        return HATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def attn_fwd_raw(q, k, v, out, dtype, B, h, n_q, n_k, d_k, d_v, scale, mask_kind, key_lens,
                 stream) -> int:
    """The C entry point with raw pointers (ints) or tensors; returns the status code."""
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), int(dtype), int(B), int(h),
                           int(n_q), int(n_k), int(d_k), int(d_v), float(scale), int(mask_kind),
                           _ptr(key_lens), _stream(stream))


def attn_fwd(q, k, v, out=None, scale=None, mask_kind=MASK_NONE, key_lens=None, stream=None):
    """Multi-head attention on [B, n, h, d] CUDA tensors (fp32 or bf16). Returns out."""
    import torch
    B, n_q, h, d_k = q.shape
    n_k, d_v = k.shape[1], v.shape[3]
    if out is None:
        out = torch.empty((B, n_q, h, d_v), dtype=q.dtype, device=q.device)
    if scale is None:
        scale = d_k ** -0.5
    for t in (q, k, v, out):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("attn_fwd needs contiguous CUDA tensors")
    rc = attn_fwd_raw(q, k, v, out, _dtype_code(q), B, h, n_q, n_k, d_k, d_v, scale, mask_kind,
                      key_lens, stream)
    if rc != OK:
        raise HattnError(rc, "attn_fwd")
    return out


def mha_workspace_bytes(dtype, B, n_q, n_k, d_model, h, d_k, d_v) -> int:
    return int(load().mha_workspace_bytes(int(dtype), int(B), int(n_q), int(n_k), int(d_model),
                                          int(h), int(d_k), int(d_v)))


def mha_fwd_raw(x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, y, dtype, B, n_q, n_k, d_model, h,
                d_k, d_v, mask_kind, key_lens, workspace, ws_bytes, stream) -> int:
    return load().mha_fwd(_ptr(x_q), _ptr(x_kv), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo),
                          _ptr(gamma), _ptr(beta), float(eps), _ptr(y), int(dtype), int(B),
                          int(n_q), int(n_k), int(d_model), int(h), int(d_k), int(d_v),
                          int(mask_kind), _ptr(key_lens), _ptr(workspace), int(ws_bytes),
                          _stream(stream))


def mha_fwd(x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, h, y=None, mask_kind=MASK_NONE,
            key_lens=None, workspace=None, stream=None):
    """Post-norm MHA sublayer on bf16 CUDA tensors x_q [B, n_q, d_model], x_kv [B, n_k, d_model]."""
    import torch
    B, n_q, d_model = x_q.shape
    n_k = x_kv.shape[1]
    d_k = wq.shape[1] // h
    d_v = wv.shape[1] // h
    if y is None:
        y = torch.empty_like(x_q)
    need = mha_workspace_bytes(HATTN_BF16, B, n_q, n_k, d_model, h, d_k, d_v)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x_q.device)
    rc = mha_fwd_raw(x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, y, _dtype_code(x_q), B, n_q, n_k,
                     d_model, h, d_k, d_v, mask_kind, key_lens, workspace, workspace.numel(),
                     stream)
    if rc != OK:
        raise HattnError(rc, "mha_fwd")
    return y


def mha_fwd_noalloc_raw(x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, y, dtype, B, n_q, n_k,
                        d_model, h, d_k, d_v, mask_kind, key_lens, stream) -> int:
    """mha_fwd without a workspace argument: the library's static scratch is used."""
    return load().mha_fwd_noalloc(_ptr(x_q), _ptr(x_kv), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo),
                                  _ptr(gamma), _ptr(beta), float(eps), _ptr(y), int(dtype), int(B),
                                  int(n_q), int(n_k), int(d_model), int(h), int(d_k), int(d_v),
                                  int(mask_kind), _ptr(key_lens), _stream(stream))


def attn_decode_workspace_bytes(B, h, n_max, d) -> int:
    return int(load().attn_decode_workspace_bytes(int(B), int(h), int(n_max), int(d)))


def attn_decode_fwd_raw(q, k_cache, v_cache, out, dtype, B, h, n_max, d, scale, kv_lens,
                        workspace, ws_bytes, stream) -> int:
    return load().attn_decode_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), int(dtype),
                                  int(B), int(h), int(n_max), int(d), float(scale), _ptr(kv_lens),
                                  _ptr(workspace), int(ws_bytes), _stream(stream))


def attn_decode_fwd(q, k_cache, v_cache, kv_lens, out=None, scale=None, workspace=None,
                    stream=None):
    """One decoding step: q [B, 1, h, d] against the first kv_lens[b] rows of the
    caches [B, n_max, h, d] (bf16 CUDA tensors). Returns out [B, 1, h, d]."""
    import torch
    B, _, h, d = q.shape
    n_max = k_cache.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_bytes(B, h, n_max, d), dtype=torch.uint8,
                                device=q.device)
    rc = attn_decode_fwd_raw(q, k_cache, v_cache, out, _dtype_code(q), B, h, n_max, d, scale,
                             kv_lens, workspace, workspace.numel(), stream)
    if rc != OK:
        raise HattnError(rc, "attn_decode_fwd")
    return out


def pos_encoding_fwd_raw(emb, out, dtype, B, n, d_model, emb_scale, pos0, stream) -> int:
    return load().pos_encoding_fwd(_ptr(emb), _ptr(out), int(dtype), int(B), int(n),
                                   int(d_model), float(emb_scale), int(pos0), _stream(stream))


def pos_encoding_fwd(out, emb=None, emb_scale=None, pos0=0, stream=None):
    """out [B, n, d_model] = emb * emb_scale + sinusoidal encoding (emb may be None).
    emb_scale defaults to sqrt(d_model)."""
    B, n, d_model = out.shape
    if emb_scale is None:
        emb_scale = d_model ** 0.5
    rc = pos_encoding_fwd_raw(emb, out, _dtype_code(out), B, n, d_model, emb_scale, pos0, stream)
    if rc != OK:
        raise HattnError(rc, "pos_encoding_fwd")
    return out


def check_device_error(stream=None) -> int:
    return int(load().hattn_check_device_error(_stream(stream)))


def version() -> int:
    return int(load().hattn_version())


def selftest_wait_timeout(stream=None) -> int:
    """Enqueues the kernel whose device wait never completes and must give up on
    its own (HATTN_ETIMEOUT in the device error word); returns the launch status."""
    return int(load().hattn_selftest_wait_timeout(_stream(stream)))


def ffn_workspace_bytes(dtype, M, d_model, d_ff) -> int:
    return int(load().ffn_workspace_bytes(int(dtype), int(M), int(d_model), int(d_ff)))


def ffn_fwd_raw(x, w1, b1, w2, b2, gamma, beta, eps, y, dtype, M, d_model, d_ff, workspace,
                ws_bytes, stream) -> int:
    return load().ffn_fwd(_ptr(x), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), _ptr(gamma),
                          _ptr(beta), float(eps), _ptr(y), int(dtype), int(M), int(d_model),
                          int(d_ff), _ptr(workspace), int(ws_bytes), _stream(stream))


def ffn_fwd(x, w1, b1, w2, b2, gamma, beta, eps, y=None, workspace=None, stream=None):
    """Post-norm feed-forward sublayer on bf16 CUDA tensors x [..., d_model]; b1, b2, gamma,
    beta fp32 (b1/b2 may be None)."""
    import torch
    d_model = x.shape[-1]
    M = x.numel() // d_model
    d_ff = w1.shape[1]
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = torch.empty(ffn_workspace_bytes(_dtype_code(x), M, d_model, d_ff),
                                dtype=torch.uint8, device=x.device)
    rc = ffn_fwd_raw(x, w1, b1, w2, b2, gamma, beta, eps, y, _dtype_code(x), M, d_model, d_ff,
                     workspace, workspace.numel(), stream)
    if rc != OK:
        raise HattnError(rc, "ffn_fwd")
    return y


def mha_weights(wq, wk, wv, wo, gamma, beta) -> MhaWeights:
    return MhaWeights(_ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(gamma), _ptr(beta))


def ffn_weights(w1, b1, w2, b2, gamma, beta) -> FfnWeights:
    return FfnWeights(_ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), _ptr(gamma), _ptr(beta))


def encoder_layer_workspace_bytes(dtype, B, n, d_model, h, d_k, d_ff) -> int:
    return int(load().encoder_layer_workspace_bytes(int(dtype), int(B), int(n), int(d_model),
                                                    int(h), int(d_k), int(d_ff)))


def encoder_layer_fwd_raw(x, attn, ffn, eps, y, dtype, B, n, d_model, h, d_k, d_ff, key_lens,
                          workspace, ws_bytes, stream) -> int:
    return load().encoder_layer_fwd(_ptr(x), ctypes.byref(attn) if attn is not None else None,
                                    ctypes.byref(ffn) if ffn is not None else None, float(eps),
                                    _ptr(y), int(dtype), int(B), int(n), int(d_model), int(h),
                                    int(d_k), int(d_ff), _ptr(key_lens), _ptr(workspace),
                                    int(ws_bytes), _stream(stream))


def encoder_layer_fwd(x, attn, ffn, eps, h, key_lens=None, y=None, workspace=None, stream=None):
    """One post-norm encoder layer on x [B, n, d_model] (bf16 CUDA). attn / ffn are dicts of
    CUDA tensors with keys wq, wk, wv, wo, gamma, beta / w1, b1, w2, b2, gamma, beta."""
    import torch
    B, n, d_model = x.shape
    d_k = attn["wq"].shape[1] // h
    d_ff = ffn["w1"].shape[1]
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = torch.empty(encoder_layer_workspace_bytes(_dtype_code(x), B, n, d_model, h,
                                                              d_k, d_ff),
                                dtype=torch.uint8, device=x.device)
    aw = mha_weights(*(attn[k] for k in ("wq", "wk", "wv", "wo", "gamma", "beta")))
    fw = ffn_weights(*(ffn[k] for k in ("w1", "b1", "w2", "b2", "gamma", "beta")))
    rc = encoder_layer_fwd_raw(x, aw, fw, eps, y, _dtype_code(x), B, n, d_model, h, d_k, d_ff,
                               key_lens, workspace, workspace.numel(), stream)
    if rc != OK:
        raise HattnError(rc, "encoder_layer_fwd")
    return y


def decoder_layer_workspace_bytes(dtype, B, n_tgt, n_src, d_model, h, d_k, d_ff) -> int:
    return int(load().decoder_layer_workspace_bytes(int(dtype), int(B), int(n_tgt), int(n_src),
                                                    int(d_model), int(h), int(d_k), int(d_ff)))


def decoder_layer_fwd_raw(x, memory, self_attn, cross_attn, ffn, eps, y, dtype, B, n_tgt, n_src,
                          d_model, h, d_k, d_ff, src_lens, workspace, ws_bytes, stream) -> int:
    ref = lambda s: ctypes.byref(s) if s is not None else None
    return load().decoder_layer_fwd(_ptr(x), _ptr(memory), ref(self_attn), ref(cross_attn),
                                    ref(ffn), float(eps), _ptr(y), int(dtype), int(B), int(n_tgt),
                                    int(n_src), int(d_model), int(h), int(d_k), int(d_ff),
                                    _ptr(src_lens), _ptr(workspace), int(ws_bytes),
                                    _stream(stream))


def decoder_layer_fwd(x, memory, self_attn, cross_attn, ffn, eps, h, src_lens=None, y=None,
                      workspace=None, stream=None):
    """One post-norm decoder layer: x [B, n_tgt, d_model], memory [B, n_src, d_model]
    (bf16 CUDA); weight dicts as for encoder_layer_fwd."""
    import torch
    B, n_tgt, d_model = x.shape
    n_src = memory.shape[1]
    d_k = self_attn["wq"].shape[1] // h
    d_ff = ffn["w1"].shape[1]
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = torch.empty(decoder_layer_workspace_bytes(_dtype_code(x), B, n_tgt, n_src,
                                                              d_model, h, d_k, d_ff),
                                dtype=torch.uint8, device=x.device)
    keys = ("wq", "wk", "wv", "wo", "gamma", "beta")
    sw = mha_weights(*(self_attn[k] for k in keys))
    cw = mha_weights(*(cross_attn[k] for k in keys))
    fw = ffn_weights(*(ffn[k] for k in ("w1", "b1", "w2", "b2", "gamma", "beta")))
    rc = decoder_layer_fwd_raw(x, memory, sw, cw, fw, eps, y, _dtype_code(x), B, n_tgt, n_src,
                               d_model, h, d_k, d_ff, src_lens, workspace, workspace.numel(),
                               stream)
    if rc != OK:
        raise HattnError(rc, "decoder_layer_fwd")
    return y


def attn_fwd_lse_raw(q, k, v, out, lse, dtype, B, h, n_q, n_k, d_k, d_v, scale, mask_kind, key_lens,
                     stream) -> int:
    return load().attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(dtype), int(B),
                               int(h), int(n_q), int(n_k), int(d_k), int(d_v), float(scale),
                               int(mask_kind), _ptr(key_lens), _stream(stream))


def attn_fwd_lse(q, k, v, out=None, lse=None, scale=None, mask_kind=MASK_NONE, key_lens=None,
                 stream=None):
    """attn_fwd that also returns the per-row log-sum-exp lse [B, h, n_q] (fp32)."""
    import torch
    B, n_q, h, d_k = q.shape
    n_k, d_v = k.shape[1], v.shape[3]
    if out is None:
        out = torch.empty((B, n_q, h, d_v), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, h, n_q), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d_k ** -0.5
    rc = attn_fwd_lse_raw(q, k, v, out, lse, _dtype_code(q), B, h, n_q, n_k, d_k, d_v, scale,
                          mask_kind, key_lens, stream)
    if rc != OK:
        raise HattnError(rc, "attn_fwd_lse")
    return out, lse


def attn_bwd_workspace_bytes(B, h, n_q) -> int:
    return int(load().attn_bwd_workspace_bytes(int(B), int(h), int(n_q)))


def attn_bwd_raw(q, k, v, out, dout, lse, dq, dk, dv, dtype, B, h, n_q, n_k, d_k, d_v, scale,
                 mask_kind, key_lens, workspace, ws_bytes, stream) -> int:
    return load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                           _ptr(dk), _ptr(dv), int(dtype), int(B), int(h), int(n_q), int(n_k),
                           int(d_k), int(d_v), float(scale), int(mask_kind), _ptr(key_lens),
                           _ptr(workspace), int(ws_bytes), _stream(stream))


def attn_bwd(q, k, v, out, dout, lse, scale=None, mask_kind=MASK_NONE, key_lens=None, dq=None,
             dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attention given dout; out and lse from attn_fwd_lse."""
    import torch
    B, n_q, h, d_k = q.shape
    n_k, d_v = k.shape[1], v.shape[3]
    if scale is None:
        scale = d_k ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_bytes(B, h, n_q), dtype=torch.uint8,
                                device=q.device)
    rc = attn_bwd_raw(q, k, v, out, dout, lse, dq, dk, dv, _dtype_code(q), B, h, n_q, n_k, d_k, d_v,
                      scale, mask_kind, key_lens, workspace, workspace.numel(), stream)
    if rc != OK:
        raise HattnError(rc, "attn_bwd")
    return dq, dk, dv
