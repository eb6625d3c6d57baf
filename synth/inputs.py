"""Seeded synthetic inputs for the attention workloads.

Draws come from numpy's Philox counter-based generator, keyed by
``(seed, stream_id, chunk)``: every tensor of a workload has its own
independent stream, cut into fixed 2^22-element chunks that are drawn in
parallel, so the values do not depend on the host or its thread count. Normal draws are fp64; they are rounded
to the dtype the kernel reads (fp32, or bf16 by round-to-nearest-even via
fp32) *before* either side sees them, and the oracle receives the rounded
values widened back to fp64.

Nothing here computes attention: no dot product, softmax or normalisation.
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np

# Stream ids: one independent substream per tensor of a workload.
STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2
STREAM_XQ, STREAM_XKV = 3, 4
STREAM_WQ, STREAM_WK, STREAM_WV, STREAM_WO = 5, 6, 7, 8
STREAM_KEYLEN = 9
STREAM_W1, STREAM_B1, STREAM_W2, STREAM_B2 = 10, 11, 12, 13
STREAM_DOUT = 14  # upstream gradient of the attention output (backward workloads)
# A second set of sublayer weights (the decoder layer's cross-attention) draws
# from the MHA streams offset by this much.
STREAM_CROSS_OFFSET = 100

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2


_CHUNK = 1 << 22  # elements per independently keyed chunk


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(
        np.random.Philox(np.random.SeedSequence([int(seed), int(stream), int(chunk)])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunked(n: int, fill) -> None:
    """Runs fill(chunk_index, start, stop) over fixed-size chunks on a thread pool.

    Chunk boundaries and keys do not depend on the thread count, so the draws
    are the same on every host.
    """
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for i, a in enumerate(starts):
            fill(i, a, min(n, a + _CHUNK))
        return
    with concurrent.futures.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(lambda ia: fill(ia[0], ia[1], min(n, ia[1] + _CHUNK)), enumerate(starts)))


def draw_normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """i.i.d. N(0, std^2) draws in fp64."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)

    def fill(i, a, b):
        _rng(seed, stream, i).standard_normal(size=b - a, dtype=np.float64, out=out[a:b])
        if std != 1.0:
            out[a:b] *= std

    _chunked(n, fill)
    return out.reshape(shape)


def draw_key_lens(seed: int, stream: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """One integer key length per batch element, uniform on [lo, hi] inclusive."""
    return _rng(seed, stream).integers(lo, hi + 1, size=batch, dtype=np.int64).astype(np.int32)


def round_to_f32(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)


def _bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    u = x32.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE); returns the bf16 bit patterns as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.empty(flat.size, dtype=np.uint16)

    def fill(i, a, b):
        out[a:b] = _bf16_bits_from_f32(flat[a:b].astype(np.float32))

    _chunked(flat.size, fill)
    return out.reshape(x.shape)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to fp64."""
    bits = np.ascontiguousarray(bits)
    flat = bits.reshape(-1)
    out = np.empty(flat.size, dtype=np.float64)

    def fill(i, a, b):
        out[a:b] = (flat[a:b].astype(np.uint32) << np.uint32(16)).view(np.float32)

    _chunked(flat.size, fill)
    return out.reshape(bits.shape)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic attention (or MHA sublayer) problem.

    Layout of every activation is [B, n, h, d] (heads concatenated along the
    feature axis), which is also the row-major [B*n, h*d] matrix X.W gives.
    """

    name: str
    dtype: str  # "f32" or "bf16"
    B: int
    h: int
    n_q: int
    n_k: int
    d_k: int
    d_v: int
    mask_kind: int
    seed: int
    key_len_range: tuple | None = None  # inclusive (lo, hi) when KEY_PADDING
    d_model: int = 0  # > 0 for the MHA sublayer (and the embedding width for "pe")
    description: str = ""
    kind: str = "attn"  # "attn", "mha", "decode" (n_q = 1 over a K/V prefix), "pe", "encoder", "decoder", "bwd"
    d_ff: int = 0  # feed-forward width of the encoder / decoder layer

    @property
    def scale(self) -> float:
        """1/sqrt(d_k), as the fp32 value passed to the kernels."""
        return float(np.float32(1.0 / math.sqrt(self.d_k)))

    @property
    def is_mha(self) -> bool:
        return self.kind == "mha"

    def attn_flops(self) -> float:
        """4*B*h*n_q*n_k*d, halved for causal (the defined metric's FLOP count)."""
        f = 4.0 * self.B * self.h * self.n_q * self.n_k * self.d_k
        return f * 0.5 if self.mask_kind & MASK_CAUSAL else f

    def proj_flops(self) -> float:
        if not self.is_mha:
            return 0.0
        hd = self.h * self.d_k
        return 2.0 * self.B * (self.n_q * self.d_model * hd + 2 * self.n_k * self.d_model * hd
                               + self.n_q * self.h * self.d_v * self.d_model)

    def layer_flops(self) -> float:
        """Defined FLOPs of one encoder / decoder layer: every attention at the metric's
        count (causal halved), every projection and both FFN GEMMs (2 per multiply-add)."""
        if self.kind not in ("encoder", "decoder"):
            return 0.0
        dm, hd = self.d_model, self.h * self.d_k
        Mq, Mk = self.B * self.n_q, self.B * self.n_k
        ffn = 2.0 * 2.0 * Mq * dm * self.d_ff
        self_proj = 2.0 * Mq * dm * hd * 4  # Q, K, V, O over the target rows
        self_attn = 4.0 * self.B * self.h * self.n_q * self.n_q * self.d_k
        if self.kind == "encoder":
            return ffn + self_proj + self_attn
        cross_proj = 2.0 * dm * hd * (2 * Mq + 2 * Mk)  # Q, O over the target; K, V over the source
        cross_attn = 4.0 * self.B * self.h * self.n_q * self.n_k * self.d_k
        return ffn + self_proj + 0.5 * self_attn + cross_proj + cross_attn

    def tokens(self) -> int:
        return self.B * self.n_q

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "enc_self_f32": Workload(
        "enc_self_f32", "f32", B=2, h=8, n_q=64, n_k=64, d_k=64, d_v=64,
        mask_kind=MASK_NONE, seed=0,
        description="encoder self-attention, fp32, B=2 h=8 n=64 d=64, unmasked"),
    "dec_causal_bf16": Workload(
        "dec_causal_bf16", "bf16", B=32, h=8, n_q=100, n_k=100, d_k=64, d_v=64,
        mask_kind=MASK_CAUSAL, seed=1,
        description="decoder masked self-attention, bf16, B=32 h=8 n=100 d=64, causal"),
    "cross_bf16": Workload(
        "cross_bf16", "bf16", B=64, h=8, n_q=128, n_k=256, d_k=64, d_v=64,
        mask_kind=MASK_KEY_PADDING, seed=2, key_len_range=(64, 256),
        description="cross-attention, bf16, B=64 h=8 n_q=128 n_k=256 d=64, key lengths U[64,256]"),
    "mha_bf16": Workload(
        "mha_bf16", "bf16", B=16, h=8, n_q=512, n_k=512, d_k=64, d_v=64,
        mask_kind=MASK_NONE, seed=3, d_model=512, kind="mha",
        description="post-norm MHA sublayer, bf16, B=16 n=512 d_model=512 h=8 d=64"),
    "encoder_layer_bf16": Workload(
        "encoder_layer_bf16", "bf16", B=16, h=8, n_q=512, n_k=512, d_k=64, d_v=64,
        mask_kind=MASK_NONE, seed=8, d_model=512, d_ff=2048, kind="encoder",
        description="post-norm encoder layer (MHA + FFN sublayers), bf16, B=16 n=512 d_model=512 "
                    "h=8 d=64 d_ff=2048"),
    "decoder_layer_bf16": Workload(
        "decoder_layer_bf16", "bf16", B=16, h=8, n_q=512, n_k=512, d_k=64, d_v=64,
        mask_kind=MASK_KEY_PADDING, seed=9, d_model=512, d_ff=2048, kind="decoder",
        key_len_range=(256, 512),
        description="post-norm decoder layer (causal self-attention, cross-attention over "
                    "source lengths U[256,512], FFN), bf16, B=16 n_tgt=n_src=512 d_model=512 h=8 "
                    "d=64 d_ff=2048"),
    "attn_bwd_bf16": Workload(
        "attn_bwd_bf16", "bf16", B=16, h=8, n_q=512, n_k=512, d_k=64, d_v=64,
        mask_kind=MASK_CAUSAL, seed=10, kind="bwd",
        description="attention backward (dQ, dK, dV), causal self-attention, bf16, B=16 h=8 "
                    "n=512 d=64"),
    "attn_bwd_long_d128": Workload(
        "attn_bwd_long_d128", "bf16", B=4, h=16, n_q=8192, n_k=8192, d_k=128, d_v=128,
        mask_kind=MASK_CAUSAL, seed=11, kind="bwd",
        description="attention backward (dQ, dK, dV) of the long-sequence causal self-attention, "
                    "bf16, B=4 h=16 n=8192 d=128"),
    "long_causal_d128": Workload(
        "long_causal_d128", "bf16", B=4, h=16, n_q=8192, n_k=8192, d_k=128, d_v=128,
        mask_kind=MASK_CAUSAL, seed=4,
        description="long-sequence causal self-attention, bf16, B=4 h=16 n=8192 d=128"),
    "decode_bf16": Workload(
        "decode_bf16", "bf16", B=32, h=32, n_q=1, n_k=8192, d_k=128, d_v=128,
        mask_kind=MASK_KEY_PADDING, seed=6, key_len_range=(4096, 8192), kind="decode",
        description="decode step, bf16, B=32 h=32 d=128, one query over a K/V prefix of "
                    "U[4096,8192] keys (cache capacity 8192)"),
    "pos_encoding_bf16": Workload(
        "pos_encoding_bf16", "bf16", B=16, h=1, n_q=8192, n_k=8192, d_k=512, d_v=512,
        mask_kind=MASK_NONE, seed=7, d_model=512, kind="pe",
        description="sinusoidal positional encoding added to sqrt(d_model)-scaled embeddings, "
                    "bf16, B=16 n=8192 d_model=512"),
    "long_causal_d64": Workload(
        "long_causal_d64", "bf16", B=4, h=32, n_q=8192, n_k=8192, d_k=64, d_v=64,
        mask_kind=MASK_CAUSAL, seed=5,
        description="long-sequence causal self-attention, bf16, B=4 h=32 n=8192 d=64"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def _to_kernel_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return round_to_f32(x)
    if dtype == "bf16":
        return round_to_bf16_bits(x)
    raise ValueError(dtype)


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Kernel-dtype array (fp32, or bf16 bits) -> exact fp64 copy for the oracle."""
    if dtype == "f32":
        return x.astype(np.float64)
    return bf16_bits_to_f64(x)


def attn_inputs(w: Workload) -> dict:
    """Q, K, V in [B, n, h, d] at the kernel dtype (fp32 arrays or bf16 bits), plus key lengths."""
    out = {
        "q": _to_kernel_dtype(draw_normal(w.seed, STREAM_Q, (w.B, w.n_q, w.h, w.d_k)), w.dtype),
        "k": _to_kernel_dtype(draw_normal(w.seed, STREAM_K, (w.B, w.n_k, w.h, w.d_k)), w.dtype),
        "v": _to_kernel_dtype(draw_normal(w.seed, STREAM_V, (w.B, w.n_k, w.h, w.d_v)), w.dtype),
        "key_lens": None,
    }
    if w.mask_kind & MASK_KEY_PADDING:
        lo, hi = w.key_len_range if w.key_len_range else (1, w.n_k)
        out["key_lens"] = draw_key_lens(w.seed, STREAM_KEYLEN, w.B, lo, hi)
    return out


def mha_inputs(w: Workload, self_attention: bool = True) -> dict:
    """X (and X_kv), the four projection matrices ~ N(0, 1/d_model), gamma=1, beta=0."""
    dm, hdk, hdv = w.d_model, w.h * w.d_k, w.h * w.d_v
    wstd = 1.0 / math.sqrt(dm)
    x_q = _to_kernel_dtype(draw_normal(w.seed, STREAM_XQ, (w.B, w.n_q, dm)), w.dtype)
    if self_attention:
        x_kv = x_q
    else:
        x_kv = _to_kernel_dtype(draw_normal(w.seed, STREAM_XKV, (w.B, w.n_k, dm)), w.dtype)
    out = {
        "x_q": x_q,
        "x_kv": x_kv,
        "wq": _to_kernel_dtype(draw_normal(w.seed, STREAM_WQ, (dm, hdk), wstd), w.dtype),
        "wk": _to_kernel_dtype(draw_normal(w.seed, STREAM_WK, (dm, hdk), wstd), w.dtype),
        "wv": _to_kernel_dtype(draw_normal(w.seed, STREAM_WV, (dm, hdv), wstd), w.dtype),
        "wo": _to_kernel_dtype(draw_normal(w.seed, STREAM_WO, (hdv, dm), wstd), w.dtype),
        "gamma": np.ones(dm, dtype=np.float32),
        "beta": np.zeros(dm, dtype=np.float32),
        "eps": 1e-6,
        "key_lens": None,
    }
    if w.mask_kind & MASK_KEY_PADDING:
        lo, hi = w.key_len_range if w.key_len_range else (1, w.n_k)
        out["key_lens"] = draw_key_lens(w.seed, STREAM_KEYLEN, w.B, lo, hi)
    return out


def ffn_inputs(w: Workload, seed_offset: int = 0) -> dict:
    """Feed-forward sublayer weights: W1 ~ N(0, 1/d_model), W2 ~ N(0, 1/d_ff) in the
    kernel dtype, biases b1, b2 ~ N(0, 0.1^2) in fp32, gamma = 1, beta = 0."""
    dm, dff = w.d_model, w.d_ff
    s = w.seed + seed_offset
    return {
        "w1": _to_kernel_dtype(draw_normal(s, STREAM_W1, (dm, dff), 1.0 / math.sqrt(dm)), w.dtype),
        "b1": draw_normal(s, STREAM_B1, (dff,), 0.1).astype(np.float32),
        "w2": _to_kernel_dtype(draw_normal(s, STREAM_W2, (dff, dm), 1.0 / math.sqrt(dff)), w.dtype),
        "b2": draw_normal(s, STREAM_B2, (dm,), 0.1).astype(np.float32),
        "gamma": np.ones(dm, dtype=np.float32),
        "beta": np.zeros(dm, dtype=np.float32),
        "eps": 1e-6,
    }


def _mha_weights(w: Workload, offset: int) -> dict:
    dm, hdk, hdv = w.d_model, w.h * w.d_k, w.h * w.d_v
    wstd = 1.0 / math.sqrt(dm)
    return {
        "wq": _to_kernel_dtype(draw_normal(w.seed, offset + STREAM_WQ, (dm, hdk), wstd), w.dtype),
        "wk": _to_kernel_dtype(draw_normal(w.seed, offset + STREAM_WK, (dm, hdk), wstd), w.dtype),
        "wv": _to_kernel_dtype(draw_normal(w.seed, offset + STREAM_WV, (dm, hdv), wstd), w.dtype),
        "wo": _to_kernel_dtype(draw_normal(w.seed, offset + STREAM_WO, (hdv, dm), wstd), w.dtype),
        "gamma": np.ones(dm, dtype=np.float32),
        "beta": np.zeros(dm, dtype=np.float32),
    }


def layer_inputs(w: Workload) -> dict:
    """Inputs of one encoder layer (kind "encoder": x [B, n_q, d_model], self-attention
    weights, FFN weights, optional key lengths) or decoder layer (kind "decoder": also the
    encoder output ("memory") [B, n_k, d_model], cross-attention weights, source lengths)."""
    out = {
        "x": _to_kernel_dtype(draw_normal(w.seed, STREAM_XQ, (w.B, w.n_q, w.d_model)), w.dtype),
        "self_attn": _mha_weights(w, 0),
        "ffn": ffn_inputs(w),
        "eps": 1e-6,
        "key_lens": None,
    }
    if w.kind == "decoder":
        out["memory"] = _to_kernel_dtype(draw_normal(w.seed, STREAM_XKV, (w.B, w.n_k, w.d_model)),
                                         w.dtype)
        out["cross_attn"] = _mha_weights(w, STREAM_CROSS_OFFSET)
    if w.mask_kind & MASK_KEY_PADDING:
        lo, hi = w.key_len_range if w.key_len_range else (1, w.n_k)
        out["key_lens"] = draw_key_lens(w.seed, STREAM_KEYLEN, w.B, lo, hi)
    return out


def attn_bwd_inputs(w: Workload) -> dict:
    """attn_inputs plus the upstream gradient dout ~ N(0, 1) [B, n_q, h, d_v] in the kernel dtype."""
    out = attn_inputs(w)
    out["dout"] = _to_kernel_dtype(draw_normal(w.seed, STREAM_DOUT, (w.B, w.n_q, w.h, w.d_v)), w.dtype)
    return out
