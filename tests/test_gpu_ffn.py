"""GPU parity of the feed-forward sublayer and of the encoder / decoder layers
(through the C ABI) against the fp64 oracle.

The layers are compositions of bf16-in / bf16-out sublayers, so the oracle
side composes oracle.mha / oracle.ffn with each sublayer's output rounded to
bf16, exactly as the API hands it to the next sublayer; everything inside a
sublayer stays fp64 on the oracle side."""

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import (assert_close, chained_tol, from_device, keylens_device, to_device,
                            torch)

pytestmark = pytest.mark.gpu


def _w(x):
    return synth.widen(x, "bf16")


def _rb(x):
    """Round an fp64 array to bf16 and back (a sublayer's bf16 output)."""
    return synth.bf16_bits_to_f64(synth.round_to_bf16_bits(x))


def _dev_ffn(f):
    t = torch()
    return {"w1": to_device(f["w1"], "bf16"), "w2": to_device(f["w2"], "bf16"),
            "b1": t.from_numpy(f["b1"]).cuda(), "b2": t.from_numpy(f["b2"]).cuda(),
            "gamma": t.from_numpy(f["gamma"]).cuda(), "beta": t.from_numpy(f["beta"]).cuda()}


def _dev_mha(m):
    t = torch()
    d = {k: to_device(m[k], "bf16") for k in ("wq", "wk", "wv", "wo")}
    d["gamma"] = t.from_numpy(m["gamma"]).cuda()
    d["beta"] = t.from_numpy(m["beta"]).cuda()
    return d


def _oracle_ffn(x64, f, rows=None):
    return oracle.ffn(x64, _w(f["w1"]), f["b1"].astype(np.float64), _w(f["w2"]),
                      f["b2"].astype(np.float64), f["gamma"], f["beta"], f["eps"])


def _oracle_mha(xq64, xkv64, m, eps, h, mask, kl):
    return oracle.mha(xq64, xkv64, _w(m["wq"]), _w(m["wk"]), _w(m["wv"]), _w(m["wo"]),
                      m["gamma"].astype(np.float64), m["beta"].astype(np.float64), eps, h, mask, kl)


@pytest.mark.parametrize("M,dm,dff,biases", [(300, 128, 256, True), (1000, 512, 2048, True),
                                             (64, 64, 64, True), (129, 256, 320, False)])
def test_ffn_matches_oracle(M, dm, dff, biases):
    hattn.build()
    w = synth.Workload("ffn_case", "bf16", B=1, h=1, n_q=M, n_k=M, d_k=64, d_v=64, mask_kind=0,
                       seed=40 + dm,
                       d_model=dm, d_ff=dff, kind="encoder")
    f = synth.ffn_inputs(w)
    if not biases:
        f["b1"] = np.zeros_like(f["b1"])
        f["b2"] = np.zeros_like(f["b2"])
    x = synth.round_to_bf16_bits(synth.draw_normal(w.seed, synth.STREAM_XQ, (M, dm)))
    d = _dev_ffn(f)
    y = hattn.ffn_fwd(to_device(x, "bf16"), d["w1"], d["b1"] if biases else None, d["w2"],
                      d["b2"] if biases else None, d["gamma"], d["beta"], f["eps"])
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    ref = _oracle_ffn(_w(x), f)
    assert_close(from_device(y), ref, "bf16", f"ffn {M} {dm} {dff}")


@pytest.mark.parametrize("padding", [False, True])
def test_encoder_layer_matches_oracle(padding):
    w = synth.Workload("enc_case", "bf16", B=2, h=2, n_q=200, n_k=200, d_k=64, d_v=64,
                       mask_kind=synth.MASK_KEY_PADDING if padding else 0, seed=51,
                       key_len_range=(60, 200), d_model=128, d_ff=256, kind="encoder")
    inp = synth.layer_inputs(w)
    kl = inp["key_lens"]
    y = hattn.encoder_layer_fwd(to_device(inp["x"], "bf16"), _dev_mha(inp["self_attn"]),
                                _dev_ffn(inp["ffn"]), inp["eps"], w.h,
                                key_lens=keylens_device(kl))
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    y1 = _oracle_mha(_w(inp["x"]), _w(inp["x"]), inp["self_attn"], inp["eps"], w.h,
                     synth.MASK_KEY_PADDING if padding else 0, kl)
    ref = _oracle_ffn(_rb(y1), inp["ffn"])
    assert_close(from_device(y), ref, "bf16", "encoder layer", tol=chained_tol(2))


def test_decoder_layer_matches_oracle():
    w = synth.Workload("dec_case", "bf16", B=2, h=2, n_q=150, n_k=260, d_k=64, d_v=64,
                       mask_kind=synth.MASK_KEY_PADDING, seed=52, key_len_range=(50, 260),
                       d_model=128, d_ff=256, kind="decoder")
    inp = synth.layer_inputs(w)
    kl = inp["key_lens"]
    y = hattn.decoder_layer_fwd(to_device(inp["x"], "bf16"), to_device(inp["memory"], "bf16"),
                                _dev_mha(inp["self_attn"]), _dev_mha(inp["cross_attn"]),
                                _dev_ffn(inp["ffn"]), inp["eps"], w.h, src_lens=keylens_device(kl))
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    x64 = _w(inp["x"])
    y1 = _rb(_oracle_mha(x64, x64, inp["self_attn"], inp["eps"], w.h, synth.MASK_CAUSAL, None))
    y2 = _rb(_oracle_mha(y1, _w(inp["memory"]), inp["cross_attn"], inp["eps"], w.h,
                         synth.MASK_KEY_PADDING, kl))
    ref = _oracle_ffn(y2, inp["ffn"])
    assert_close(from_device(y), ref, "bf16", "decoder layer", tol=chained_tol(3))


def _sample_bt(B, n, count, seed):
    rng = np.random.default_rng(seed)
    edges = [(0, 0), (B - 1, n - 1), (0, 127), (0, 128), (B - 1, n // 2)]
    rand = [(int(b), int(t)) for b, t in zip(rng.integers(0, B, count), rng.integers(0, n, count))]
    return np.array(sorted(set(edges + rand)), dtype=np.int32)


def test_encoder_layer_full_size_sampled():
    """The bench's encoder-layer workload at full size, checked on sampled rows (the
    FFN is position-wise, so a row of y needs only that row of y1)."""
    w = synth.workload("encoder_layer_bf16")
    inp = synth.layer_inputs(w)
    y = hattn.encoder_layer_fwd(to_device(inp["x"], "bf16"), _dev_mha(inp["self_attn"]),
                                _dev_ffn(inp["ffn"]), inp["eps"], w.h)
    torch().cuda.synchronize()
    got = from_device(y)
    sel = _sample_bt(w.B, w.n_q, 24, seed=8)
    m = inp["self_attn"]
    x64 = _w(inp["x"])
    y1 = oracle.mha_rows(x64, x64, _w(m["wq"]), _w(m["wk"]), _w(m["wv"]), _w(m["wo"]),
                         m["gamma"].astype(np.float64), m["beta"].astype(np.float64), inp["eps"],
                         w.h, sel)
    ref = _oracle_ffn(_rb(y1), inp["ffn"])
    assert_close(got[sel[:, 0], sel[:, 1]], ref, "bf16", "encoder_layer_bf16 sampled",
                 tol=chained_tol(2))


def test_decoder_layer_full_size_sampled():
    w = synth.workload("decoder_layer_bf16")
    inp = synth.layer_inputs(w)
    kl = inp["key_lens"]
    y = hattn.decoder_layer_fwd(to_device(inp["x"], "bf16"), to_device(inp["memory"], "bf16"),
                                _dev_mha(inp["self_attn"]), _dev_mha(inp["cross_attn"]),
                                _dev_ffn(inp["ffn"]), inp["eps"], w.h, src_lens=keylens_device(kl))
    torch().cuda.synchronize()
    got = from_device(y)
    sel = _sample_bt(w.B, w.n_q, 16, seed=9)
    x64 = _w(inp["x"])
    ms, mc = inp["self_attn"], inp["cross_attn"]
    g = lambda m: (m["gamma"].astype(np.float64), m["beta"].astype(np.float64))
    y1 = _rb(oracle.mha_rows(x64, x64, _w(ms["wq"]), _w(ms["wk"]), _w(ms["wv"]), _w(ms["wo"]),
                             *g(ms), inp["eps"], w.h, sel, synth.MASK_CAUSAL))
    # Row t of the cross-attention output reads only row t of its query input.
    xq = np.zeros((w.B, w.n_q, w.d_model))
    xq[sel[:, 0], sel[:, 1]] = y1
    y2 = _rb(oracle.mha_rows(xq, _w(inp["memory"]), _w(mc["wq"]), _w(mc["wk"]), _w(mc["wv"]),
                             _w(mc["wo"]), *g(mc), inp["eps"], w.h, sel, synth.MASK_KEY_PADDING,
                             kl))
    ref = _oracle_ffn(y2, inp["ffn"])
    assert_close(got[sel[:, 0], sel[:, 1]], ref, "bf16", "decoder_layer_bf16 sampled",
                 tol=chained_tol(3))
