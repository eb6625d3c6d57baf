"""GPU parity of the feed-forward sublayer and of the encoder / decoder layers
(through the C ABI) against the fp64 oracle.

The layers are compositions of bf16-in / bf16-out sublayers. Each sublayer is
checked at the single bf16 tolerance against the oracle run on the GPU's own
input to that sublayer, and the layer entry points are checked to be bit for
bit the composition of the sublayer entry points. The composed checks compare
the layer output with the oracle's own composition (oracle.mha / oracle.ffn
with each sublayer's output rounded to bf16, as the API hands it on), at the
chained tolerance; everything inside a sublayer stays fp64 on the oracle side."""

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


@pytest.mark.parametrize("offset", [8.0, -60.0])
def test_ffn_layernorm_rows_far_from_zero(offset):
    # Rows whose values sit far from zero (x = offset + N(0, 1)): the LayerNorm's mean and
    # variance must come out without cancellation (a plain sum of squares in fp32 would
    # lose the variance against offset^2).
    hattn.build()
    M, dm, dff = 640, 512, 512
    w = synth.Workload("ffn_offset", "bf16", B=1, h=1, n_q=M, n_k=M, d_k=64, d_v=64, mask_kind=0,
                       seed=77, d_model=dm, d_ff=dff, kind="encoder")
    f = synth.ffn_inputs(w)
    x = synth.round_to_bf16_bits(offset + synth.draw_normal(w.seed, synth.STREAM_XQ, (M, dm)))
    d = _dev_ffn(f)
    y = hattn.ffn_fwd(to_device(x, "bf16"), d["w1"], d["b1"], d["w2"], d["b2"], d["gamma"],
                      d["beta"], f["eps"])
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    assert_close(from_device(y), _oracle_ffn(_w(x), f), "bf16", f"ffn offset {offset}")


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


def _gpu_mha(xq_dev, xkv_dev, m_dev, eps, h, mask, kl_dev):
    return hattn.mha_fwd(xq_dev, xkv_dev, m_dev["wq"], m_dev["wk"], m_dev["wv"], m_dev["wo"],
                         m_dev["gamma"], m_dev["beta"], eps, h, mask_kind=mask, key_lens=kl_dev)


def _gpu_ffn(x_dev, f_dev, eps):
    return hattn.ffn_fwd(x_dev, f_dev["w1"], f_dev["b1"], f_dev["w2"], f_dev["b2"],
                         f_dev["gamma"], f_dev["beta"], eps)


ENCODER_CASES = [
    synth.Workload("enc_case", "bf16", B=2, h=2, n_q=200, n_k=200, d_k=64, d_v=64,
                   mask_kind=synth.MASK_KEY_PADDING, seed=51, key_len_range=(60, 200),
                   d_model=128, d_ff=256, kind="encoder"),
    synth.workload("encoder_layer_bf16"),
]
DECODER_CASES = [
    synth.Workload("dec_case", "bf16", B=2, h=2, n_q=150, n_k=260, d_k=64, d_v=64,
                   mask_kind=synth.MASK_KEY_PADDING, seed=52, key_len_range=(50, 260),
                   d_model=128, d_ff=256, kind="decoder"),
    synth.workload("decoder_layer_bf16"),
]


@pytest.mark.parametrize("w", ENCODER_CASES, ids=lambda w: w.name)
def test_encoder_layer_each_sublayer_at_the_single_tolerance(w):
    """Each sublayer of the encoder layer against the oracle run on the GPU's own
    input to that sublayer, at the single bf16 tolerance (not the chained one):
    y1 = MHA(x) against oracle.mha(x); y = FFN(y1) against oracle.ffn(y1 as the
    GPU produced it); and the layer entry point's output is bit for bit the
    composition of the two sublayer entry points."""
    inp = synth.layer_inputs(w)
    kl = inp["key_lens"]
    mask = synth.MASK_KEY_PADDING if kl is not None else 0
    x = to_device(inp["x"], "bf16")
    m, f = _dev_mha(inp["self_attn"]), _dev_ffn(inp["ffn"])
    kl_dev = keylens_device(kl)
    y1 = _gpu_mha(x, x, m, inp["eps"], w.h, mask, kl_dev)
    y = _gpu_ffn(y1, f, inp["eps"])
    layer = hattn.encoder_layer_fwd(x, m, f, inp["eps"], w.h, key_lens=kl_dev)
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    assert torch().equal(layer, y), "layer != FFN(MHA(x))"
    x64 = _w(inp["x"])
    y1_host = from_device(y1)
    assert_close(y1_host, _oracle_mha(x64, x64, inp["self_attn"], inp["eps"], w.h, mask, kl),
                 "bf16", f"{w.name}: MHA sublayer")
    assert_close(from_device(y), _oracle_ffn(y1_host, inp["ffn"]), "bf16",
                 f"{w.name}: FFN sublayer on the GPU's y1")


@pytest.mark.parametrize("w", DECODER_CASES, ids=lambda w: w.name)
def test_decoder_layer_each_sublayer_at_the_single_tolerance(w):
    """The decoder layer's three sublayers, each against the oracle on the GPU's
    own input at the single bf16 tolerance, and the layer entry point bit for bit
    equal to their composition."""
    inp = synth.layer_inputs(w)
    kl = inp["key_lens"]
    x, mem = to_device(inp["x"], "bf16"), to_device(inp["memory"], "bf16")
    ms, mc, f = _dev_mha(inp["self_attn"]), _dev_mha(inp["cross_attn"]), _dev_ffn(inp["ffn"])
    kl_dev = keylens_device(kl)
    y1 = _gpu_mha(x, x, ms, inp["eps"], w.h, synth.MASK_CAUSAL, None)
    y2 = _gpu_mha(y1, mem, mc, inp["eps"], w.h, synth.MASK_KEY_PADDING, kl_dev)
    y = _gpu_ffn(y2, f, inp["eps"])
    layer = hattn.decoder_layer_fwd(x, mem, ms, mc, f, inp["eps"], w.h, src_lens=kl_dev)
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    assert torch().equal(layer, y), "layer != FFN(cross(self(x)))"
    x64, mem64 = _w(inp["x"]), _w(inp["memory"])
    y1_host, y2_host = from_device(y1), from_device(y2)
    assert_close(y1_host, _oracle_mha(x64, x64, inp["self_attn"], inp["eps"], w.h,
                                      synth.MASK_CAUSAL, None),
                 "bf16", f"{w.name}: causal self-attention sublayer")
    assert_close(y2_host, _oracle_mha(y1_host, mem64, inp["cross_attn"], inp["eps"], w.h,
                                      synth.MASK_KEY_PADDING, kl),
                 "bf16", f"{w.name}: cross-attention sublayer on the GPU's y1")
    assert_close(from_device(y), _oracle_ffn(y2_host, inp["ffn"]), "bf16",
                 f"{w.name}: FFN sublayer on the GPU's y2")


def test_encoder_layer_full_size_composed():
    """The bench's encoder-layer workload at full size, every element against the
    oracle's composition of its sublayers (chained tolerance)."""
    w = synth.workload("encoder_layer_bf16")
    inp = synth.layer_inputs(w)
    y = hattn.encoder_layer_fwd(to_device(inp["x"], "bf16"), _dev_mha(inp["self_attn"]),
                                _dev_ffn(inp["ffn"]), inp["eps"], w.h)
    torch().cuda.synchronize()
    x64 = _w(inp["x"])
    y1 = _oracle_mha(x64, x64, inp["self_attn"], inp["eps"], w.h, 0, None)
    ref = _oracle_ffn(_rb(y1), inp["ffn"])
    assert_close(from_device(y), ref, "bf16", "encoder_layer_bf16", tol=chained_tol(2))


def test_decoder_layer_full_size_composed():
    w = synth.workload("decoder_layer_bf16")
    inp = synth.layer_inputs(w)
    kl = inp["key_lens"]
    y = hattn.decoder_layer_fwd(to_device(inp["x"], "bf16"), to_device(inp["memory"], "bf16"),
                                _dev_mha(inp["self_attn"]), _dev_mha(inp["cross_attn"]),
                                _dev_ffn(inp["ffn"]), inp["eps"], w.h, src_lens=keylens_device(kl))
    torch().cuda.synchronize()
    x64 = _w(inp["x"])
    y1 = _rb(_oracle_mha(x64, x64, inp["self_attn"], inp["eps"], w.h, synth.MASK_CAUSAL, None))
    y2 = _rb(_oracle_mha(y1, _w(inp["memory"]), inp["cross_attn"], inp["eps"], w.h,
                         synth.MASK_KEY_PADDING, kl))
    ref = _oracle_ffn(y2, inp["ffn"])
    assert_close(from_device(y), ref, "bf16", "decoder_layer_bf16", tol=chained_tol(3))
