"""GPU parity of pos_encoding_fwd (through the C ABI) against the fp64 oracle."""

import math

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import from_device, to_device, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,n,d_model,pos0,with_emb", [(1, 5, 4, 0, False), (2, 100, 512, 0, True),
                                                       (1, 8192, 512, 0, False), (3, 77, 128, 40000, True),
                                                       (1, 16, 64, (1 << 24) - 16, False),
                                                       (4, 1, 2, 7, True),
                                                       # >= 16 MB: the bulk-copy path (ragged last
                                                       # chunk; batch rows in two groups; no emb)
                                                       (3, 5000, 768, 0, True), (2, 3000, 1000, 123, True),
                                                       (10, 600, 4096, 0, True), (4, 8192, 512, 5, False)])
def test_pos_encoding_matches_oracle(dtype, B, n, d_model, pos0, with_emb):
    t = torch()
    hattn.build()
    emb = None
    emb_dev = None
    if with_emb:
        raw = synth.draw_normal(21, 0, (B, n, d_model))
        emb = raw.astype(np.float32) if dtype == "f32" else synth.round_to_bf16_bits(raw)
        emb_dev = to_device(emb, dtype)
    out = t.empty((B, n, d_model), dtype=t.float32 if dtype == "f32" else t.bfloat16, device="cuda")
    scale = math.sqrt(d_model)
    hattn.pos_encoding_fwd(out, emb=emb_dev, emb_scale=scale, pos0=pos0)
    t.cuda.synchronize()
    assert hattn.check_device_error() == 0
    ref = oracle.pos_encoding(B, n, d_model, None if emb is None else synth.widen(emb, dtype),
                              float(np.float32(scale)), pos0)
    got = from_device(out)
    if dtype == "f32":
        # fp32 output of an fp32 scale * emb sum: a few ulp of the largest term.
        tol = 4e-6 * (1 + np.abs(ref).max())
        assert np.abs(got - ref).max() <= tol
    else:
        # One bf16 rounding of the result: relative 2^-9, plus the fp32 sum.
        np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-5)


def test_pos_encoding_in_place():
    t = torch()
    x = t.randn(2, 33, 64, device="cuda")
    ref = x.clone()
    hattn.pos_encoding_fwd(x, emb=x, emb_scale=2.0)
    t.cuda.synchronize()
    pe = oracle.pos_encoding(1, 33, 64)[0]
    np.testing.assert_allclose(from_device(x), from_device(ref) * 2.0 + pe[None], atol=1e-5)


def test_pos_encoding_in_place_bulk_path():
    # 32 MB of fp32: large enough for the bulk-copy path, which reads each chunk
    # before it writes it back to the same addresses.
    t = torch()
    x = t.randn(2, 8192, 512, device="cuda")
    ref = x.clone()
    hattn.pos_encoding_fwd(x, emb=x, emb_scale=2.0, pos0=9)
    t.cuda.synchronize()
    assert hattn.check_device_error() == 0
    want = from_device(ref) * 2.0 + oracle.pos_encoding(1, 8192, 512, None, 1.0, 9)[0][None]
    assert np.abs(from_device(x) - want).max() <= 4e-6 * (1 + np.abs(want).max())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pos_encoding_8_byte_aligned_buffers(dtype):
    """Buffers that are 8- but not 16-byte aligned take the one-pair-per-thread path."""
    t = torch()
    tdt = t.float32 if dtype == "f32" else t.bfloat16
    B, n, d_model = 3, 50, 64
    off = 2 if dtype == "f32" else 4  # 8 bytes
    base_e = t.randn(B * n * d_model + off, device="cuda").to(tdt)
    base_o = t.empty(B * n * d_model + off, dtype=tdt, device="cuda")
    emb = base_e[off:].view(B, n, d_model)
    out = base_o[off:].view(B, n, d_model)
    assert out.data_ptr() % 16 == 8 and emb.data_ptr() % 16 == 8
    hattn.pos_encoding_fwd(out, emb=emb, emb_scale=8.0, pos0=3)
    t.cuda.synchronize()
    ref = oracle.pos_encoding(B, n, d_model, from_device(emb), 8.0, 3)
    tol = dict(rtol=0, atol=4e-6 * (1 + np.abs(ref).max())) if dtype == "f32" else dict(rtol=2 ** -8, atol=1e-5)
    np.testing.assert_allclose(from_device(out), ref, **tol)
