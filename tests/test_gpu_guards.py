"""Out-of-bounds writes, caught without a sanitizer: every output (and
workspace) buffer sits inside a larger allocation whose guard regions before
and after it hold a canary pattern. After each call the guards must still hold
it bit for bit, and the output must still match the oracle (or, for the MHA
sublayer, the same call on an unguarded buffer)."""

import math

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import assert_close, from_device, keylens_device, to_device, torch

pytestmark = pytest.mark.gpu

GUARD = 1024  # elements on each side (a multiple of 16 bytes for every dtype used)


def _canary(dtype):
    t = torch()
    if dtype == t.bfloat16:
        return t.int16, 0x7F21   # a NaN payload no kernel writes
    if dtype == t.float32:
        return t.int32, 0x7FC0DEAD
    return t.uint8, 0xA5


def guarded(shape, dtype):
    """(buffer, view): view is a contiguous tensor of `shape` in the middle of buffer."""
    t = torch()
    n = math.prod(shape)
    buf = t.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    bits_t, pattern = _canary(dtype)
    buf.view(bits_t).fill_(pattern)
    return buf, buf[GUARD:GUARD + n].view(shape)


def assert_guards_intact(buf, n, what):
    t = torch()
    t.cuda.synchronize()
    bits_t, pattern = _canary(buf.dtype)
    bits = buf.view(bits_t)
    assert bool((bits[:GUARD] == pattern).all()), f"{what}: write before the buffer"
    assert bool((bits[GUARD + n:] == pattern).all()), f"{what}: write past the buffer"


@pytest.fixture(scope="module", autouse=True)
def _built():
    hattn.build()
    hattn.load()


@pytest.mark.parametrize("dtype,B,h,n_q,n_k,d,mask", [
    ("bf16", 2, 3, 300, 300, 128, 3),   # tensor cores, causal + ragged key lengths
    ("bf16", 3, 5, 100, 200, 64, 2),    # short-sequence kernel, two key blocks, key padding
    ("bf16", 2, 3, 77, 120, 128, 2),    # short-sequence kernel at d = 128, rows past n_q clipped
    ("bf16", 2, 4, 128, 256, 64, 0),    # short-sequence kernel, full 128-row tile
    ("bf16", 3, 5, 130, 200, 64, 2),    # persistent tensor-core kernel, key padding
    ("f32", 2, 2, 70, 70, 64, 1),       # CUDA cores, fp32
    ("bf16", 1, 3, 50, 50, 32, 0),      # CUDA cores, bf16 head size the tensor cores do not take
])
def test_attention_writes_only_its_output(dtype, B, h, n_q, n_k, d, mask):
    t = torch()
    w = synth.Workload("guards", dtype, B=B, h=h, n_q=n_q, n_k=n_k, d_k=d, d_v=d, mask_kind=mask,
                       seed=900 + d, key_len_range=(1, n_k) if mask & 2 else None)
    inp = synth.attn_inputs(w)
    q, k, v = (to_device(inp[n], dtype) for n in ("q", "k", "v"))
    buf, out = guarded((B, n_q, h, d), t.float32 if dtype == "f32" else t.bfloat16)
    hattn.attn_fwd(q, k, v, out=out, scale=w.scale, mask_kind=mask,
                   key_lens=keylens_device(inp["key_lens"]))
    assert_guards_intact(buf, out.numel(), f"attn_fwd {dtype} d={d}")
    assert hattn.check_device_error() == 0
    ref = oracle.attn(*(synth.widen(inp[n], dtype) for n in ("q", "k", "v")), w.scale, mask,
                      inp["key_lens"])
    assert_close(from_device(out), ref, dtype, "attn_fwd inside guards")


def test_mha_writes_only_its_output_and_workspace():
    t = torch()
    w = synth.Workload("guards_mha", "bf16", B=2, h=2, n_q=100, n_k=100, d_k=64, d_v=64,
                       mask_kind=0, seed=913, d_model=128, kind="mha")
    inp = synth.mha_inputs(w)
    dev = {n: to_device(inp[n], "bf16") for n in ("x_q", "x_kv", "wq", "wk", "wv", "wo")}
    gamma, beta = t.from_numpy(inp["gamma"]).cuda(), t.from_numpy(inp["beta"]).cuda()
    args = (dev["x_q"], dev["x_kv"], dev["wq"], dev["wk"], dev["wv"], dev["wo"], gamma, beta,
            inp["eps"], w.h)
    ref = hattn.mha_fwd(*args)
    need = hattn.mha_workspace_bytes(hattn.HATTN_BF16, w.B, w.n_q, w.n_k, w.d_model, w.h, w.d_k,
                                     w.d_v)
    ybuf, y = guarded(tuple(ref.shape), t.bfloat16)
    wbuf, ws = guarded((need,), t.uint8)
    hattn.mha_fwd(*args, y=y, workspace=ws)
    assert_guards_intact(ybuf, y.numel(), "mha_fwd output")
    assert_guards_intact(wbuf, ws.numel(), "mha_fwd workspace")
    assert hattn.check_device_error() == 0
    assert_close(from_device(y), from_device(ref), "bf16", "mha_fwd inside guards")


def test_decode_writes_only_its_output_and_workspace():
    t = torch()
    B, h, n_max, d = 3, 4, 600, 128
    w = synth.Workload("guards_decode", "bf16", B=B, h=h, n_q=1, n_k=n_max, d_k=d, d_v=d,
                       mask_kind=synth.MASK_KEY_PADDING, seed=914, key_len_range=(1, n_max))
    inp = synth.attn_inputs(w)
    q, k, v = (to_device(inp[n], "bf16") for n in ("q", "k", "v"))
    obuf, out = guarded((B, 1, h, d), t.bfloat16)
    wbuf, ws = guarded((hattn.attn_decode_workspace_bytes(B, h, n_max, d),), t.uint8)
    hattn.attn_decode_fwd(q, k, v, keylens_device(inp["key_lens"]), out=out, scale=w.scale,
                          workspace=ws)
    assert_guards_intact(obuf, out.numel(), "attn_decode_fwd output")
    assert_guards_intact(wbuf, ws.numel(), "attn_decode_fwd workspace")
    assert hattn.check_device_error() == 0
    ref = oracle.attn(*(synth.widen(inp[n], "bf16") for n in ("q", "k", "v")), w.scale,
                      synth.MASK_KEY_PADDING, inp["key_lens"])
    assert_close(from_device(out), ref, "bf16", "decode inside guards")


@pytest.mark.parametrize("B,n,d_model", [(2, 37, 64), (3, 5000, 768)])
def test_positional_encoding_writes_only_its_output(B, n, d_model):
    t = torch()
    raw = synth.draw_normal(21, 0, (B, n, d_model))
    emb = synth.round_to_bf16_bits(raw)
    buf, out = guarded((B, n, d_model), t.bfloat16)
    scale = math.sqrt(d_model)
    hattn.pos_encoding_fwd(out, emb=to_device(emb, "bf16"), emb_scale=scale, pos0=3)
    assert_guards_intact(buf, out.numel(), "pos_encoding_fwd")
    assert hattn.check_device_error() == 0
    ref = oracle.pos_encoding(B, n, d_model, synth.widen(emb, "bf16"), float(np.float32(scale)), 3)
    np.testing.assert_allclose(from_device(out), ref, rtol=2 ** -8, atol=1e-5)
