"""GPU parity of attn_decode_fwd (through the C ABI) against the fp64 oracle:
one query per (batch, head) over the first kv_lens[b] cached keys, i.e. the
oracle's attention with n_q = 1 and key padding."""

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import assert_close, from_device, keylens_device, to_device, torch

pytestmark = pytest.mark.gpu


def _run(w, inp):
    q, k, v = (to_device(inp[n], "bf16") for n in ("q", "k", "v"))
    out = hattn.attn_decode_fwd(q, k, v, keylens_device(inp["key_lens"]), scale=w.scale)
    torch().cuda.synchronize()
    return from_device(out)


@pytest.mark.parametrize("B,h,n_max,d,lens", [
    (2, 3, 1, 64, [1, 1]),
    (3, 2, 300, 128, [1, 129, 300]),
    (4, 4, 1000, 256, [999, 1000, 17, 512]),
    (1, 1, 70000, 128, [70000]),
    (8, 16, 777, 64, None),
])
def test_decode_matches_oracle(B, h, n_max, d, lens):
    hattn.build()
    w = synth.Workload("decode_case", "bf16", B=B, h=h, n_q=1, n_k=n_max, d_k=d, d_v=d,
                       mask_kind=synth.MASK_KEY_PADDING, seed=300 + n_max + d,
                       key_len_range=(1, n_max))
    inp = synth.attn_inputs(w)
    if lens is not None:
        inp["key_lens"] = np.array(lens, dtype=np.int32)
    got = _run(w, inp)
    assert hattn.check_device_error() == 0
    ref = oracle.attn(*(synth.widen(inp[n], "bf16") for n in ("q", "k", "v")), w.scale,
                      synth.MASK_KEY_PADDING, inp["key_lens"])
    assert_close(got, ref, "bf16", f"decode {B} {h} {n_max} {d}")


def test_decode_named_workload_full():
    """The bench's decode workload at full size, every output against the oracle
    over the first kv_lens[b] cached rows of each batch element."""
    w = synth.workload("decode_bf16")
    inp = synth.attn_inputs(w)
    got = _run(w, inp)
    assert hattn.check_device_error() == 0
    ref = np.empty_like(got)
    for b in range(w.B):
        L = int(inp["key_lens"][b])
        q = synth.widen(inp["q"][b:b + 1], "bf16")
        k, v = (synth.widen(inp[n][b:b + 1, :L], "bf16") for n in ("k", "v"))
        ref[b:b + 1] = oracle.attn(q, k, v, w.scale, synth.MASK_NONE, None)
    assert_close(got, ref, "bf16", "decode_bf16")


def test_decode_matches_attn_fwd_and_ignores_rows_past_length():
    t = torch()
    w = synth.Workload("decode_case", "bf16", B=2, h=4, n_q=1, n_k=640, d_k=128, d_v=128,
                       mask_kind=synth.MASK_KEY_PADDING, seed=9, key_len_range=(1, 640))
    inp = synth.attn_inputs(w)
    q, k, v = (to_device(inp[n], "bf16") for n in ("q", "k", "v"))
    kl = keylens_device(np.array([200, 640], dtype=np.int32))
    out1 = hattn.attn_decode_fwd(q, k, v, kl)
    k2, v2 = k.clone(), v.clone()
    k2[0, 200:] = 1e4
    v2[0, 200:] = -1e4
    out2 = hattn.attn_decode_fwd(q, k2, v2, kl)
    full = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=2, key_lens=kl)
    t.cuda.synchronize()
    assert t.equal(out1, out2)
    assert_close(from_device(out1), from_device(full), "bf16", "decode vs attn_fwd")


@pytest.mark.parametrize("d", [64, 256])
def test_decode_bad_length_zeroes_and_raises(d):
    t = torch()
    w = synth.Workload("decode_case", "bf16", B=2, h=2, n_q=1, n_k=256, d_k=d, d_v=d,
                       mask_kind=synth.MASK_KEY_PADDING, seed=10, key_len_range=(1, 256))
    inp = synth.attn_inputs(w)
    q, k, v = (to_device(inp[n], "bf16") for n in ("q", "k", "v"))
    out = t.full_like(q, float("nan"))
    hattn.attn_decode_fwd(q, k, v, keylens_device(np.array([0, 100], dtype=np.int32)), out=out)
    assert hattn.check_device_error() == hattn._binding.EKEYLEN
    got = from_device(out)
    assert np.all(got[0] == 0.0) and np.all(np.isfinite(got[1]))
