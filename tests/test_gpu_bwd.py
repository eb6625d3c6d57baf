"""GPU parity of attn_fwd_lse (the forward's row log-sum-exp) and attn_bwd (the
gradients of attention) through the C ABI, against the fp64 oracle."""

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import TOL, errors, from_device, keylens_device, to_device, torch

pytestmark = pytest.mark.gpu


def grad_tol(dtype, ref):
    """fp32: max |err| <= 2e-5 (1 + max|ref|) (fp32 sums over up to n rows of unit-size
    terms). bf16: the bf16 tolerances (2e-2 max, 2e-3 mean) scaled by the reference's
    magnitude when it exceeds 1: gradients are sums over many rows, and the relative
    error of a bf16 result does not depend on its scale."""
    scale_max = max(1.0, float(np.abs(ref).max()))
    if dtype == "f32":
        return 2e-5 * (1.0 + float(np.abs(ref).max())), None
    scale_mean = max(1.0, float(np.sqrt(np.mean(ref ** 2))))
    return TOL["bf16"][0] * scale_max, TOL["bf16"][1] * scale_mean


def check(got, ref, dtype, what):
    mx_tol, mn_tol = grad_tol(dtype, ref)
    assert np.all(np.isfinite(got)), what
    mx, mn = errors(got, ref)
    assert mx <= mx_tol, f"{what}: max |err| {mx:.3g} > {mx_tol:.3g} (mean {mn:.3g})"
    if mn_tol is not None:
        assert mn <= mn_tol, f"{what}: mean |err| {mn:.3g} > {mn_tol:.3g}"


CASES = [
    # dtype, B, h, n_q, n_k, d_k, d_v, mask, key_len_range
    ("f32", 2, 2, 64, 64, 64, 64, 0, None),
    ("f32", 1, 3, 100, 100, 32, 32, 1, None),
    ("bf16", 2, 2, 200, 200, 64, 64, 1, None),
    ("bf16", 3, 2, 77, 130, 64, 64, 2, (1, 130)),
    ("bf16", 2, 2, 300, 300, 128, 128, 3, (100, 300)),
    ("bf16", 1, 2, 150, 90, 64, 32, 2, (40, 90)),
    ("bf16", 2, 4, 512, 512, 64, 64, 1, None),
    ("bf16", 2, 2, 256, 384, 128, 128, 0, None),
    ("bf16", 1, 3, 333, 333, 128, 128, 1, None),
    ("bf16", 4, 1, 129, 257, 64, 64, 2, (1, 257)),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-n{c[3]}x{c[4]}-d{c[5]}/{c[6]}-m{c[7]}" for c in CASES])
def test_attn_bwd_matches_oracle(case):
    dtype, B, h, n_q, n_k, d_k, d_v, mask, klr = case
    hattn.build()
    w = synth.Workload("bwd_case", dtype, B=B, h=h, n_q=n_q, n_k=n_k, d_k=d_k, d_v=d_v,
                       mask_kind=mask, seed=600 + n_q + d_k, key_len_range=klr)
    inp = synth.attn_bwd_inputs(w)
    q, k, v, g = (to_device(inp[n], dtype) for n in ("q", "k", "v", "dout"))
    kl = keylens_device(inp["key_lens"])
    out, lse = hattn.attn_fwd_lse(q, k, v, scale=w.scale, mask_kind=mask, key_lens=kl)
    dq, dk, dv = hattn.attn_bwd(q, k, v, out, g, lse, scale=w.scale, mask_kind=mask, key_lens=kl)
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    wd = lambda a: synth.widen(a, dtype)
    rq, rk, rv, rlse = oracle.attn_bwd(wd(inp["q"]), wd(inp["k"]), wd(inp["v"]), wd(inp["dout"]),
                                       w.scale, mask, inp["key_lens"])
    # The forward's log-sum-exp: fp32 scores of the same inputs.
    np.testing.assert_allclose(from_device(lse), rlse, rtol=0, atol=1e-4 * (1 + np.abs(rlse).max()))
    # attn_fwd_lse writes exactly what attn_fwd writes.
    plain = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=mask, key_lens=kl)
    torch().cuda.synchronize()
    assert torch().equal(plain, out)
    check(from_device(dq), rq, dtype, "dq")
    check(from_device(dk), rk, dtype, "dk")
    check(from_device(dv), rv, dtype, "dv")


def test_attn_bwd_padded_rows_get_no_gradient():
    t = torch()
    w = synth.Workload("bwd_pad", "bf16", B=2, h=2, n_q=64, n_k=96, d_k=64, d_v=64,
                       mask_kind=2, seed=77, key_len_range=(1, 96))
    inp = synth.attn_bwd_inputs(w)
    q, k, v, g = (to_device(inp[n], "bf16") for n in ("q", "k", "v", "dout"))
    kl = keylens_device(np.array([40, 96], dtype=np.int32))
    out, lse = hattn.attn_fwd_lse(q, k, v, mask_kind=2, key_lens=kl)
    dq, dk, dv = hattn.attn_bwd(q, k, v, out, g, lse, mask_kind=2, key_lens=kl)
    t.cuda.synchronize()
    assert bool((dk[0, 40:] == 0).all()) and bool((dv[0, 40:] == 0).all())
    assert bool((dk[1, 90:] != 0).any())


def test_attn_bwd_bad_length_zeroes_and_raises():
    t = torch()
    w = synth.Workload("bwd_bad", "bf16", B=2, h=2, n_q=64, n_k=64, d_k=64, d_v=64,
                       mask_kind=2, seed=78, key_len_range=(1, 64))
    inp = synth.attn_bwd_inputs(w)
    q, k, v, g = (to_device(inp[n], "bf16") for n in ("q", "k", "v", "dout"))
    good = keylens_device(np.array([64, 64], dtype=np.int32))
    out, lse = hattn.attn_fwd_lse(q, k, v, mask_kind=2, key_lens=good)
    bad = keylens_device(np.array([0, 64], dtype=np.int32))
    dq, dk, dv = (t.full_like(x, float("nan")) for x in (q, k, v))
    hattn.attn_bwd(q, k, v, out, g, lse, mask_kind=2, key_lens=bad, dq=dq, dk=dk, dv=dv)
    assert hattn.check_device_error() == hattn._binding.EKEYLEN
    for x in (dq, dk, dv):
        assert bool((x[0] == 0).all()) and bool(t.isfinite(x[1]).all())
