"""GPU parity of attn_fwd (through the C ABI) against the fp64 CPU oracle.

Every case draws seeded inputs, rounds them to the kernel dtype, runs the
CUDA kernel and compares element by element with the oracle on the same
(rounded) inputs: fp32 max |err| <= 1e-5; bf16 max |err| <= 2e-2 and mean
|err| <= 2e-3. The full-size long-sequence workloads are checked on every
output element as well.
"""

import math

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import (TOL, assert_close, from_device, keylens_device, sample_rows,
                            to_device, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    hattn.build()
    hattn.load()


def run_kernel(w, inp):
    q, k, v = (to_device(inp[n], w.dtype) for n in ("q", "k", "v"))
    kl = keylens_device(inp["key_lens"])
    out = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl)
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    return from_device(out)


def oracle_full(w, inp):
    wq, wk, wv = (synth.widen(inp[n], w.dtype) for n in ("q", "k", "v"))
    return oracle.attn(wq, wk, wv, w.scale, w.mask_kind, inp["key_lens"])


def check_full(w, what=""):
    inp = synth.attn_inputs(w)
    got = run_kernel(w, inp)
    ref = oracle_full(w, inp)
    return assert_close(got, ref, w.dtype, what or w.name)


# ---------------------------------------------------------------- named workloads

@pytest.mark.parametrize("name", ["enc_self_f32", "dec_causal_bf16", "cross_bf16"])
def test_named_workload_full_parity(name):
    check_full(synth.workload(name))


@pytest.mark.parametrize("name", ["long_causal_d128", "long_causal_d64"])
def test_long_sequence_full_parity(name):
    """The long causal workloads at full size, every output element against the
    oracle (one batch element at a time to bound host memory), in the launch
    configuration the bench times."""
    w = synth.workload(name)
    inp = synth.attn_inputs(w)
    got = run_kernel(w, inp)
    assert np.all(np.isfinite(got))
    # Convexity at any size: every output lies within the range of the value entries.
    vmax = np.abs(synth.widen(inp["v"], w.dtype)).max()
    assert np.abs(got).max() <= vmax * (1 + 1e-2)
    err_max, err_sum = 0.0, 0.0
    for b in range(w.B):
        wq, wk, wv = (synth.widen(inp[n][b:b + 1], w.dtype) for n in ("q", "k", "v"))
        ref = oracle.attn(wq, wk, wv, w.scale, w.mask_kind, None)
        d = np.abs(got[b:b + 1] - ref)
        err_max = max(err_max, float(d.max()))
        err_sum += float(d.sum())
    err_mean = err_sum / got.size
    max_tol, mean_tol = TOL[w.dtype]
    assert err_max <= max_tol, f"{name}: max |err| {err_max:.3g} > {max_tol}"
    assert err_mean <= mean_tol, f"{name}: mean |err| {err_mean:.3g} > {mean_tol}"


# ---------------------------------------------------------------- shape sweeps

# n_q <= 128 runs two heads per unit on the tensor-core path: (3, 3, ...) pairs heads of
# different batches (different key lengths) and leaves the last unit's second tile empty.
SHAPES = [(1, 1, 1, 1), (2, 3, 100, 100), (1, 2, 129, 129), (2, 2, 300, 300), (1, 1, 520, 520),
          (3, 2, 77, 300), (2, 1, 256, 64), (1, 1, 1, 700), (3, 3, 50, 200), (3, 3, 128, 128)]


def _sweep_workload(dtype, B, h, n_q, n_k, d_k, d_v, mask_kind):
    seed = 1000 + 7 * B + 13 * h + 17 * n_q + 19 * n_k + 23 * d_k + 29 * d_v + mask_kind
    return synth.Workload("sweep", dtype, B=B, h=h, n_q=n_q, n_k=n_k, d_k=d_k, d_v=d_v,
                          mask_kind=mask_kind, seed=seed, key_len_range=(1, n_k))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
@pytest.mark.parametrize("shape", SHAPES)
def test_bf16_tensor_core_shapes(d, mask_kind, shape):
    B, h, n_q, n_k = shape
    if mask_kind & 1 and n_q != n_k:
        pytest.skip("causal needs n_q == n_k")
    check_full(_sweep_workload("bf16", B, h, n_q, n_k, d, d, mask_kind), f"bf16 d={d} {shape}")


@pytest.mark.parametrize("dtype,d_k,d_v", [("f32", 64, 64), ("f32", 128, 128), ("f32", 32, 96),
                                           ("f32", 4, 4), ("bf16", 32, 32), ("bf16", 256, 256),
                                           ("bf16", 128, 64), ("bf16", 8, 8)])
@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 3, 100, 100), (1, 2, 129, 129),
                                   (3, 2, 77, 300), (2, 3, 64, 64), (3, 2, 33, 33), (2, 2, 50, 40)])
def test_cuda_core_shapes(dtype, d_k, d_v, mask_kind, shape):
    B, h, n_q, n_k = shape
    if mask_kind & 1 and n_q != n_k:
        pytest.skip("causal needs n_q == n_k")
    check_full(_sweep_workload(dtype, B, h, n_q, n_k, d_k, d_v, mask_kind),
               f"{dtype} dk={d_k} dv={d_v} {shape}")


@pytest.mark.parametrize("shape,d", [((256, 16, 64, 64), 64), ((1, 1, 1, 8192), 128),
                                     ((2, 4, 2048, 2048), 128)])
def test_large_grids(shape, d):
    B, h, n_q, n_k = shape
    w = _sweep_workload("bf16", B, h, n_q, n_k, d, d, 0)
    inp = synth.attn_inputs(w)
    got = run_kernel(w, inp)
    sel = sample_rows(B, n_q, h, 128, seed=3)
    wq, wk, wv = (synth.widen(inp[n], w.dtype) for n in ("q", "k", "v"))
    ref = oracle.attn_rows(wq, wk, wv, w.scale, sel, 0, None)
    assert_close(got[sel[:, 0], sel[:, 1], sel[:, 2]], ref, "bf16", str(shape))


# n_q <= 128 with n_k <= 256 at d = 64 (n_k <= 128 at d = 128) runs the short-sequence
# kernel (one CTA per head): key lengths on both sides of the 128-key block edge, a single
# query row, full tiles.
@pytest.mark.parametrize("d,n_q,n_k", [(64, 128, 256), (64, 1, 129), (64, 100, 256),
                                       (64, 77, 130), (128, 128, 128), (128, 1, 1),
                                       (128, 100, 127)])
def test_short_kernel_key_lengths_around_the_block_edge(d, n_q, n_k):
    lens = sorted({1, min(127, n_k), min(128, n_k), min(129, n_k), max(1, n_k - 1), n_k})
    w = _sweep_workload("bf16", len(lens), 3, n_q, n_k, d, d, synth.MASK_KEY_PADDING)
    inp = synth.attn_inputs(w)
    inp["key_lens"] = np.array(lens, dtype=np.int32)
    assert_close(run_kernel(w, inp), oracle_full(w, inp), "bf16", f"short d={d} {n_q}x{n_k}")


@pytest.mark.parametrize("d,n", [(64, 128), (64, 37), (128, 128), (128, 65)])
def test_short_kernel_log_sum_exp(d, n):
    # attn_fwd_lse on the short-sequence kernel: the row log-sum-exp of the scaled scores.
    w = _sweep_workload("bf16", 2, 3, n, n, d, d, synth.MASK_CAUSAL)
    inp = synth.attn_inputs(w)
    q, k, v = (to_device(inp[x], "bf16") for x in ("q", "k", "v"))
    out, lse = hattn.attn_fwd_lse(q, k, v, scale=w.scale, mask_kind=1)
    torch().cuda.synchronize()
    assert hattn.check_device_error() == 0
    wq, wk, wv = (synth.widen(inp[x], "bf16") for x in ("q", "k", "v"))
    assert_close(from_device(out), oracle.attn(wq, wk, wv, w.scale, 1, None), "bf16", "lse out")
    rlse = oracle.attn_bwd(wq, wk, wv, np.zeros_like(wv), w.scale, 1, None)[3]
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, rtol=0, atol=1e-4 * (1 + np.abs(rlse).max()))


# ---------------------------------------------------------------- invariants

def _device_inputs(w, inp):
    return [to_device(inp[n], w.dtype) for n in ("q", "k", "v")]


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_causal_future_perturbation_is_bitwise_invisible(dtype, d):
    n, t0 = 300, 150
    w = _sweep_workload(dtype, 2, 2, n, n, d, d, synth.MASK_CAUSAL)
    inp = synth.attn_inputs(w)
    q, k, v = _device_inputs(w, inp)
    out1 = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=1)
    k2, v2 = k.clone(), v.clone()
    k2[:, t0 + 1:] = 1e4
    v2[:, t0 + 1:] = -1e4
    out2 = hattn.attn_fwd(q, k2, v2, scale=w.scale, mask_kind=1)
    torch().cuda.synchronize()
    assert torch().equal(out1[:, :t0 + 1], out2[:, :t0 + 1])
    assert not torch().equal(out1[:, t0 + 1:], out2[:, t0 + 1:])


@pytest.mark.parametrize("dtype,d,n_k", [("bf16", 64, 300), ("bf16", 128, 300), ("f32", 64, 300),
                                         ("bf16", 64, 200), ("f32", 64, 60)])
def test_padding_contents_are_bitwise_invisible(dtype, d, n_k):
    # n_k = 200 runs the short-sequence tensor-core kernel, n_k = 60 in fp32 the CUDA-core
    # kernel with the head's keys resident in shared memory.
    w = _sweep_workload(dtype, 4, 2, 100, n_k, d, d, synth.MASK_KEY_PADDING)
    inp = synth.attn_inputs(w)
    q, k, v = _device_inputs(w, inp)
    kl_host = np.array([1, min(129, n_k - 3), min(255, n_k - 1), n_k], dtype=np.int32)
    kl = keylens_device(kl_host)
    out1 = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=2, key_lens=kl)
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate(kl_host):
        k2[b, L:] = 1e4
        v2[b, L:] = -1e4
    out2 = hattn.attn_fwd(q, k2, v2, scale=w.scale, mask_kind=2, key_lens=kl)
    torch().cuda.synchronize()
    assert torch().equal(out1, out2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask_kind", [0, 1])
def test_growing_row_max_is_rescaled(d, mask_kind):
    # Scores that climb with the key index (q_0 = 1, k_j0 = j / 16, scale 1):
    # every 128-key block raises the row max by 8 = 2^3 in base e, i.e. by more
    # than 2^8 in the base-2 exponent, so the running sum and O are rescaled at
    # every block and the result must still match the oracle.
    n = 700
    w = _sweep_workload("bf16", 2, 2, n, n, d, d, mask_kind)
    inp = synth.attn_inputs(w)
    q = synth.widen(inp["q"], "bf16").copy()
    k = synth.widen(inp["k"], "bf16").copy()
    q[..., 1:] *= 0.25  # keeps the random part of the scores small against the ramp
    q[..., 0] = 1.0
    k[..., 0] = (np.arange(n) / 16.0)[None, :, None]
    qb, kb = synth.round_to_bf16_bits(q), synth.round_to_bf16_bits(k)
    qd, kd, vd = to_device(qb, "bf16"), to_device(kb, "bf16"), to_device(inp["v"], "bf16")
    got = from_device(hattn.attn_fwd(qd, kd, vd, scale=1.0, mask_kind=mask_kind))
    assert hattn.check_device_error() == 0
    ref = oracle.attn(synth.widen(qb, "bf16"), synth.widen(kb, "bf16"), synth.widen(inp["v"], "bf16"),
                      1.0, mask_kind, None)
    assert_close(got, ref, "bf16", f"growing max d={d}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_weights_sum_to_one(dtype, d):
    # V = 1 everywhere: every output is the sum of the row's weights, i.e. 1.
    w = _sweep_workload(dtype, 2, 2, 257, 257, d, d, synth.MASK_CAUSAL)
    inp = synth.attn_inputs(w)
    q, k, _ = _device_inputs(w, inp)
    tdt = torch().float32 if dtype == "f32" else torch().bfloat16
    v = torch().ones(k.shape, dtype=tdt, device="cuda")
    out = from_device(hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=1))
    assert_close(out, np.ones_like(out), dtype, "row sums")


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_printed_softmax_through_kernel(dtype, d):
    # Scores [1, 2, 3] (q = e_0, k_j = (j+1) e_0, scale 1) and V = identity rows:
    # the output row is the weight row, printed as [0.090, 0.245, 0.665].
    t = torch()
    tdt = t.float32 if dtype == "f32" else t.bfloat16
    q = t.zeros((1, 1, 1, d), dtype=tdt, device="cuda")
    q[0, 0, 0, 0] = 1
    k = t.zeros((1, 3, 1, d), dtype=tdt, device="cuda")
    v = t.zeros((1, 3, 1, d), dtype=tdt, device="cuda")
    for j in range(3):
        k[0, j, 0, 0] = j + 1
        v[0, j, 0, j] = 1
    w = from_device(hattn.attn_fwd(q, k, v, scale=1.0))[0, 0, 0, :3]
    if dtype == "f32":
        assert np.array_equal(np.round(w, 3), [0.090, 0.245, 0.665])
    else:
        np.testing.assert_allclose(w, [0.0900306, 0.2447285, 0.6652410], atol=2e-2 / 4)


def test_worked_example_through_kernel():
    # The worked example's printed weights and output (reconstructed inputs,
    # d_k = d_v = 2, zero-padded to 4 for 16-byte rows).
    t = torch()
    q = t.tensor([[1, 1, 0, 0]], dtype=t.float32).reshape(1, 1, 1, 4).cuda()
    k = t.tensor([[1, 0, 0, 0], [0, 0, 0, 0], [0, 1, 0, 0]], dtype=t.float32).reshape(1, 3, 1, 4).cuda()
    v = t.tensor([[2, 1, 0, 0], [0, 2, 0, 0], [2, 1, 0, 0]], dtype=t.float32).reshape(1, 3, 1, 4).cuda()
    scale = 1 / math.sqrt(2)
    out = from_device(hattn.attn_fwd(q, k, v, scale=scale))[0, 0, 0]
    assert np.array_equal(np.round(out[:2], 4), [1.6044, 1.1978])
    eye = t.eye(3, 4, dtype=t.float32).reshape(1, 3, 1, 4).cuda()
    wts = from_device(hattn.attn_fwd(q, k, eye, scale=scale))[0, 0, 0, :3]
    assert np.array_equal(np.round(wts, 4), [0.4011, 0.1978, 0.4011])


def test_repeatable_bitwise():
    w = synth.workload("cross_bf16")
    inp = synth.attn_inputs(w)
    q, k, v = _device_inputs(w, inp)
    kl = keylens_device(inp["key_lens"])
    o1 = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl)
    o2 = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl)
    torch().cuda.synchronize()
    assert torch().equal(o1, o2)


# ---------------------------------------------------------------- device-side errors

@pytest.mark.parametrize("d", [64, 128])
def test_bad_key_length_in_paired_units(d):
    # n_q <= 128 with h = 3: a unit's two heads can come from different batch
    # elements, so one tile of a unit is valid while the other is not.
    t = torch()
    w = _sweep_workload("bf16", 3, 3, 100, 200, d, d, synth.MASK_KEY_PADDING)
    inp = synth.attn_inputs(w)
    q, k, v = _device_inputs(w, inp)
    kl_host = np.array([50, 0, 201], dtype=np.int32)  # only batch 0 is valid
    out = t.full((3, 100, 3, d), float("nan"), device="cuda", dtype=t.bfloat16)
    hattn.attn_fwd(q, k, v, out=out, scale=w.scale, mask_kind=2, key_lens=keylens_device(kl_host))
    assert hattn.check_device_error() == hattn._binding.EKEYLEN
    got = from_device(out)
    assert np.all(got[1:] == 0.0)
    wq, wk, wv = (synth.widen(inp[n], w.dtype) for n in ("q", "k", "v"))
    ref = oracle.attn(wq[:1], wk[:1], wv[:1], w.scale, 2, kl_host[:1])
    assert_close(got[:1], ref, "bf16", "valid batch element")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64), ("bf16", 32)])
def test_bad_key_length_zeroes_that_batch_and_raises(dtype, d):
    t = torch()
    w = _sweep_workload(dtype, 3, 2, 130, 200, d, d, synth.MASK_KEY_PADDING)
    inp = synth.attn_inputs(w)
    q, k, v = _device_inputs(w, inp)
    kl_host = np.array([50, 0, 201], dtype=np.int32)  # only batch 0 is valid
    out = t.full((3, 130, 2, d), float("nan"), device="cuda",
                 dtype=t.float32 if dtype == "f32" else t.bfloat16)
    hattn.attn_fwd(q, k, v, out=out, scale=w.scale, mask_kind=2, key_lens=keylens_device(kl_host))
    assert hattn.check_device_error() == hattn._binding.EKEYLEN
    assert hattn.check_device_error() == 0  # the word was cleared
    got = from_device(out)
    assert np.all(got[1:] == 0.0)
    wq, wk, wv = (synth.widen(inp[n], w.dtype) for n in ("q", "k", "v"))
    ref = oracle.attn(wq[:1], wk[:1], wv[:1], w.scale, 2, kl_host[:1])
    assert_close(got[:1], ref, dtype, "valid batch element")
