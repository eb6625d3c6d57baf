"""Helpers for the GPU parity tests: moving seeded host inputs to the device,
reading results back exactly, and the tolerances the comparisons use."""

import numpy as np

from synth import inputs as synth

# Tolerances against the fp64 oracle: fp32 path max |err| <= 1e-5; bf16 path
# (bf16 inputs, fp32 accumulation, bf16 output) max |err| <= 2e-2 and
# mean |err| <= 2e-3.
TOL = {"f32": (1e-5, None), "bf16": (2e-2, 2e-3)}


def torch():
    import torch as _t
    return _t


def to_device(arr, dtype):
    t = torch()
    if dtype == "f32":
        return t.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()
    return t.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(t.bfloat16)


def from_device(x) -> np.ndarray:
    t = torch()
    if x.dtype == t.bfloat16:
        bits = x.contiguous().view(t.int16).cpu().numpy().view(np.uint16)
        return synth.bf16_bits_to_f64(bits)
    return x.cpu().numpy().astype(np.float64)


def keylens_device(key_lens):
    if key_lens is None:
        return None
    t = torch()
    return t.from_numpy(np.ascontiguousarray(key_lens, dtype=np.int32)).cuda()


def errors(got, ref):
    d = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64))
    return float(d.max()), float(d.mean())


def assert_close(got, ref, dtype, what="", tol=None):
    max_tol, mean_tol = tol if tol is not None else TOL[dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mn = errors(got, ref)
    assert mx <= max_tol, f"{what}: max |err| {mx:.3g} > {max_tol} (mean {mn:.3g})"
    if mean_tol is not None:
        assert mn <= mean_tol, f"{what}: mean |err| {mn:.3g} > {mean_tol} (max {mx:.3g})"
    return mx, mn


def chained_tol(sublayers: int):
    """bf16 tolerance of k chained sublayers. Each sublayer's bf16 output is the next
    one's input and reaches the next output through the residual with a gain of at
    most about 1 (LayerNorm divides by sigma(x + F(x)) >= ~1 for unit-variance x), so
    a sublayer's own error (its bf16 roundings, up to a flipped rounding of its
    input, 2^-8 |y|) adds to those before it: the per-sublayer max and mean
    tolerances add up once per sublayer (triangle inequality)."""
    max_tol, mean_tol = TOL["bf16"]
    return (sublayers * max_tol, sublayers * mean_tol)


def sample_rows(B, n_q, h, count, seed=0, n_tile=128):
    """Rows (b, t, i) to check one by one: every tile edge and ragged tail in
    the first and last rows, plus random rows."""
    rng = np.random.default_rng(seed)
    edges = sorted({0, 1, n_tile - 1, n_tile, 2 * n_tile - 1, 2 * n_tile, n_q // 2,
                    n_q - 2, n_q - 1} & set(range(n_q)))
    rows = []
    for t in edges:
        rows.append((int(rng.integers(B)), t, int(rng.integers(h))))
    rows.append((B - 1, n_q - 1, h - 1))
    rows.append((0, 0, 0))
    while len(rows) < count:
        rows.append((int(rng.integers(B)), int(rng.integers(n_q)), int(rng.integers(h))))
    return np.array(rows, dtype=np.int32)
