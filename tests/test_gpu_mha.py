"""GPU parity of mha_fwd (the post-norm MHA sublayer, through the C ABI)
against the fp64 CPU oracle: bf16 max |err| <= 2e-2, mean |err| <= 2e-3."""

import numpy as np
import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import assert_close, from_device, keylens_device, to_device, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    hattn.build()
    hattn.load()


def run_mha(w, inp):
    t = torch()
    dev = {n: to_device(inp[n], "bf16") for n in ("x_q", "x_kv", "wq", "wk", "wv", "wo")}
    gamma = t.from_numpy(inp["gamma"]).cuda()
    beta = t.from_numpy(inp["beta"]).cuda()
    kl = keylens_device(inp["key_lens"])
    y = hattn.mha_fwd(dev["x_q"], dev["x_kv"], dev["wq"], dev["wk"], dev["wv"], dev["wo"], gamma,
                      beta, inp["eps"], w.h, mask_kind=w.mask_kind, key_lens=kl)
    t.cuda.synchronize()
    assert hattn.check_device_error() == 0
    return from_device(y)


def oracle_mha(w, inp):
    wd = {n: synth.widen(inp[n], "bf16") for n in ("x_q", "x_kv", "wq", "wk", "wv", "wo")}
    return oracle.mha(wd["x_q"], wd["x_kv"], wd["wq"], wd["wk"], wd["wv"], wd["wo"],
                      inp["gamma"].astype(np.float64), inp["beta"].astype(np.float64), inp["eps"],
                      w.h, w.mask_kind, inp["key_lens"])


def test_named_mha_full_parity():
    w = synth.workload("mha_bf16")
    inp = synth.mha_inputs(w)
    assert_close(run_mha(w, inp), oracle_mha(w, inp), "bf16", w.name)


@pytest.mark.parametrize("B,n_q,n_k,d_model,h,d,mask_kind,cross", [
    (3, 100, 300, 256, 4, 64, synth.MASK_KEY_PADDING, True),
    (2, 200, 200, 512, 4, 128, synth.MASK_CAUSAL, False),
    (1, 77, 77, 128, 2, 64, synth.MASK_NONE, False),
    (2, 129, 129, 192, 3, 64, synth.MASK_CAUSAL | synth.MASK_KEY_PADDING, False),
    (1, 1, 5, 64, 1, 64, synth.MASK_NONE, True),
])
def test_mha_shapes(B, n_q, n_k, d_model, h, d, mask_kind, cross):
    w = synth.Workload("mha_sweep", "bf16", B=B, h=h, n_q=n_q, n_k=n_k, d_k=d, d_v=d,
                       mask_kind=mask_kind, seed=500 + n_q + d_model, key_len_range=(1, n_k),
                       d_model=d_model, kind="mha")
    inp = synth.mha_inputs(w, self_attention=not cross)
    rng = np.random.default_rng(7)
    inp["gamma"] = rng.uniform(0.5, 1.5, d_model).astype(np.float32)
    inp["beta"] = rng.uniform(-0.5, 0.5, d_model).astype(np.float32)
    assert_close(run_mha(w, inp), oracle_mha(w, inp), "bf16", f"mha {B} {n_q} {n_k} {d_model}")


def test_mha_several_row_tiles_per_cta():
    # 24 x 1024 rows: 192 row tiles of 128, so every CTA pair of the LayerNorm GEMM takes
    # two or three tiles (both exchange barriers, several phases each) and the projection
    # GEMM's CTAs take up to ten. No row depends on which CTA or tile computed it, so the
    # result must equal, bit for bit, three launches of 8 x 1024 rows (one row tile per
    # CTA pair); one of those is held to the oracle.
    w = synth.Workload("mha_many_tiles", "bf16", B=24, h=8, n_q=1024, n_k=1024, d_k=64, d_v=64,
                       mask_kind=synth.MASK_NONE, seed=612, d_model=512, kind="mha")
    inp = synth.mha_inputs(w)
    y_all = run_mha(w, inp)
    for k in range(3):
        wk = synth.Workload("mha_many_tiles", "bf16", B=8, h=8, n_q=1024, n_k=1024, d_k=64, d_v=64,
                            mask_kind=synth.MASK_NONE, seed=612, d_model=512, kind="mha")
        part = dict(inp)
        part["x_q"] = part["x_kv"] = inp["x_q"][8 * k:8 * k + 8]
        y_k = run_mha(wk, part)
        # (bf16 results widened exactly to fp64: equal arrays are equal bits)
        assert np.array_equal(y_all[8 * k:8 * k + 8], y_k), f"rows of batch slice {k} differ"
        if k == 0:
            assert_close(y_k, oracle_mha(wk, part), "bf16", "mha 8 x 1024")
