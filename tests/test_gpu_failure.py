"""Failure detection on the GPU without a fault: a device wait that never
completes gives up by itself, reports HATTN_ETIMEOUT through the device error
word, and leaves the CUDA context usable for the next call."""

import time

import pytest

import head_attention_gb300 as hattn
import oracle
from synth import inputs as synth
from tests.gpu_util import assert_close, from_device, to_device, torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    t = torch()
    hattn.build()
    assert hattn.check_device_error() == hattn.OK
    t0 = time.monotonic()
    assert hattn.selftest_wait_timeout() == hattn.OK
    assert hattn.check_device_error() == hattn.ETIMEOUT
    waited = time.monotonic() - t0
    # The limit is a few billion SM cycles: on the order of seconds, not forever.
    assert 0.1 < waited < 30.0, waited
    # Read once, the word is clear again.
    assert hattn.check_device_error() == hattn.OK
    # The context still runs real work, and correctly.
    w = synth.Workload("after_timeout", "bf16", B=1, h=2, n_q=130, n_k=130, d_k=64, d_v=64,
                       mask_kind=hattn.MASK_CAUSAL, seed=11)
    inp = synth.attn_inputs(w)
    q, k, v = (to_device(inp[n], w.dtype) for n in ("q", "k", "v"))
    out = hattn.attn_fwd(q, k, v, scale=w.scale, mask_kind=w.mask_kind)
    t.cuda.synchronize()
    assert hattn.check_device_error() == hattn.OK
    wq, wk, wv = (synth.widen(inp[n], w.dtype) for n in ("q", "k", "v"))
    ref = oracle.attn(wq, wk, wv, w.scale, w.mask_kind, inp["key_lens"])
    assert_close(from_device(out), ref, "bf16", "attention after a timeout")
