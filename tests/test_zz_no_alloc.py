"""mha_fwd_noalloc: the MHA sublayer for callers that may not allocate device
memory (the library supplies its own static 32 MiB scratch instead of a
caller-provided workspace).

It must give the same result as mha_fwd with a caller-provided workspace,
call after call, although every call reuses the same static buffer. This file
is collected last so that a failure here does not stop the other tests of a
run that stops at the first failure.
"""

import numpy as np
import pytest

import head_attention_gb300 as hattn
from synth import inputs as synth
from tests.gpu_util import assert_close, from_device, to_device, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name_or_shape", ["mha_bf16", (3, 100, 300, 256, 4, 64, 2)])
def test_noalloc_matches_workspace_entry_point_twice(name_or_shape):
    t = torch()
    hattn.build()
    if isinstance(name_or_shape, str):
        w = synth.workload(name_or_shape)
        inp = synth.mha_inputs(w)
    else:
        B, n_q, n_k, dm, h, d, mask = name_or_shape
        w = synth.Workload("noalloc_cross", "bf16", B=B, h=h, n_q=n_q, n_k=n_k, d_k=d, d_v=d,
                           mask_kind=mask, seed=77, key_len_range=(1, n_k), d_model=dm, kind="mha")
        inp = synth.mha_inputs(w, self_attention=False)
    dev = {n: to_device(inp[n], "bf16") for n in ("x_q", "x_kv", "wq", "wk", "wv", "wo")}
    gamma = t.from_numpy(inp["gamma"]).cuda()
    beta = t.from_numpy(inp["beta"]).cuda()
    kl = None if inp["key_lens"] is None else t.from_numpy(inp["key_lens"]).cuda()
    args = (dev["x_q"], dev["x_kv"], dev["wq"], dev["wk"], dev["wv"], dev["wo"], gamma, beta,
            inp["eps"])
    dims = (w.B, w.n_q, w.n_k, w.d_model, w.h, w.d_k, w.d_v)

    ref = hattn.mha_fwd(*args, w.h, mask_kind=w.mask_kind, key_lens=kl)
    for _ in range(2):
        y = t.full_like(ref, float("nan"))
        rc = hattn.mha_fwd_noalloc_raw(*args, y, hattn.HATTN_BF16, *dims, w.mask_kind, kl, None)
        assert rc == 0, hattn.status_str(rc)
        t.cuda.synchronize()
        assert hattn.check_device_error() == 0
        assert_close(from_device(y), from_device(ref), "bf16", "noalloc vs workspace")
