"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every declared symbol, and rejects bad arguments before touching the
device (a rejected call enqueues nothing, so none of these reach CUDA)."""

import os
import re

import pytest

import head_attention_gb300 as hattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    hattn.build()
    return hattn.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hattn.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(hattn.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert hattn.status_str(code) not in ("", "unknown status")
    assert hattn.status_str(12345) == "unknown status"
    assert hattn.version() >= 100


A = 0x10000  # 16-byte aligned fake device addresses: validation never dereferences them
GOOD = dict(q=A, k=2 * A, v=3 * A, out=4 * A, dtype=1, B=2, h=4, n_q=128, n_k=128, d_k=64, d_v=64,
            scale=0.125, mask_kind=0, key_lens=None, stream=0)


def call(**kw):
    args = dict(GOOD)
    args.update(kw)
    return hattn.attn_fwd_raw(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), hattn._binding.EINVAL),
    (dict(out=None), hattn._binding.EINVAL),
    (dict(B=0), hattn._binding.EINVAL),
    (dict(h=-1), hattn._binding.EINVAL),
    (dict(n_q=0), hattn._binding.EINVAL),
    (dict(d_v=0), hattn._binding.EINVAL),
    (dict(dtype=7), hattn._binding.EINVAL),
    (dict(mask_kind=4), hattn._binding.EINVAL),
    (dict(mask_kind=1, n_k=127), hattn._binding.EINVAL),        # causal needs n_q == n_k
    (dict(mask_kind=2, key_lens=None), hattn._binding.EINVAL),  # padding needs key_lens
    (dict(q=A + 8), hattn._binding.EINVAL),                     # misaligned
    (dict(out=A + 2), hattn._binding.EINVAL),
    (dict(d_k=60, d_v=60), hattn._binding.EINVAL),              # row not a multiple of 16 bytes
    (dict(scale=float("nan")), hattn._binding.EINVAL),
    (dict(scale=float("inf")), hattn._binding.EINVAL),
    (dict(dtype=0, d_k=192, d_v=192), hattn._binding.EUNSUPPORTED),
    (dict(d_k=512, d_v=512), hattn._binding.EUNSUPPORTED),
])
def test_attn_fwd_rejects_bad_arguments(lib, kw, code):
    assert call(**kw) == code


MHA = dict(x_q=A, x_kv=A, wq=2 * A, wk=3 * A, wv=4 * A, wo=5 * A, gamma=6 * A, beta=7 * A, eps=1e-6,
           y=8 * A, dtype=1, B=16, n_q=512, n_k=512, d_model=512, h=8, d_k=64, d_v=64, mask_kind=0,
           key_lens=None, workspace=0x100000, ws_bytes=1 << 40, stream=0)


def mha_call(**kw):
    args = dict(MHA)
    args.update(kw)
    return hattn.mha_fwd_raw(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(x_q=None), hattn._binding.EINVAL),
    (dict(gamma=None), hattn._binding.EINVAL),
    (dict(dtype=0), hattn._binding.EUNSUPPORTED),
    (dict(dtype=3), hattn._binding.EINVAL),
    (dict(eps=0.0), hattn._binding.EINVAL),
    (dict(eps=float("nan")), hattn._binding.EINVAL),
    (dict(mask_kind=1, n_k=256), hattn._binding.EINVAL),
    (dict(wo=5 * A + 4), hattn._binding.EINVAL),
    (dict(d_k=32, d_v=32), hattn._binding.EUNSUPPORTED),
    (dict(d_model=1024), hattn._binding.EUNSUPPORTED),
    (dict(d_model=500), hattn._binding.EUNSUPPORTED),
    (dict(workspace=None), hattn._binding.EWORKSPACE),
    (dict(workspace=0x100010), hattn._binding.EWORKSPACE),   # not 256-byte aligned
    (dict(ws_bytes=1024), hattn._binding.EWORKSPACE),
])
def test_mha_fwd_rejects_bad_arguments(lib, kw, code):
    assert mha_call(**kw) == code


def test_workspace_size_is_q_k_v_and_heads(lib):
    # Q, K, V, A in bf16, each region rounded up to 256 bytes.
    n = hattn.mha_workspace_bytes(1, 16, 512, 512, 512, 8, 64, 64)
    assert n == 4 * 16 * 512 * 512 * 2
    n2 = hattn.mha_workspace_bytes(1, 1, 3, 5, 64, 1, 64, 64)
    up = lambda x: (x + 255) // 256 * 256
    assert n2 == up(3 * 64 * 2) + 2 * up(5 * 64 * 2) + up(3 * 64 * 2)
    assert hattn.mha_workspace_bytes(0, 16, 512, 512, 512, 8, 64, 64) == 0
    assert hattn.mha_workspace_bytes(1, 0, 512, 512, 512, 8, 64, 64) == 0


def test_noalloc_rejects_problems_beyond_its_static_scratch(lib):
    # Checked before any CUDA call, so it runs without a GPU.
    args = dict(MHA)
    del args["workspace"], args["ws_bytes"]
    assert hattn.mha_workspace_bytes(1, 16, 512, 512, 512, 8, 64, 64) == hattn._binding.NOALLOC_SCRATCH_BYTES
    args.update(B=17)
    assert hattn.mha_fwd_noalloc_raw(**args) == hattn._binding.ESCRATCH
    args.update(B=16, n_q=1024, n_k=1024)
    assert hattn.mha_fwd_noalloc_raw(**args) == hattn._binding.ESCRATCH


def test_noalloc_reports_bad_buffers_before_the_size(lib):
    # An oversized call with a missing or misaligned buffer, or a wrong dtype, is
    # reported as that argument error, not as a scratch shortage.
    args = dict(MHA)
    del args["workspace"], args["ws_bytes"]
    args.update(B=17)
    assert hattn.mha_fwd_noalloc_raw(**dict(args, y=None)) == hattn._binding.EINVAL
    assert hattn.mha_fwd_noalloc_raw(**dict(args, x_q=args["x_q"] + 8)) == hattn._binding.EINVAL
    assert hattn.mha_fwd_noalloc_raw(**dict(args, dtype=0)) == hattn._binding.EUNSUPPORTED
    assert hattn.mha_fwd_noalloc_raw(**dict(args, dtype=7)) == hattn._binding.EINVAL


@pytest.mark.parametrize("kw,code", [
    (dict(out=None), hattn._binding.EINVAL),
    (dict(dtype=5), hattn._binding.EINVAL),
    (dict(d_model=63), hattn._binding.EINVAL),
    (dict(n=0), hattn._binding.EINVAL),
    (dict(pos0=-1), hattn._binding.EINVAL),
    (dict(pos0=(1 << 24) - 15), hattn._binding.EINVAL),
    (dict(out=A + 4), hattn._binding.EINVAL),
    (dict(emb_scale=float("nan")), hattn._binding.EINVAL),
])
def test_pos_encoding_rejects_bad_arguments(lib, kw, code):
    args = dict(emb=None, out=A, dtype=1, B=2, n=16, d_model=64, emb_scale=8.0, pos0=0, stream=0)
    args.update(kw)
    assert hattn.pos_encoding_fwd_raw(**args) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), hattn._binding.EINVAL),
    (dict(kv_lens=None), hattn._binding.EINVAL),
    (dict(dtype=0), hattn._binding.EUNSUPPORTED),
    (dict(d=96), hattn._binding.EUNSUPPORTED),
    (dict(n_max=0), hattn._binding.EINVAL),
    (dict(k_cache=A + 8), hattn._binding.EINVAL),
    (dict(workspace=None), hattn._binding.EWORKSPACE),
    (dict(ws_bytes=16), hattn._binding.EWORKSPACE),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    args = dict(q=A, k_cache=2 * A, v_cache=3 * A, out=4 * A, dtype=1, B=2, h=4, n_max=512, d=128,
                scale=0.088, kv_lens=5 * A, workspace=6 * A, ws_bytes=1 << 30, stream=0)
    args.update(kw)
    assert hattn.attn_decode_fwd_raw(**args) == code


def test_decode_workspace_size():
    n = hattn.attn_decode_workspace_bytes(32, 32, 8192, 128)
    assert n > 0 and n % (4 * 130) == 0
    assert hattn.attn_decode_workspace_bytes(1, 1, 1, 128) == 4 * 130
    assert hattn.attn_decode_workspace_bytes(1, 1, 1, 100) == 0


FFN_GOOD = dict(x=A, w1=2 * A, b1=3 * A, w2=4 * A, b2=5 * A, gamma=6 * A, beta=7 * A, eps=1e-6,
                y=8 * A, dtype=1, M=256, d_model=512, d_ff=2048, workspace=0x100000,
                ws_bytes=256 * 2048 * 2, stream=0)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), hattn._binding.EINVAL),
    (dict(w2=None), hattn._binding.EINVAL),
    (dict(gamma=None), hattn._binding.EINVAL),
    (dict(dtype=0), hattn._binding.EUNSUPPORTED),
    (dict(dtype=7), hattn._binding.EINVAL),
    (dict(M=0), hattn._binding.EINVAL),
    (dict(eps=0.0), hattn._binding.EINVAL),
    (dict(y=A), hattn._binding.EINVAL),            # y aliases x
    (dict(x=A + 8), hattn._binding.EINVAL),        # misaligned
    (dict(b1=3 * A + 4), hattn._binding.EINVAL),
    (dict(d_model=576), hattn._binding.EUNSUPPORTED),
    (dict(d_model=96), hattn._binding.EUNSUPPORTED),
    (dict(d_ff=100), hattn._binding.EUNSUPPORTED),
    (dict(workspace=None), hattn._binding.EWORKSPACE),
    (dict(workspace=0x100010), hattn._binding.EWORKSPACE),
    (dict(ws_bytes=256 * 2048 * 2 - 1), hattn._binding.EWORKSPACE),
])
def test_ffn_rejects_bad_arguments(lib, kw, code):
    args = dict(FFN_GOOD)
    args.update(kw)
    assert hattn.ffn_fwd_raw(**args) == code


def test_ffn_and_layer_workspace_sizes(lib):
    assert hattn.ffn_workspace_bytes(1, 8192, 512, 2048) == 8192 * 2048 * 2
    assert hattn.ffn_workspace_bytes(1, 3, 64, 64) == 512  # rounded up to 256 bytes
    assert hattn.ffn_workspace_bytes(0, 8192, 512, 2048) == 0
    mha = hattn.mha_workspace_bytes(1, 16, 512, 512, 512, 8, 64, 64)
    act = 16 * 512 * 512 * 2
    assert hattn.encoder_layer_workspace_bytes(1, 16, 512, 512, 8, 64, 2048) == max(
        mha, 8192 * 2048 * 2) + act
    cross = hattn.mha_workspace_bytes(1, 16, 512, 300, 512, 8, 64, 64)
    assert hattn.decoder_layer_workspace_bytes(1, 16, 512, 300, 512, 8, 64, 2048) == max(
        mha, cross, 8192 * 2048 * 2) + 2 * act
    assert hattn.encoder_layer_workspace_bytes(1, 0, 512, 512, 8, 64, 2048) == 0


def _weights():
    aw = hattn.mha_weights(2 * A, 3 * A, 4 * A, 5 * A, 6 * A, 7 * A)
    fw = hattn.ffn_weights(8 * A, 9 * A, 10 * A, 11 * A, 12 * A, 13 * A)
    return aw, fw


def test_layers_reject_bad_arguments(lib):
    aw, fw = _weights()
    ws = hattn.encoder_layer_workspace_bytes(1, 2, 128, 512, 8, 64, 2048)
    enc = dict(x=A, attn=aw, ffn=fw, eps=1e-6, y=20 * A, dtype=1, B=2, n=128, d_model=512, h=8,
               d_k=64, d_ff=2048, key_lens=None, workspace=0x1000000, ws_bytes=ws, stream=0)
    for kw, code in [(dict(x=None), hattn._binding.EINVAL), (dict(attn=None), hattn._binding.EINVAL),
                     (dict(ffn=None), hattn._binding.EINVAL), (dict(B=0), hattn._binding.EINVAL),
                     (dict(dtype=0), hattn._binding.EUNSUPPORTED),
                     (dict(ws_bytes=ws - 1), hattn._binding.EWORKSPACE),
                     (dict(workspace=0x1000010), hattn._binding.EWORKSPACE)]:
        args = dict(enc)
        args.update(kw)
        assert hattn.encoder_layer_fwd_raw(**args) == code, kw
    ws = hattn.decoder_layer_workspace_bytes(1, 2, 128, 96, 512, 8, 64, 2048)
    dec = dict(x=A, memory=30 * A, self_attn=aw, cross_attn=aw, ffn=fw, eps=1e-6, y=20 * A,
               dtype=1, B=2, n_tgt=128, n_src=96, d_model=512, h=8, d_k=64, d_ff=2048,
               src_lens=None, workspace=0x1000000, ws_bytes=ws, stream=0)
    for kw, code in [(dict(memory=None), hattn._binding.EINVAL),
                     (dict(cross_attn=None), hattn._binding.EINVAL),
                     (dict(n_src=0), hattn._binding.EINVAL),
                     (dict(ws_bytes=ws - 1), hattn._binding.EWORKSPACE)]:
        args = dict(dec)
        args.update(kw)
        assert hattn.decoder_layer_fwd_raw(**args) == code, kw


BWD_GOOD = dict(q=A, k=2 * A, v=3 * A, out=4 * A, dout=5 * A, lse=6 * A, dq=7 * A, dk=8 * A,
                dv=9 * A, dtype=1, B=2, h=4, n_q=128, n_k=128, d_k=64, d_v=64, scale=0.125,
                mask_kind=0, key_lens=None, workspace=0x100000, ws_bytes=2 * 2 * 4 * 128 * 4, stream=0)


@pytest.mark.parametrize("kw,code", [
    (dict(dout=None), hattn._binding.EINVAL),
    (dict(lse=None), hattn._binding.EINVAL),
    (dict(dk=None), hattn._binding.EINVAL),
    (dict(lse=6 * A + 4), hattn._binding.EINVAL),
    (dict(mask_kind=1, n_k=64), hattn._binding.EINVAL),
    (dict(mask_kind=2), hattn._binding.EINVAL),
    (dict(d_k=256, dtype=0), hattn._binding.EUNSUPPORTED),
    (dict(workspace=None), hattn._binding.EWORKSPACE),
    (dict(ws_bytes=2 * 2 * 4 * 128 * 4 - 4), hattn._binding.EWORKSPACE),
])
def test_attn_bwd_rejects_bad_arguments(lib, kw, code):
    args = dict(BWD_GOOD)
    args.update(kw)
    assert hattn.attn_bwd_raw(**args) == code


def test_attn_fwd_lse_rejects_bad_arguments(lib):
    args = dict(GOOD, lse=6 * A)
    assert hattn.attn_fwd_lse_raw(**dict(args, lse=None)) == hattn._binding.EINVAL
    assert hattn.attn_fwd_lse_raw(**dict(args, lse=6 * A + 8)) == hattn._binding.EINVAL
    assert hattn.attn_fwd_lse_raw(**dict(args, q=None)) == hattn._binding.EINVAL
    # Two fp32 arrays (D and the base-2 log-sum-exp) of B * h rows padded to 128.
    assert hattn.attn_bwd_workspace_bytes(2, 4, 128) == 2 * 4 * 2 * 4 * 128
    assert hattn.attn_bwd_workspace_bytes(1, 1, 1) == 2 * 4 * 128
    assert hattn.attn_bwd_workspace_bytes(1, 1, 129) == 2 * 4 * 256
