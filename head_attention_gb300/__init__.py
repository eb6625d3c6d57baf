"""hattn: multi-head scaled dot-product attention for NVIDIA GB300 (sm_103a).

The compute path is libhattn.so (hand-written tcgen05/TMA CUDA kernels behind
a C ABI declared in include/hattn.h); this package only builds it and binds it.
"""

from ._binding import (  # noqa: F401
    EXPORTED,
    HATTN_BF16,
    HATTN_F32,
    MASK_CAUSAL,
    MASK_KEY_PADDING,
    MASK_NONE,
    HattnError,
    attn_bwd,
    attn_bwd_raw,
    attn_bwd_workspace_bytes,
    attn_decode_fwd,
    attn_decode_fwd_raw,
    attn_decode_workspace_bytes,
    attn_fwd,
    attn_fwd_lse,
    attn_fwd_lse_raw,
    attn_fwd_raw,
    check_device_error,
    decoder_layer_fwd,
    decoder_layer_fwd_raw,
    decoder_layer_workspace_bytes,
    encoder_layer_fwd,
    encoder_layer_fwd_raw,
    encoder_layer_workspace_bytes,
    ffn_fwd,
    ffn_fwd_raw,
    ffn_weights,
    ffn_workspace_bytes,
    load,
    mha_fwd,
    mha_weights,
    mha_fwd_noalloc_raw,
    mha_fwd_raw,
    mha_workspace_bytes,
    pos_encoding_fwd,
    pos_encoding_fwd_raw,
    status_str,
    version,
)
from .builder import build  # noqa: F401
