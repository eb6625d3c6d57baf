/*
 * hattn — multi-head scaled dot-product attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libhattn.so. Every entry point takes plain pointers and sizes; no
 * PyTorch or C++ types cross this boundary. The caller owns every buffer and
 * the stream. All compute entry points are asynchronous: a return of HATTN_OK
 * means "validated and enqueued on `stream`"; device-side conditions (a bad
 * key length, a pipeline wait that gave up) are reported later by
 * hattn_check_device_error().
 *
 * Sources for the operations (explanatory pages on "Attention Is All You
 * Need"):
 *   [P1] hex4c59.cc, "读懂 Attention Is All You Need：从一次加权求和到完整
 *        Transformer"
 *   [P4] devpress.csdn.net, "【深度学习】Transformer（Attention Is All You Need）"
 *
 * Layout. Activations are row-major [B, n, h, d]: head i of token t of batch
 * element b is the d-vector starting at element ((b*n + t)*h + i)*d. This is
 * the concatenation of heads along the feature axis, i.e. exactly the
 * row-major [B*n, h*d] matrix that X.W produces ([P1] §多头注意力让一次读取
 * 有多组投影: head outputs are concatenated along the feature dimension).
 */
#ifndef HATTN_H
#define HATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* hattn_stream_t;

/* Element types. */
#define HATTN_F32 0  /* fp32 in, fp32 out, fp32 arithmetic                    */
#define HATTN_BF16 1 /* bf16 in, bf16 out, fp32 accumulation                   */

/* mask_kind bits; they may be combined. */
#define HATTN_MASK_NONE 0
#define HATTN_MASK_CAUSAL 1      /* key j invisible to query t when j > t      */
#define HATTN_MASK_KEY_PADDING 2 /* key j invisible when j >= key_lens[b]      */

/* Status codes (0 or negative). */
#define HATTN_OK 0
#define HATTN_EINVAL (-1)       /* null pointer, bad size, bad mask bits, misaligned pointer */
#define HATTN_EUNSUPPORTED (-2) /* a valid request no kernel here implements          */
#define HATTN_ECUDA (-3)        /* a CUDA runtime/driver call failed (launch, tensor map) */
#define HATTN_ETIMEOUT (-4)     /* device: a pipeline wait gave up (reported asynchronously) */
#define HATTN_EKEYLEN (-5)      /* device: key_lens[b] outside [1, n_k] (reported asynchronously) */
#define HATTN_EWORKSPACE (-6)   /* workspace NULL or smaller than mha_workspace_bytes()   */
#define HATTN_ESCRATCH (-7)     /* problem needs more scratch than mha_fwd_noalloc's static buffer */

/*
 * attn_fwd — multi-head scaled dot-product attention,
 *     out[b,t,i,:] = sum_j softmax_j( scale * q[b,t,i,:].k[b,j,i,:] ) v[b,j,i,:]
 * over the keys j visible to query t.
 *
 * Defined in [P1] §六步算完一行注意力 (dot products, scaling, row softmax,
 * weighted sum of values) and §把所有位置合并，就是那条核心公式
 * (Attention(Q,K,V) = softmax(QK^T/sqrt(d_k))V); masking before the softmax in
 * [P1] §掩码必须在 softmax 之前生效 and [P4] §3.1 (triu -inf, diagonal
 * visible); cross-attention with n_q != n_k in [P1] §解码器有两种读取 and
 * [P4] §3.2. A masked key gets weight exactly 0.
 *
 *   q        device, [B, n_q, h, d_k], dtype elements, 16-byte aligned
 *   k        device, [B, n_k, h, d_k]
 *   v        device, [B, n_k, h, d_v]
 *   out      device, [B, n_q, h, d_v]; written, never read; must not overlap inputs
 *   dtype    HATTN_F32 or HATTN_BF16
 *   scale    multiplies q.k; normally 1/sqrt(d_k)
 *   mask_kind  bitwise OR of HATTN_MASK_*; CAUSAL requires n_q == n_k
 *   key_lens device int32[B], read only with HATTN_MASK_KEY_PADDING (else may
 *            be NULL). Each value must lie in [1, n_k]; a value outside makes
 *            the kernel zero that batch element's output and raise
 *            HATTN_EKEYLEN in the device error word.
 *   stream   the CUDA stream to enqueue on
 *
 * Supported: HATTN_F32 with d_k, d_v <= 128; HATTN_BF16 with d_k, d_v <= 256
 * (d_k == d_v in {64, 128} runs on the tensor-core kernel, other sizes on a
 * CUDA-core kernel). Returns HATTN_OK, HATTN_EINVAL, HATTN_EUNSUPPORTED or
 * HATTN_ECUDA; on an error return nothing was enqueued.
 * Allocates nothing; caches tensor-map descriptors per (pointer, shape).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, int dtype, int B, int h,
             int n_q, int n_k, int d_k, int d_v, float scale, int mask_kind,
             const int32_t* key_lens, hattn_stream_t stream);

/*
 * mha_fwd — the post-norm multi-head-attention sublayer,
 *     Q = x_q Wq,  K = x_kv Wk,  V = x_kv Wv                      (no biases)
 *     A = Concat_i attn(Q_i, K_i, V_i)        (scale 1/sqrt(d_k), mask_kind)
 *     y = LayerNorm(x_q + A Wo) * gamma + beta
 * with LayerNorm over the d_model features of each token, biased variance
 * and eps inside the square root.
 *
 * Defined in [P1] §Q、K、V 是三种计算角色 (Q = X W^Q, W^Q of shape
 * d_model x d_k per head), §多头注意力让一次读取有多组投影 (heads, concat,
 * W^O), §Add & Norm 里究竟发生了什么？ (LayerNorm(x + F(x)), post-LN) and
 * [P4] §2.2 (W^O of shape h*d_v x d_model).
 *
 *   x_q      device, [B, n_q, d_model] bf16
 *   x_kv     device, [B, n_k, d_model] bf16; pass x_q (and n_k = n_q) for self-attention
 *   Wq, Wk   device, [d_model, h*d_k] bf16 row-major; column block i is head i
 *   Wv       device, [d_model, h*d_v] bf16
 *   Wo       device, [h*d_v, d_model] bf16; row block i is head i
 *   gamma, beta  device, fp32 [d_model]
 *   eps      LayerNorm epsilon (> 0)
 *   y        device, [B, n_q, d_model] bf16 output
 *   dtype    HATTN_BF16 (the only type this entry point implements)
 *   workspace  device scratch of at least mha_workspace_bytes(...) bytes,
 *            256-byte aligned, owned by the caller, not used concurrently by
 *            another call; holds Q, K, V and the concatenated heads A.
 *
 * Supported: d_model a multiple of 64 and <= 512, d_k == d_v in {64, 128},
 * h*d_k a multiple of 64. Returns HATTN_OK, HATTN_EINVAL, HATTN_EUNSUPPORTED,
 * HATTN_EWORKSPACE or HATTN_ECUDA.
 */
int mha_fwd(const void* x_q, const void* x_kv, const void* Wq, const void* Wk, const void* Wv,
            const void* Wo, const float* gamma, const float* beta, float eps, void* y, int dtype,
            int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v, int mask_kind,
            const int32_t* key_lens, void* workspace, size_t ws_bytes, hattn_stream_t stream);

/*
 * mha_fwd_noalloc — mha_fwd for callers that must not allocate device memory.
 *
 * The explanatory pages have no counterpart to this entry point; it exists
 * for deployment. Some callers are not allowed to allocate device memory
 * themselves: a plugin inside a host process that owns the whole device-memory
 * budget, or latency-critical code that forbids allocation after start-up
 * (cudaMalloc can synchronise the device and can fail under memory pressure).
 * Such callers cannot provide the workspace mha_fwd needs. This entry point
 * takes the same arguments as mha_fwd minus the workspace and uses instead a
 * scratch buffer of HATTN_NOALLOC_SCRATCH_BYTES (32 MiB) that the library
 * holds as a static device array: every GPU that loads the library keeps those
 * 32 MiB until the process exits. It allocates no device memory: neither this
 * function nor anything it calls calls cudaMalloc, cudaFree or a device
 * allocator (only the host-side cache of tensor-map descriptors that every
 * entry point of this library shares may grow).
 *
 *   - The first call on a device looks up the buffer's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Null or misaligned buffers and a dtype other than HATTN_BF16 are
 *     reported first (HATTN_EINVAL / HATTN_EUNSUPPORTED, as mha_fwd reports
 *     them); then sizes whose mha_workspace_bytes() exceeds the buffer are
 *     rejected with HATTN_ESCRATCH before anything is enqueued (the B=16,
 *     n=512, d_model=512, h=8, d=64 sublayer needs exactly 32 MiB).
 *   - Every call shares the one buffer and overwrites it completely before
 *     reading it (nothing in it has to start at zero); calls whose work overlaps
 *     on the GPU (different streams, or different host threads) race on it and
 *     give undefined results. Serialise them, e.g. on one stream.
 * Other arguments, supported sizes and status codes are those of mha_fwd.
 */
#define HATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int mha_fwd_noalloc(const void* x_q, const void* x_kv, const void* Wq, const void* Wk,
                    const void* Wv, const void* Wo, const float* gamma, const float* beta,
                    float eps, void* y, int dtype, int B, int n_q, int n_k, int d_model, int h,
                    int d_k, int d_v, int mask_kind, const int32_t* key_lens,
                    hattn_stream_t stream);

/*
 * pos_encoding_fwd — sinusoidal positional encoding added to scaled embeddings,
 *     out[b,t,2i]   = emb_scale * emb[b,t,2i]   + sin((pos0 + t) / 10000^(2i/d_model))
 *     out[b,t,2i+1] = emb_scale * emb[b,t,2i+1] + cos((pos0 + t) / 10000^(2i/d_model))
 *
 * Defined in [P3] research-heat.pages.dev "做法 · Attention Is All You Need",
 * §去掉循环，因而须补回顺序 (the sin/cos formulas) and [P1] §没有循环，模型怎样
 * 知道词序？ (the embedding is multiplied by sqrt(d_model), then the encoding
 * is added); values tabulated in [P4] §四、位置编码, table 4.1.
 *
 *   emb      device [B, n, d_model] (dtype elements), or NULL for the encoding alone
 *   out      device [B, n, d_model]; may be the same buffer as emb (in place)
 *   dtype    HATTN_F32 or HATTN_BF16
 *   d_model  even; emb_scale normally sqrt(d_model); pos0 >= 0 is the position of row 0,
 *            and pos0 + n <= 2^24 (positions are exact fp32 integers in the kernel)
 * Pointers 8-byte aligned. The encoding term is within 1e-6 of the exact
 * sin/cos; the sum is rounded once to dtype. Returns HATTN_OK, HATTN_EINVAL or
 * HATTN_ECUDA; large problems run a bulk-copy pipeline whose bounded waits
 * raise HATTN_ETIMEOUT on the device error word if one ever gives up.
 */
int pos_encoding_fwd(const void* emb, void* out, int dtype, int B, int n, int d_model,
                     float emb_scale, int pos0, hattn_stream_t stream);

/*
 * attn_decode_fwd — one decoding step: a single new query per (batch, head)
 * attends over that sequence's first kv_lens[b] cached keys and values,
 *     out[b,0,i,:] = sum_{j < kv_lens[b]} softmax_j(scale * q[b,0,i,:].k[b,j,i,:]) v[b,j,i,:]
 * (the same attention as attn_fwd with n_q = 1 and key padding).
 *
 * Defined by the autoregressive generation of [P1] §训练能并行，不意味着一次生成
 * 整句话 (each step predicts from the prefix produced so far) and
 * [research-heat] §解码器不能看见尚未写出的词 (generation proceeds word by word);
 * the attention itself is [P1] §六步算完一行注意力.
 *
 *   q        device [B, 1, h, d] bf16;   out device [B, 1, h, d] bf16
 *   k_cache, v_cache  device [B, n_max, h, d] bf16 (rows >= kv_lens[b] are not read)
 *   kv_lens  device int32[B], each in [1, n_max]; a value outside zeroes that
 *            output and raises HATTN_EKEYLEN in the device error word
 *   workspace  device scratch of attn_decode_workspace_bytes() bytes (16-byte
 *            aligned, caller-owned, not shared with a concurrent call)
 * Supported: dtype HATTN_BF16, d in {64, 128, 256}; pointers 16-byte aligned.
 * Returns HATTN_OK, HATTN_EINVAL, HATTN_EUNSUPPORTED, HATTN_EWORKSPACE or HATTN_ECUDA.
 */
int attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, void* out, int dtype,
                    int B, int h, int n_max, int d, float scale, const int32_t* kv_lens,
                    void* workspace, size_t ws_bytes, hattn_stream_t stream);

/* Bytes of workspace attn_decode_fwd needs for these sizes (0 on bad sizes). */
size_t attn_decode_workspace_bytes(int B, int h, int n_max, int d);

/*
 * attn_fwd_lse — attn_fwd that also writes, for every (b, i, t), the natural
 * log-sum-exp of the scaled scores over the visible keys,
 *     lse[(b*h + i)*n_q + t] = ln sum_j exp(scale * q_t . k_j)    (fp32 [B, h, n_q]),
 * which the backward pass uses to recompute the attention weights
 * exp(scale q.k - lse). Same arguments, constraints and returns as attn_fwd;
 * lse must be 16-byte aligned. A batch element with an invalid key length gets
 * lse = -inf (and zero output) and HATTN_EKEYLEN.
 */
int attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int dtype,
                 int B, int h, int n_q, int n_k, int d_k, int d_v, float scale, int mask_kind,
                 const int32_t* key_lens, hattn_stream_t stream);

/*
 * attn_bwd — gradients of multi-head attention: given dout = dL/dout for
 * out = attn_fwd(q, k, v), writes dq, dk, dv (the layouts and dtype of q, k, v):
 *     P = exp(scale q.k - lse),  D_t = dout_t . out_t,  dS = P (dout.v - D)
 *     dv_j = sum_t P_tj dout_t,  dk_j = scale sum_t dS_tj q_t,  dq_t = scale sum_j dS_tj k_j
 * Training sends the loss gradient back through the attention weights ([P1]
 * §参数是怎样学出来的？); these are the chain rule applied to the definition of
 * attn_fwd. out and lse must come from attn_fwd_lse with the same inputs, scale
 * and mask. bf16 with d_k == d_v in {64, 128} and scale > 0 runs on the tensor
 * cores (bf16 P and dS, fp32 accumulation); every other shape attn_fwd accepts
 * runs on CUDA cores in fp32.
 *   workspace  attn_bwd_workspace_bytes(B, h, n_q) bytes, 256-byte aligned
 *              (fp32 D and base-2 log-sum-exp per row, rows padded to 128)
 * Returns HATTN_OK, HATTN_EINVAL, HATTN_EUNSUPPORTED, HATTN_EWORKSPACE or
 * HATTN_ECUDA; a bad key length zeroes that batch element's gradients and raises
 * HATTN_EKEYLEN on the device error word.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int dtype, int B, int h, int n_q,
             int n_k, int d_k, int d_v, float scale, int mask_kind, const int32_t* key_lens,
             void* workspace, size_t ws_bytes, hattn_stream_t stream);

size_t attn_bwd_workspace_bytes(int B, int h, int n_q);

/* Bytes of caller-owned workspace mha_fwd needs for these sizes (0 on bad sizes). */
size_t mha_workspace_bytes(int dtype, int B, int n_q, int n_k, int d_model, int h, int d_k,
                           int d_v);

/*
 * ffn_fwd — the post-norm position-wise feed-forward sublayer,
 *     y = LayerNorm(x + max(0, x W1 + b1) W2 + b2) * gamma + beta   (row by row)
 *
 * Defined in [P4] §2.3 (x + FFN(x) = x + max(0, x W1 + b1) W2 + b2, then norm2) and
 * [P1] §前馈网络为什么放在注意力后面？ (the same FFN for every position; ReLU;
 * 512 -> 2048 -> 512 in the base model).
 *
 *   x      device [M, d_model] (M = B * n rows; rows are independent)
 *   W1     device [d_model, d_ff] row-major;  b1 fp32 [d_ff] or NULL (zero bias)
 *   W2     device [d_ff, d_model] row-major;  b2 fp32 [d_model] or NULL
 *   gamma, beta  fp32 [d_model];  eps > 0
 *   y      device [M, d_model] (must not alias x)
 *   workspace  device scratch of ffn_workspace_bytes() bytes, 256-byte aligned,
 *          caller-owned; holds the hidden activations max(0, x W1 + b1) in bf16
 * Supported: dtype HATTN_BF16; d_model a multiple of 64 and <= 512; d_ff a
 * multiple of 64; every pointer 16-byte aligned. fp32 accumulation; the
 * hidden activations are rounded to bf16 once, y once.
 * Returns HATTN_OK, HATTN_EINVAL, HATTN_EUNSUPPORTED, HATTN_EWORKSPACE or
 * HATTN_ECUDA; asynchronous on `stream`.
 */
int ffn_fwd(const void* x, const void* W1, const float* b1, const void* W2, const float* b2,
            const float* gamma, const float* beta, float eps, void* y, int dtype, int M,
            int d_model, int d_ff, void* workspace, size_t ws_bytes, hattn_stream_t stream);

/* Bytes of caller-owned workspace ffn_fwd needs for these sizes (0 on bad sizes). */
size_t ffn_workspace_bytes(int dtype, int M, int d_model, int d_ff);

/* Weights of one post-norm MHA sublayer (see mha_fwd): W^Q, W^K, W^V [d_model, h*d_k],
 * W^O [h*d_k, d_model] (dtype elements), LayerNorm gamma/beta fp32 [d_model]. */
typedef struct hattn_mha_weights {
    const void* Wq;
    const void* Wk;
    const void* Wv;
    const void* Wo;
    const float* gamma;
    const float* beta;
} hattn_mha_weights;

/* Weights of one feed-forward sublayer (see ffn_fwd). */
typedef struct hattn_ffn_weights {
    const void* W1;
    const float* b1;
    const void* W2;
    const float* b2;
    const float* gamma;
    const float* beta;
} hattn_ffn_weights;

/*
 * encoder_layer_fwd — one encoder layer: the MHA sublayer (self-attention) then
 * the feed-forward sublayer, each post-norm,
 *     y1 = LayerNorm1(x + MHA(x, x));  y = LayerNorm2(y1 + FFN(y1)).
 * Defined in [P1] §编码器：交互之后，还要逐位置处理信息 (two sublayers, each with
 * residual and LayerNorm) and [P4] §2.3 (the order self-attention -> norm1 ->
 * FFN -> norm2). key_lens (device int32 [B]) masks padded source positions as
 * keys (mask_kind HATTN_MASK_KEY_PADDING of mha_fwd), or NULL for none.
 * x, y: device [B, n, d_model]; the sublayer output y1 is rounded to bf16 (it is
 * the bf16 input of the second sublayer). workspace: encoder_layer_workspace_bytes()
 * bytes, 256-byte aligned. Constraints: those of mha_fwd (d_k in {64, 128}) and
 * ffn_fwd. Returns as mha_fwd / ffn_fwd.
 */
int encoder_layer_fwd(const void* x, const hattn_mha_weights* attn, const hattn_ffn_weights* ffn,
                      float eps, void* y, int dtype, int B, int n, int d_model, int h, int d_k,
                      int d_ff, const int32_t* key_lens, void* workspace, size_t ws_bytes,
                      hattn_stream_t stream);

size_t encoder_layer_workspace_bytes(int dtype, int B, int n, int d_model, int h, int d_k,
                                     int d_ff);

/*
 * decoder_layer_fwd — one decoder layer: masked self-attention, encoder-decoder
 * (cross) attention over the encoder output `memory`, then the feed-forward
 * sublayer, each post-norm:
 *     y1 = LN1(x + MHA_causal(x, x));  y2 = LN2(y1 + MHA(y1, memory));  y = LN3(y2 + FFN(y2)).
 * Defined in [P1] §解码器有两种读取：看前缀，以及看源句 (three sublayers, each with
 * its own Add & Norm; queries from the decoder, keys and values from the encoder
 * output) and the causal mask of §右移目标，是为了让输入与标签错开一位.
 *   x, y     device [B, n_tgt, d_model];  memory device [B, n_src, d_model]
 *   src_lens device int32 [B] (cross-attention key lengths) or NULL for none
 * workspace: decoder_layer_workspace_bytes() bytes, 256-byte aligned.
 * Returns as mha_fwd / ffn_fwd.
 */
int decoder_layer_fwd(const void* x, const void* memory, const hattn_mha_weights* self_attn,
                      const hattn_mha_weights* cross_attn, const hattn_ffn_weights* ffn, float eps,
                      void* y, int dtype, int B, int n_tgt, int n_src, int d_model, int h,
                      int d_k, int d_ff, const int32_t* src_lens, void* workspace,
                      size_t ws_bytes, hattn_stream_t stream);

size_t decoder_layer_workspace_bytes(int dtype, int B, int n_tgt, int n_src, int d_model, int h,
                                     int d_k, int d_ff);

/* Static text for a status code. */
const char* hattn_status_str(int status);

/*
 * Synchronises `stream`, then reads and clears the device error word that the
 * kernels of this library set on the current device. Returns HATTN_OK,
 * HATTN_ETIMEOUT, HATTN_EKEYLEN, or HATTN_ECUDA when the synchronisation
 * itself failed.
 */
int hattn_check_device_error(hattn_stream_t stream);

/* Library version, major*10000 + minor*100 + patch. */
int hattn_version(void);

/*
 * hattn_selftest_wait_timeout — exercises the failure path of the pipelines.
 *
 * Not an operation of the pages: a check that a device-side wait which never
 * completes ends by itself. It enqueues on `stream` one small kernel whose
 * single thread waits on a shared-memory barrier that nothing arrives on,
 * through the same bounded wait (about two seconds of SM clock cycles) that
 * every pipeline of this library uses. When the wait gives up the kernel sets
 * HATTN_ETIMEOUT in the device error word and returns normally: no trap, no
 * fault, and the CUDA context stays usable. Afterwards
 * hattn_check_device_error(stream) returns HATTN_ETIMEOUT (and clears it).
 * Returns HATTN_OK once the kernel is enqueued, or HATTN_ECUDA.
 */
int hattn_selftest_wait_timeout(hattn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HATTN_H */
