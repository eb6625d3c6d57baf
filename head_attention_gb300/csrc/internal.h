// Declarations shared between the C-ABI host code and the kernel translation
// units of libhattn.so. Nothing here is part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "hattn.h"

namespace hattn {

// One validated attention request (see attn_fwd in hattn.h).
struct AttnArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    int dtype;
    int B, h, n_q, n_k, d_k, d_v;
    float scale;
    int mask_kind;
    const int32_t* key_lens;
    cudaStream_t stream;
    int* err_word;     // device error word of the current device
    float* lse = nullptr;  // optional fp32 [B, h, n_q]: ln sum_j exp(scale q.k_j)
};

// Tensor maps of one attention call on the tensor-core path: Q, K, V viewed as
// 4-D [B][n][h][d] bf16 tensors, loaded as 128-row x 64-column boxes.
struct AttnMaps {
    CUtensorMap q, k, v;
    CUtensorMap o;  // the output, [B][n_q][h][d] (short-sequence kernel only)
};

// CUDA-core kernel: fp32 (d <= 128) and bf16 (d <= 256), any d_k / d_v.
cudaError_t launch_attn_simt(const AttnArgs& a);

// Tensor-core (tcgen05) kernel: bf16, d_k == d_v in {64, 128}.
// Streaming multiprocessors of the current device (152 on GB300 if the query fails).
int sm_count();

bool attn_tc_supported(const AttnArgs& a);
cudaError_t launch_attn_tc(const AttnArgs& a, const AttnMaps& maps);

// Tensor-core kernel for short sequences (one CTA per head, no work loop): bf16,
// n_q <= 128, d_k == d_v == 64 with n_k <= 256 or d_k == d_v == 128 with n_k <= 128.
// Needs maps.o as well.
bool attn_short_supported(const AttnArgs& a);
cudaError_t launch_attn_short(const AttnArgs& a, const AttnMaps& maps);

// Encodes a tensor map through the driver entry point. Returns false on failure.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

// [B][n][h][d] bf16 tensor as a 4-D map with 64-element x `box_rows` boxes,
// 128-byte swizzle, zero fill past n within each batch element.
bool make_bnhd_map(CUtensorMap* map, const void* base, int B, int n, int h, int d, int box_rows);

// Attention backward: dQ, dK, dV from Q, K, V, O, dO and the forward's row
// log-sum-exp. Scratch (fp32, rows padded to nqp = n_q rounded up to 128), both
// written negated by the preparation kernel: dsum [B, h, nqp] = -(dO . O) (0
// past n_q) and lse2 [B, h, nqp] = -lse * log2(e) (-inf past n_q).
struct AttnBwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* out;
    const void* dout;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    float* dsum;
    float* lse2;
    int dtype;
    int B, h, n_q, n_k, d_k, d_v;
    float scale;
    int mask_kind;
    const int32_t* key_lens;
    cudaStream_t stream;
    int* err_word;
};
cudaError_t launch_attn_bwd_prep(const AttnBwdArgs& a);
cudaError_t launch_attn_bwd_simt(const AttnBwdArgs& a);  // CUDA cores, any supported shape
bool attn_bwd_tc_supported(const AttnBwdArgs& a);          // bf16, d_k == d_v in {64, 128}
cudaError_t launch_attn_bwd_tc(const AttnBwdArgs& a, const AttnMaps& maps, const CUtensorMap& tm_dout);

// Sinusoidal positional encoding added to scaled embeddings (emb may be NULL).
cudaError_t launch_pos_encoding(const void* emb, void* out, int dtype, int B, int n, int d_model,
                                float emb_scale, int pos0, int* err_word, cudaStream_t stream);

// Decode attention: one query per (b, h) over a per-sequence K/V prefix.
struct DecodeLaunch {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    const int32_t* kv_lens;
    void* workspace;  // fp32 partials [B, h, splits, d + 2]
    int B, h, n_max, d, splits, chunk;
    float scale;
    cudaStream_t stream;
    int* err_word;
};
void decode_split_plan(int B, int h, int n_max, int* splits, int* chunk);
cudaError_t launch_attn_decode(const DecodeLaunch& a);

// ---- tcgen05 GEMMs of the MHA sublayer

// One output problem of the projection GEMM: C[M, N] = A[M, K] . W[K, N] (bf16, row-major).
struct ProjProblem {
    CUtensorMap a;  // A [M][K], 64 x 128 boxes, K-major
    CUtensorMap w;  // W [K][N], 64 x 64 boxes, N-major
    CUtensorMap cmap;  // C [M][N], 64 x 32 boxes: the output, stored by TMA (one box per epilogue warp)
    void* c;        // bf16 [M][N]
    int M, N, K;
    const float* bias = nullptr;  // optional fp32 [N], added to every row
    bool relu = false;            // max(0, .) after the bias
};

// Up to three independent projection GEMMs in one launch (Q, K, V).
cudaError_t launch_proj_gemm(const ProjProblem* problems, int count, cudaStream_t stream,
                             int* err_word);

// y = LayerNorm(x + A . Wo [+ bias]) * gamma + beta over rows of length N = d_model.
struct OutProjLnArgs {
    CUtensorMap a;   // A [M][K] bf16, K-major boxes 64 x 128
    CUtensorMap wo;  // Wo [K][N] bf16, N-major boxes 64 x 64
    const void* x;   // residual, bf16 [M][N]
    CUtensorMap xmap;  // the residual as 64 x 128 boxes (loaded into shared memory by TMA)
    CUtensorMap ymap;  // the output as 64 x 32 boxes (each epilogue warp stores its rows by TMA)
    const float* gamma;
    const float* beta;
    float eps;
    void* y;  // bf16 [M][N]
    int M, N, K;
    const float* bias = nullptr;  // optional fp32 [N], added before the residual
};
cudaError_t launch_outproj_ln(const OutProjLnArgs& args, cudaStream_t stream, int* err_word);

}  // namespace hattn
