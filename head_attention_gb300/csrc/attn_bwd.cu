// Attention backward on CUDA cores (fp32 arithmetic, fp32 / bf16 in and out).
//
// Gradients of sum(dO * O), O = softmax(scale * Q K^T [masked]) V, per (batch,
// head), with the forward's row log-sum-exp lse_i = ln sum_j exp(scale q_i.k_j)
// (from attn_fwd_lse) so that P is recomputed exactly, not stored:
//   P_ij  = exp(scale q_i.k_j - lse_i)          (0 for masked keys)
//   D_i   = dO_i . O_i                          (= sum_j P_ij dP_ij)
//   dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
// Training sends the loss gradient back through the attention weights
// ("读懂 Attention Is All You Need", §参数是怎样学出来的？); the formulas are the
// chain rule applied to the forward definition (§六步算完一行注意力).
//
// Three kernels, no atomics: row_dot computes D; key_grads gives each CTA a
// block of keys of one (b, h) and streams the query rows through shared memory
// (dK, dV in registers); query_grads gives each CTA a block of queries and
// streams the keys (dQ in registers). Both recompute P and dP. Within a warp,
// a score phase puts one query (or key) per lane, and an accumulation phase puts
// the output columns on the lanes and broadcasts p / dS by shuffles.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kInner = 32;     // streamed rows per shared-memory tile (one per lane)

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const void* out;
    const void* dout;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    float* dsum;  // -D, fp32 [B, h, nqp]
    float* lse2;  // minus the base-2 log-sum-exp, fp32 [B, h, nqp]
    int B, h, n_q, n_k, d_k, d_v, nqp;
    float scale;
    int mask_kind;
    const int32_t* key_lens;
    int* err_word;
};

__device__ __forceinline__ int key_length(const BwdParams& p, int b)
{
    return (p.mask_kind & HATTN_MASK_KEY_PADDING) ? p.key_lens[b] : p.n_k;
}

// Copies rows [row0, row0 + rows) of one head (row stride h*d elements) into
// fp32 shared memory with row stride `ld`; rows past n are zero.
template <typename T>
__device__ __forceinline__ void stage(float* dst, int ld, const T* src, size_t stride, int row0,
                                      int rows, int n, int d)
{
    for (int idx = threadIdx.x; idx < rows * d; idx += kThreads) {
        const int r = idx / d, c = idx % d;
        dst[r * ld + c] = (row0 + r < n) ? to_f32(src[(size_t)(row0 + r) * stride + c]) : 0.0f;
    }
}

// -D_t = -(dO_t . O_t) and -lse2_t = -lse_t log2(e) for every (b, head, t)
// with t over the padded rows (0 and -inf past n_q); stored negated so that the
// kernels add them in packed fp32 instructions. A group of kL lanes (a power of
// two) covers one row with 16-byte loads, groups of a warp take consecutive
// rows, and the partial dot products meet by shuffles within the group.
template <typename T, int kL>
__global__ void __launch_bounds__(kThreads) row_dot_kernel(const BwdParams p)
{
    constexpr int kV = 16 / sizeof(T);  // elements per 16-byte load
    const int lane = threadIdx.x % 32, gl = lane % kL;
    const long long row = ((long long)blockIdx.x * kThreads + threadIdx.x) / kL;
    const long long rows = (long long)p.B * p.h * p.nqp;
    const bool in = row < rows;
    const int t = in ? static_cast<int>(row % p.nqp) : 0;
    const long long bh = in ? row / p.nqp : 0;
    const int head = static_cast<int>(bh % p.h), b = static_cast<int>(bh / p.h);
    float acc = 0.0f;
    if (in && t < p.n_q) {
        const size_t at = (((size_t)b * p.n_q + t) * p.h + head) * p.d_v;
        const T* o = static_cast<const T*>(p.out) + at;
        const T* g = static_cast<const T*>(p.dout) + at;
        for (int c = gl * kV; c < p.d_v; c += kL * kV) {
            const uint4 ov = *reinterpret_cast<const uint4*>(o + c);
            const uint4 gv = *reinterpret_cast<const uint4*>(g + c);
            const T* oe = reinterpret_cast<const T*>(&ov);
            const T* ge = reinterpret_cast<const T*>(&gv);
#pragma unroll
            for (int e = 0; e < kV; ++e) acc = fmaf(to_f32(oe[e]), to_f32(ge[e]), acc);
        }
    }
#pragma unroll
    for (int off = kL / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in && gl == 0) {
        p.dsum[row] = -acc;
        p.lse2[row] = t < p.n_q ? -p.lse[bh * p.n_q + t] * 1.4426950408889634f : -INFINITY;
    }
}

// dK and dV of kPW * 4 keys of one (b, h): the query rows stream through shared
// memory 32 at a time. kCols = output columns per lane (d <= 32 * kCols).
template <typename T, int kCols, int kPW>
__global__ void __launch_bounds__(kThreads) key_grads_kernel(const BwdParams p)
{
    constexpr int kKeys = 4 * kPW;
    extern __shared__ float smem[];
    const int dkp = p.d_k + 1, dvp = p.d_v + 1;
    float* k_s = smem;                    // [kKeys][dkp]
    float* v_s = k_s + kKeys * dkp;       // [kKeys][dvp]
    float* q_s = v_s + kKeys * dvp;       // [32][dkp]
    float* g_s = q_s + kInner * dkp;      // dO [32][dvp]
    float* lse_s = g_s + kInner * dvp;    // [32]
    float* d_s = lse_s + kInner;          // [32]

    const int key0 = blockIdx.x * kKeys, head = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;
    const size_t sk = (size_t)p.h * p.d_k, sv = (size_t)p.h * p.d_v;
    const T* qb = static_cast<const T*>(p.q) + (size_t)b * p.n_q * sk + (size_t)head * p.d_k;
    const T* kb = static_cast<const T*>(p.k) + (size_t)b * p.n_k * sk + (size_t)head * p.d_k;
    const T* vb = static_cast<const T*>(p.v) + (size_t)b * p.n_k * sv + (size_t)head * p.d_v;
    const T* gb = static_cast<const T*>(p.dout) + (size_t)b * p.n_q * sv + (size_t)head * p.d_v;
    T* dkb = static_cast<T*>(p.dk) + (size_t)b * p.n_k * sk + (size_t)head * p.d_k;
    T* dvb = static_cast<T*>(p.dv) + (size_t)b * p.n_k * sv + (size_t)head * p.d_v;
    const float* lse_b = p.lse + ((size_t)b * p.h + head) * p.n_q;
    const float* d_b = p.dsum + ((size_t)b * p.h + head) * p.nqp;

    const int kv_len = key_length(p, b);
    if (kv_len < 1 || kv_len > p.n_k) {
        for (int idx = threadIdx.x; idx < kKeys * p.d_k; idx += kThreads)
            if (key0 + idx / p.d_k < p.n_k) store_out(dkb + (size_t)(key0 + idx / p.d_k) * sk + idx % p.d_k, 0.0f);
        for (int idx = threadIdx.x; idx < kKeys * p.d_v; idx += kThreads)
            if (key0 + idx / p.d_v < p.n_k) store_out(dvb + (size_t)(key0 + idx / p.d_v) * sv + idx % p.d_v, 0.0f);
        if (threadIdx.x == 0) raise_device_error(p.err_word, HATTN_EKEYLEN);
        return;
    }

    stage<T>(k_s, dkp, kb, sk, key0, kKeys, p.n_k, p.d_k);
    stage<T>(v_s, dvp, vb, sv, key0, kKeys, p.n_k, p.d_v);

    float dk_acc[kPW][kCols], dv_acc[kPW][kCols];
#pragma unroll
    for (int u = 0; u < kPW; ++u)
#pragma unroll
        for (int m = 0; m < kCols; ++m) dk_acc[u][m] = dv_acc[u][m] = 0.0f;

    // Causal: queries before the first key of the block see none of its keys.
    const int q_first = causal ? (key0 / kInner) * kInner : 0;
    const bool any_key = key0 < kv_len;
    for (int qt = any_key ? q_first : p.n_q; qt < p.n_q; qt += kInner) {
        __syncthreads();  // the previous tile is no longer read
        stage<T>(q_s, dkp, qb, sk, qt, kInner, p.n_q, p.d_k);
        stage<T>(g_s, dvp, gb, sv, qt, kInner, p.n_q, p.d_v);
        if (threadIdx.x < kInner) {
            const int t = qt + threadIdx.x;
            lse_s[threadIdx.x] = t < p.n_q ? lse_b[t] : 0.0f;
            d_s[threadIdx.x] = t < p.n_q ? d_b[t] : 0.0f;
        }
        __syncthreads();
        const int t = qt + lane;  // this lane's query in the score phase
#pragma unroll
        for (int u = 0; u < kPW; ++u) {
            const int jl = warp * kPW + u, j = key0 + jl;
            const bool visible = t < p.n_q && j < kv_len && !(causal && j > t);
            float s = 0.0f, dp = 0.0f;
            const float* qr = q_s + lane * dkp;
            const float* kr = k_s + jl * dkp;
            for (int c = 0; c < p.d_k; ++c) s = fmaf(qr[c], kr[c], s);
            const float* gr = g_s + lane * dvp;
            const float* vr = v_s + jl * dvp;
            for (int c = 0; c < p.d_v; ++c) dp = fmaf(gr[c], vr[c], dp);
            const float pr = visible ? expf(p.scale * s - lse_s[lane]) : 0.0f;
            const float ds = pr * (dp + d_s[lane]);  // d_s holds -D
            for (int ii = 0; ii < kInner; ++ii) {
                const float pi = __shfl_sync(0xffffffffu, pr, ii);
                const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
                for (int m = 0; m < kCols; ++m) {
                    const int cc = lane + 32 * m;
                    if (cc < p.d_v) dv_acc[u][m] = fmaf(pi, g_s[ii * dvp + cc], dv_acc[u][m]);
                    if (cc < p.d_k) dk_acc[u][m] = fmaf(dsi, q_s[ii * dkp + cc], dk_acc[u][m]);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kPW; ++u) {
        const int j = key0 + warp * kPW + u;
        if (j >= p.n_k) continue;
#pragma unroll
        for (int m = 0; m < kCols; ++m) {
            const int cc = lane + 32 * m;
            if (cc < p.d_k) store_out(dkb + (size_t)j * sk + cc, p.scale * dk_acc[u][m]);
            if (cc < p.d_v) store_out(dvb + (size_t)j * sv + cc, dv_acc[u][m]);
        }
    }
}

// dQ of kPW * 4 queries of one (b, h): the keys stream through shared memory.
template <typename T, int kCols, int kPW>
__global__ void __launch_bounds__(kThreads) query_grads_kernel(const BwdParams p)
{
    constexpr int kRows = 4 * kPW;
    extern __shared__ float smem[];
    const int dkp = p.d_k + 1, dvp = p.d_v + 1;
    float* q_s = smem;                   // [kRows][dkp]
    float* g_s = q_s + kRows * dkp;      // dO [kRows][dvp]
    float* k_s = g_s + kRows * dvp;      // [32][dkp]
    float* v_s = k_s + kInner * dkp;     // [32][dvp]

    const int row0 = blockIdx.x * kRows, head = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;
    const size_t sk = (size_t)p.h * p.d_k, sv = (size_t)p.h * p.d_v;
    const T* qb = static_cast<const T*>(p.q) + (size_t)b * p.n_q * sk + (size_t)head * p.d_k;
    const T* kb = static_cast<const T*>(p.k) + (size_t)b * p.n_k * sk + (size_t)head * p.d_k;
    const T* vb = static_cast<const T*>(p.v) + (size_t)b * p.n_k * sv + (size_t)head * p.d_v;
    const T* gb = static_cast<const T*>(p.dout) + (size_t)b * p.n_q * sv + (size_t)head * p.d_v;
    T* dqb = static_cast<T*>(p.dq) + (size_t)b * p.n_q * sk + (size_t)head * p.d_k;
    const float* lse_b = p.lse + ((size_t)b * p.h + head) * p.n_q;
    const float* d_b = p.dsum + ((size_t)b * p.h + head) * p.nqp;

    const int kv_len = key_length(p, b);
    if (kv_len < 1 || kv_len > p.n_k) {
        for (int idx = threadIdx.x; idx < kRows * p.d_k; idx += kThreads)
            if (row0 + idx / p.d_k < p.n_q) store_out(dqb + (size_t)(row0 + idx / p.d_k) * sk + idx % p.d_k, 0.0f);
        return;  // the key-gradient kernel raises the error
    }

    stage<T>(q_s, dkp, qb, sk, row0, kRows, p.n_q, p.d_k);
    stage<T>(g_s, dvp, gb, sv, row0, kRows, p.n_q, p.d_v);
    float lse_r[kPW], d_r[kPW];
#pragma unroll
    for (int u = 0; u < kPW; ++u) {
        const int t = row0 + warp * kPW + u;
        lse_r[u] = t < p.n_q ? lse_b[t] : 0.0f;
        d_r[u] = t < p.n_q ? d_b[t] : 0.0f;
    }
    float dq_acc[kPW][kCols];
#pragma unroll
    for (int u = 0; u < kPW; ++u)
#pragma unroll
        for (int m = 0; m < kCols; ++m) dq_acc[u][m] = 0.0f;

    int key_end = kv_len;
    if (causal) key_end = min(key_end, row0 + kRows);
    for (int kt = 0; kt < key_end; kt += kInner) {
        __syncthreads();
        stage<T>(k_s, dkp, kb, sk, kt, kInner, p.n_k, p.d_k);
        stage<T>(v_s, dvp, vb, sv, kt, kInner, p.n_k, p.d_v);
        __syncthreads();
        const int j = kt + lane;  // this lane's key in the score phase
#pragma unroll
        for (int u = 0; u < kPW; ++u) {
            const int il = warp * kPW + u, t = row0 + il;
            const bool visible = t < p.n_q && j < kv_len && !(causal && j > t);
            float s = 0.0f, dp = 0.0f;
            const float* qr = q_s + il * dkp;
            const float* kr = k_s + lane * dkp;
            for (int c = 0; c < p.d_k; ++c) s = fmaf(qr[c], kr[c], s);
            const float* gr = g_s + il * dvp;
            const float* vr = v_s + lane * dvp;
            for (int c = 0; c < p.d_v; ++c) dp = fmaf(gr[c], vr[c], dp);
            const float pr = visible ? expf(p.scale * s - lse_r[u]) : 0.0f;
            const float ds = pr * (dp + d_r[u]);  // d_r holds -D
            for (int jj = 0; jj < kInner; ++jj) {
                const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
                for (int m = 0; m < kCols; ++m) {
                    const int cc = lane + 32 * m;
                    if (cc < p.d_k) dq_acc[u][m] = fmaf(dsj, k_s[jj * dkp + cc], dq_acc[u][m]);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kPW; ++u) {
        const int t = row0 + warp * kPW + u;
        if (t >= p.n_q) continue;
#pragma unroll
        for (int m = 0; m < kCols; ++m) {
            const int cc = lane + 32 * m;
            if (cc < p.d_k) store_out(dqb + (size_t)t * sk + cc, p.scale * dq_acc[u][m]);
        }
    }
}

template <typename T, int kCols, int kPW>
cudaError_t launch_typed(const BwdParams& p, cudaStream_t stream)
{
    const int dkp = p.d_k + 1, dvp = p.d_v + 1;
    constexpr int kBlock = 4 * kPW;
    const size_t smem_k = sizeof(float) * ((size_t)kBlock * (dkp + dvp) + (size_t)kInner * (dkp + dvp) + 2 * kInner);
    cudaError_t e = cudaFuncSetAttribute(key_grads_kernel<T, kCols, kPW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_k);
    if (e != cudaSuccess) return e;
    key_grads_kernel<T, kCols, kPW><<<dim3((p.n_k + kBlock - 1) / kBlock, p.h, p.B), kThreads, smem_k, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem_q = sizeof(float) * ((size_t)kBlock * (dkp + dvp) + (size_t)kInner * (dkp + dvp));
    e = cudaFuncSetAttribute(query_grads_kernel<T, kCols, kPW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
    if (e != cudaSuccess) return e;
    query_grads_kernel<T, kCols, kPW><<<dim3((p.n_q + kBlock - 1) / kBlock, p.h, p.B), kThreads, smem_q, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_cols(const BwdParams& p, cudaStream_t stream)
{
    const int d = max(p.d_k, p.d_v);
    if (d <= 64) return launch_typed<T, 2, 8>(p, stream);
    if (d <= 128) return launch_typed<T, 4, 8>(p, stream);
    return launch_typed<T, 8, 4>(p, stream);
}

BwdParams make_params(const AttnBwdArgs& a)
{
    BwdParams p;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.out = a.out;
    p.dout = a.dout;
    p.lse = a.lse;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.dsum = a.dsum;
    p.lse2 = a.lse2;
    p.B = a.B;
    p.h = a.h;
    p.n_q = a.n_q;
    p.n_k = a.n_k;
    p.d_k = a.d_k;
    p.d_v = a.d_v;
    p.nqp = (a.n_q + 127) / 128 * 128;
    p.scale = a.scale;
    p.mask_kind = a.mask_kind;
    p.key_lens = a.key_lens;
    p.err_word = a.err_word;
    return p;
}

}  // namespace

namespace {

template <typename T, int kL>
cudaError_t launch_row_dot(const BwdParams& p, cudaStream_t stream)
{
    const long long threads = (long long)p.B * p.h * p.nqp * kL;
    row_dot_kernel<T, kL><<<(unsigned)((threads + kThreads - 1) / kThreads), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_row_dot_for(const BwdParams& p, cudaStream_t stream)
{
    // Lanes per row: d / (16-byte vector) rounded up to a power of two, at most 32.
    const int vecs = (p.d_v * (int)sizeof(T) + 15) / 16;
    if (vecs <= 4) return launch_row_dot<T, 4>(p, stream);
    if (vecs <= 8) return launch_row_dot<T, 8>(p, stream);
    if (vecs <= 16) return launch_row_dot<T, 16>(p, stream);
    return launch_row_dot<T, 32>(p, stream);
}

}  // namespace

cudaError_t launch_attn_bwd_prep(const AttnBwdArgs& a)
{
    const BwdParams p = make_params(a);
    if (a.dtype == HATTN_F32) return launch_row_dot_for<float>(p, a.stream);
    return launch_row_dot_for<__nv_bfloat16>(p, a.stream);
}

cudaError_t launch_attn_bwd_simt(const AttnBwdArgs& a)
{
    const BwdParams p = make_params(a);
    if (a.dtype == HATTN_F32) return launch_cols<float>(p, a.stream);
    return launch_cols<__nv_bfloat16>(p, a.stream);
}

}  // namespace hattn
