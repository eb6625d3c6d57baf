// CUDA-core attention kernel: exact fp32 arithmetic (expf, fp32 FMA dot
// products), used for fp32 inputs and for bf16 shapes the tensor-core kernel
// does not implement (d_k != d_v, or d not in {64, 128}).
//
// Each CTA owns 16 query rows of one (batch, head); each warp owns 4 of them.
// K/V stream through shared memory 32 keys at a time. For a row, lane j scores
// key j of the tile, the row max and row sum are warp-shuffle reductions, and
// the output columns are spread over the lanes (column c on lane c % 32). The
// softmax is the streaming ("online") form: a running max m and sum l, with the
// accumulator rescaled by exp(m_old - m_new) whenever m grows, so the score
// matrix is never stored.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kRows = 16;     // query rows per CTA
constexpr int kKeys = 32;     // keys per shared-memory tile (one per lane)
constexpr int kThreads = 128; // 4 warps
constexpr int kRowsPerWarp = kRows / (kThreads / 32);
constexpr int kMaxD = 256;
constexpr int kColsPerLane = kMaxD / 32;

__device__ __forceinline__ float load_f32(const float* p) { return *p; }
__device__ __forceinline__ float load_f32(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f32(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f32(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x)
{
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     T* __restrict__ out, int n_q, int n_k, int h, int d_k, int d_v, float scale,
                     int mask_kind, const int32_t* __restrict__ key_lens, int* err_word)
{
    extern __shared__ float smem[];
    const int dkp = d_k + 1;  // padded stride: lane j reads row j without bank conflicts
    float* q_s = smem;                    // [kRows][dkp]
    float* k_s = q_s + kRows * dkp;       // [kKeys][dkp]
    float* v_s = k_s + kKeys * dkp;       // [kKeys][d_v]

    const int row0 = blockIdx.x * kRows;
    const int head = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool causal = (mask_kind & HATTN_MASK_CAUSAL) != 0;
    const size_t q_row_stride = (size_t)h * d_k, o_row_stride = (size_t)h * d_v;
    const T* q_bh = q + (size_t)b * n_q * q_row_stride + (size_t)head * d_k;
    const T* k_bh = k + (size_t)b * n_k * q_row_stride + (size_t)head * d_k;
    const T* v_bh = v + (size_t)b * n_k * o_row_stride + (size_t)head * d_v;
    T* o_bh = out + (size_t)b * n_q * o_row_stride + (size_t)head * d_v;

    int kv_len = n_k;
    if (mask_kind & HATTN_MASK_KEY_PADDING) {
        kv_len = key_lens[b];
        if (kv_len < 1 || kv_len > n_k) {
            for (int idx = threadIdx.x; idx < kRows * d_v; idx += kThreads) {
                const int t = row0 + idx / d_v;
                if (t < n_q) store_f32(o_bh + (size_t)t * o_row_stride + idx % d_v, 0.0f);
            }
            if (threadIdx.x == 0) raise_device_error(err_word, HATTN_EKEYLEN);
            return;
        }
    }
    // Keys any row of this CTA can see.
    int key_end = kv_len;
    if (causal) key_end = min(key_end, row0 + kRows);

    for (int idx = threadIdx.x; idx < kRows * d_k; idx += kThreads) {
        const int r = idx / d_k, c = idx % d_k, t = row0 + r;
        q_s[r * dkp + c] = (t < n_q) ? load_f32(q_bh + (size_t)t * q_row_stride + c) : 0.0f;
    }

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kColsPerLane];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.0f;
#pragma unroll
        for (int i = 0; i < kColsPerLane; ++i) acc[rr][i] = 0.0f;
    }

    for (int kt = 0; kt < key_end; kt += kKeys) {
        __syncthreads();  // the previous tile is no longer read
        for (int idx = threadIdx.x; idx < kKeys * d_k; idx += kThreads) {
            const int j = kt + idx / d_k, c = idx % d_k;
            k_s[(idx / d_k) * dkp + c] = (j < n_k) ? load_f32(k_bh + (size_t)j * q_row_stride + c) : 0.0f;
        }
        for (int idx = threadIdx.x; idx < kKeys * d_v; idx += kThreads) {
            const int j = kt + idx / d_v;
            v_s[idx] = (j < n_k) ? load_f32(v_bh + (size_t)j * o_row_stride + idx % d_v) : 0.0f;
        }
        __syncthreads();

#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr;
            const int t = row0 + r;
            const int j = kt + lane;
            float s = 0.0f;
            for (int c = 0; c < d_k; ++c) s = fmaf(q_s[r * dkp + c], k_s[lane * dkp + c], s);
            s *= scale;
            const bool visible = (j < kv_len) && !(causal && j > t);
            s = visible ? s : -INFINITY;
            const float m_new = fmaxf(m[rr], warp_max(s));
            if (m_new == -INFINITY) continue;  // nothing visible yet for this row (warp-uniform)
            const float alpha = expf(m[rr] - m_new);
            const float p = visible ? expf(s - m_new) : 0.0f;
            l[rr] = l[rr] * alpha + warp_sum(p);
#pragma unroll
            for (int i = 0; i < kColsPerLane; ++i) acc[rr][i] *= alpha;
            for (int jj = 0; jj < kKeys; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
                if (pj == 0.0f) continue;  // warp-uniform: pj is broadcast
#pragma unroll
                for (int i = 0; i < kColsPerLane; ++i) {
                    const int c = lane + 32 * i;
                    if (c < d_v) acc[rr][i] = fmaf(pj, v_s[jj * d_v + c], acc[rr][i]);
                }
            }
            m[rr] = m_new;
        }
    }

#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int t = row0 + warp * kRowsPerWarp + rr;
        if (t >= n_q) continue;
        const float inv = l[rr] > 0.0f ? 1.0f / l[rr] : 0.0f;
#pragma unroll
        for (int i = 0; i < kColsPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < d_v) store_f32(o_bh + (size_t)t * o_row_stride + c, acc[rr][i] * inv);
        }
    }
}

template <typename T>
cudaError_t launch_typed(const AttnArgs& a)
{
    const size_t smem = sizeof(float) * ((size_t)kRows * (a.d_k + 1) + (size_t)kKeys * (a.d_k + 1) +
                                         (size_t)kKeys * a.d_v);
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.n_q + kRows - 1) / kRows, a.h, a.B);
    attn_simt_kernel<T><<<grid, kThreads, smem, a.stream>>>(
        static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
        static_cast<T*>(a.out), a.n_q, a.n_k, a.h, a.d_k, a.d_v, a.scale, a.mask_kind,
        a.key_lens, a.err_word);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a)
{
    if (a.dtype == HATTN_F32) return launch_typed<float>(a);
    return launch_typed<__nv_bfloat16>(a);
}

}  // namespace hattn
