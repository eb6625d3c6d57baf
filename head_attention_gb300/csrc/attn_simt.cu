// CUDA-core attention kernel: exact fp32 arithmetic (expf, fp32 FMA dot
// products), used for fp32 inputs and for bf16 shapes the tensor-core kernel
// does not implement (d_k != d_v, d not in {64, 128}, scale <= 0).
//
// Each CTA owns 8 query rows of one (batch, head), each warp 2 of them (4 rows,
// one per warp, when 8-row CTAs would leave fewer than two per SM).
// K/V stream through shared memory 32 keys at a time, staged with batched
// 16-byte loads (every load of a tile is in flight before the first store). For
// a row, lane j scores key j of the tile (four independent partial dot
// products), the row max and row sum are warp-shuffle reductions, and the
// output columns are spread over the lanes (column c on lane c % 32). The
// softmax is the streaming ("online") form: a running max m and sum l, with
// the accumulator rescaled by exp(m_old - m_new) whenever m grows, so the score
// matrix is never stored.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kKeys = 32;      // keys per shared-memory tile (one per lane)
constexpr int kThreads = 128;  // 4 warps
constexpr int kMaxD = 256;

__device__ __forceinline__ void widen4(const uint4& v, const float*, float* out)
{
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ void widen4(const uint4& v, const __nv_bfloat16*, float* out)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

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

// Copies rows [row0, row0 + rows) of a [n, *] slice (row stride src_stride
// elements, d <= kMaxRowD elements per row) into fp32 shared memory with row
// stride dst_stride, zero for rows >= n. All 16-byte loads are issued before any store.
template <typename T, int kMaxRowD>
__device__ __forceinline__ void stage_rows(float* dst, int dst_stride, const T* src,
                                           size_t src_stride, int row0, int rows, int n, int d)
{
    constexpr int V = 16 / sizeof(T);           // elements per 16-byte load
    constexpr int kMaxLoads = (kKeys * kMaxRowD / V + kThreads - 1) / kThreads;
    const int per_row = d / V;
    const int total = rows * per_row;
    uint4 buf[kMaxLoads];
#pragma unroll
    for (int u = 0; u < kMaxLoads; ++u) {
        const int idx = threadIdx.x + u * kThreads;
        buf[u] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < total) {
            const int r = row0 + idx / per_row;
            if (r < n)
                buf[u] = *reinterpret_cast<const uint4*>(src + (size_t)r * src_stride + (idx % per_row) * V);
        }
    }
#pragma unroll
    for (int u = 0; u < kMaxLoads; ++u) {
        const int idx = threadIdx.x + u * kThreads;
        if (idx < total) {
            float w[V];
            widen4(buf[u], static_cast<const T*>(nullptr), w);
            float* o = dst + (idx / per_row) * dst_stride + (idx % per_row) * V;
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = w[e];
        }
    }
}

// kCols = output columns per lane (d_v <= 32 * kCols); kMaxRowD bounds d_k and d_v
// (a tighter bound unrolls less staging code: the small fp32 problems are bound
// by latency, instruction fetch included). kRows = query rows per CTA (4 or 8).
template <typename T, int kCols, int kMaxRowD, int kRows>
__global__ void __launch_bounds__(kThreads)
    attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     T* __restrict__ out, int n_q, int n_k, int h, int d_k, int d_v, float scale,
                     int mask_kind, const int32_t* __restrict__ key_lens, int* err_word,
                     float* __restrict__ lse)
{
    constexpr int kRowsPerWarp = kRows / (kThreads / 32);
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
    const size_t qk_row_stride = (size_t)h * d_k, v_row_stride = (size_t)h * d_v;
    const T* q_bh = q + (size_t)b * n_q * qk_row_stride + (size_t)head * d_k;
    const T* k_bh = k + (size_t)b * n_k * qk_row_stride + (size_t)head * d_k;
    const T* v_bh = v + (size_t)b * n_k * v_row_stride + (size_t)head * d_v;
    T* o_bh = out + (size_t)b * n_q * v_row_stride + (size_t)head * d_v;

    // While the previous kernel may still run (programmatic dependent launch): the
    // rows this CTA will read, into L2 only (Q rows, and the K and V rows its causal
    // bound allows; the key length may be the previous kernel's output, so n_k).
    {
        const int q_end = min(n_q, row0 + kRows);
        const int k_end = causal ? min(n_k, row0 + kRows) : n_k;
        const int qk_lines = (d_k * (int)sizeof(T) + 127) / 128, v_lines = (d_v * (int)sizeof(T) + 127) / 128;
        const int nq = max(0, q_end - row0) * qk_lines, nk = k_end * qk_lines, nv = k_end * v_lines;
        for (int i = threadIdx.x; i < nq + nk + nv; i += kThreads) {
            const T* a;
            if (i < nq) a = q_bh + (size_t)(row0 + i / qk_lines) * qk_row_stride + (i % qk_lines) * (128 / sizeof(T));
            else if (i < nq + nk) a = k_bh + (size_t)((i - nq) / qk_lines) * qk_row_stride + ((i - nq) % qk_lines) * (128 / sizeof(T));
            else a = v_bh + (size_t)((i - nq - nk) / v_lines) * v_row_stride + ((i - nq - nk) % v_lines) * (128 / sizeof(T));
            prefetch_l2(a);
        }
    }
    griddep_wait();
    griddep_launch_dependents();

    int kv_len = n_k;
    if (mask_kind & HATTN_MASK_KEY_PADDING) {
        kv_len = key_lens[b];
        if (kv_len < 1 || kv_len > n_k) {
            for (int idx = threadIdx.x; idx < kRows * d_v; idx += kThreads) {
                const int t = row0 + idx / d_v;
                if (t < n_q) store_f32(o_bh + (size_t)t * v_row_stride + idx % d_v, 0.0f);
            }
            if (lse)
                for (int r = threadIdx.x; r < kRows; r += kThreads)
                    if (row0 + r < n_q) lse[((size_t)b * h + head) * n_q + row0 + r] = -INFINITY;
            if (threadIdx.x == 0) raise_device_error(err_word, HATTN_EKEYLEN);
            return;
        }
    }
    // Keys any row of this CTA can see.
    int key_end = kv_len;
    if (causal) key_end = min(key_end, row0 + kRows);

    stage_rows<T, kMaxRowD>(q_s, dkp, q_bh, qk_row_stride, row0, kRows, n_q, d_k);

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kCols];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.0f;
#pragma unroll
        for (int i = 0; i < kCols; ++i) acc[rr][i] = 0.0f;
    }

    for (int kt = 0; kt < key_end; kt += kKeys) {
        __syncthreads();  // q_s is staged and the previous tile is no longer read
        stage_rows<T, kMaxRowD>(k_s, dkp, k_bh, qk_row_stride, kt, kKeys, n_k, d_k);
        stage_rows<T, kMaxRowD>(v_s, d_v, v_bh, v_row_stride, kt, kKeys, n_k, d_v);
        __syncthreads();

#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr;
            const int t = row0 + r;
            const int j = kt + lane;
            const float* qr = q_s + r * dkp;
            const float* kr = k_s + lane * dkp;
            float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
            int c = 0;
            for (; c + 4 <= d_k; c += 4) {
                s0 = fmaf(qr[c], kr[c], s0);
                s1 = fmaf(qr[c + 1], kr[c + 1], s1);
                s2 = fmaf(qr[c + 2], kr[c + 2], s2);
                s3 = fmaf(qr[c + 3], kr[c + 3], s3);
            }
            for (; c < d_k; ++c) s0 = fmaf(qr[c], kr[c], s0);
            float s = ((s0 + s1) + (s2 + s3)) * scale;
            const bool visible = (j < kv_len) && !(causal && j > t);
            s = visible ? s : -INFINITY;
            const float m_new = fmaxf(m[rr], warp_max(s));
            if (m_new == -INFINITY) continue;  // nothing visible yet for this row (warp-uniform)
            const float alpha = expf(m[rr] - m_new);
            const float p = visible ? expf(s - m_new) : 0.0f;
            l[rr] = l[rr] * alpha + warp_sum(p);
#pragma unroll
            for (int i = 0; i < kCols; ++i) acc[rr][i] *= alpha;
#pragma unroll 8
            for (int jj = 0; jj < kKeys; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int i = 0; i < kCols; ++i) {
                    const int cc = lane + 32 * i;
                    if (cc < d_v) acc[rr][i] = fmaf(pj, v_s[jj * d_v + cc], acc[rr][i]);
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
        if (lse && lane == 0) lse[((size_t)b * h + head) * n_q + t] = m[rr] + logf(l[rr]);
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
            const int cc = lane + 32 * i;
            if (cc < d_v) store_f32(o_bh + (size_t)t * v_row_stride + cc, acc[rr][i] * inv);
        }
    }
}

template <typename T, int kCols, int kMaxRowD, int kRows>
cudaError_t launch_rows(const AttnArgs& a)
{
    const size_t smem = sizeof(float) * ((size_t)kRows * (a.d_k + 1) + (size_t)kKeys * (a.d_k + 1) +
                                         (size_t)kKeys * a.d_v);
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<T, kCols, kMaxRowD, kRows>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.n_q + kRows - 1) / kRows, a.h, a.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_simt_kernel<T, kCols, kMaxRowD, kRows>, static_cast<const T*>(a.q),
                              static_cast<const T*>(a.k), static_cast<const T*>(a.v), static_cast<T*>(a.out),
                              a.n_q, a.n_k, a.h, a.d_k, a.d_v, a.scale, a.mask_kind, a.key_lens, a.err_word,
                              a.lse);
}

// 8 query rows per CTA share each staged K/V tile; when that leaves fewer than
// two CTAs per SM, 4 rows per CTA (twice the CTAs) measured faster: the fp32
// encoder workload (16 heads of 64 rows) took 8.4 us per step against 9.9 us.
template <typename T, int kCols, int kMaxRowD = kMaxD>
cudaError_t launch_typed(const AttnArgs& a)
{
    const long long ctas8 = (long long)((a.n_q + 7) / 8) * a.h * a.B;
    if (ctas8 < 2LL * sm_count()) return launch_rows<T, kCols, kMaxRowD, 4>(a);
    return launch_rows<T, kCols, kMaxRowD, 8>(a);
}

template <typename T>
cudaError_t launch_cols(const AttnArgs& a)
{
    if (a.d_v <= 64 && a.d_k <= 64) return launch_typed<T, 2, 64>(a);
    if (a.d_v <= 64) return launch_typed<T, 2>(a);
    if (a.d_v <= 128) return launch_typed<T, 4>(a);
    return launch_typed<T, 8>(a);
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a)
{
    if (a.dtype == HATTN_F32) return launch_cols<float>(a);
    return launch_cols<__nv_bfloat16>(a);
}

}  // namespace hattn
