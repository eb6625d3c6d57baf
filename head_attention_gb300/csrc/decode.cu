// Decode attention: one new query per (batch, head) against a key/value
// prefix of per-sequence length, the token-by-token generation step of
// "读懂 Attention Is All You Need", §训练能并行，不意味着一次生成整句话 (each new
// target position attends to the keys produced so far). The arithmetic is the
// same scaled dot-product attention as attn_fwd with n_q = 1.
//
// It is a GEMV per (b, h), bound by reading K and V once from HBM, so it runs
// on CUDA cores with 16-byte loads and splits the keys over CTAs:
//   phase 1  CTA (b, h, split) streams its key range: a group of D/8 lanes
//            scores one key (each lane 8 elements of q.k, shuffle reduction),
//            keeps a streaming max m, sum l and its 8-element slice of o, and
//            the CTA merges its 32 * 8 / (D/8) groups into one partial (m, l, o).
//   phase 2  one warp per (b, h) merges the splits' partials:
//            m = max m_s, l = sum l_s 2^(m_s - m), o = sum o_s 2^(m_s - m) / l.
// Base-2 exponentials with scale * log2(e) folded into the scores.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 256;
constexpr int kKeysPerStep = 4;  // keys a lane group has in flight

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

struct DecodeParams {
    const __nv_bfloat16* q;   // [B, 1, h, D]
    const __nv_bfloat16* k;   // [B, n_max, h, D]
    const __nv_bfloat16* v;
    __nv_bfloat16* out;       // [B, 1, h, D]
    const int32_t* kv_lens;   // [B]
    float* partial;           // [B, h, splits, D + 2]: o (unnormalised), m, l
    int B, h, n_max, splits, chunk;
    float scale_log2;
    int* err_word;
};

template <int D>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const DecodeParams p)
{
    constexpr int kLanes = D / 8;              // lanes per key (8 bf16 = 16 bytes each)
    constexpr int kGroups = kThreads / kLanes; // key groups per CTA
    __shared__ float s_m[kGroups], s_l[kGroups];
    __shared__ float s_o[kGroups][D];

    const int split = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
    const int g = threadIdx.x / kLanes, gl = threadIdx.x % kLanes;
    const int kv_len = p.kv_lens[b];
    float* part = p.partial + (((size_t)b * p.h + head) * p.splits + split) * (D + 2);
    if (kv_len < 1 || kv_len > p.n_max) {
        if (threadIdx.x == 0) raise_device_error(p.err_word, HATTN_EKEYLEN);
        for (int i = threadIdx.x; i < D + 2; i += kThreads) part[i] = i == D ? -INFINITY : 0.0f;
        return;
    }
    const int k0 = split * p.chunk;
    const int k1 = min(kv_len, k0 + p.chunk);

    float qf[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.h + head) * D + 8 * gl), qf);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[e] *= p.scale_log2;

    const size_t row_stride = (size_t)p.h * D;
    const __nv_bfloat16* kb = p.k + (size_t)b * p.n_max * row_stride + (size_t)head * D + 8 * gl;
    const __nv_bfloat16* vb = p.v + (size_t)b * p.n_max * row_stride + (size_t)head * D + 8 * gl;
    float m = -INFINITY, l = 0.0f, o[8] = {0, 0, 0, 0, 0, 0, 0, 0};

    // The trip count is the same for every lane (the shuffles below involve the
    // whole warp); keys past the range are masked per group.
    for (int step = k0; step < k1; step += kGroups * kKeysPerStep) {
        const int base = step + g;
        uint4 kr[kKeysPerStep], vr[kKeysPerStep];
#pragma unroll
        for (int u = 0; u < kKeysPerStep; ++u) {
            const int key = base + u * kGroups;
            kr[u] = make_uint4(0u, 0u, 0u, 0u);
            vr[u] = make_uint4(0u, 0u, 0u, 0u);
            if (key < k1) {
                kr[u] = *reinterpret_cast<const uint4*>(kb + (size_t)key * row_stride);
                vr[u] = *reinterpret_cast<const uint4*>(vb + (size_t)key * row_stride);
            }
        }
        float s[kKeysPerStep];
#pragma unroll
        for (int u = 0; u < kKeysPerStep; ++u) {
            float kf[8];
            bf16x8_to_f32(kr[u], kf);
            float a = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaf(qf[e], kf[e], a);
#pragma unroll
            for (int off = kLanes / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            s[u] = (base + u * kGroups < k1) ? a : -INFINITY;
        }
        float mx = m;
#pragma unroll
        for (int u = 0; u < kKeysPerStep; ++u) mx = fmaxf(mx, s[u]);
        if (mx == -INFINITY) continue;  // nothing in range yet (uniform in the group; no
                                        // warp-wide operation follows in this step)
        const float alpha = ex2_approx(m - mx);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= alpha;
#pragma unroll
        for (int u = 0; u < kKeysPerStep; ++u) {
            const float pu = ex2_approx(s[u] - mx);
            l += pu;
            float vf[8];
            bf16x8_to_f32(vr[u], vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = fmaf(pu, vf[e], o[e]);
        }
        m = mx;
    }

    // Merge the CTA's groups into one partial.
    if (gl == 0) {
        s_m[g] = m;
        s_l[g] = l;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s_o[g][8 * gl + e] = o[e];
    __syncthreads();
    float mt = -INFINITY;
    for (int i = 0; i < kGroups; ++i) mt = fmaxf(mt, s_m[i]);
    if (threadIdx.x < D) {
        float acc = 0.0f;
        if (mt != -INFINITY)
            for (int i = 0; i < kGroups; ++i)
                if (s_m[i] != -INFINITY) acc += s_o[i][threadIdx.x] * ex2_approx(s_m[i] - mt);
        part[threadIdx.x] = acc;
    }
    if (threadIdx.x == 0) {
        float lt = 0.0f;
        if (mt != -INFINITY)
            for (int i = 0; i < kGroups; ++i)
                if (s_m[i] != -INFINITY) lt += s_l[i] * ex2_approx(s_m[i] - mt);
        part[D] = mt;
        part[D + 1] = lt;
    }
}

template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p)
{
    const int bh = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (bh >= p.B * p.h) return;
    const int lane = threadIdx.x % 32;
    const float* part = p.partial + (size_t)bh * p.splits * (D + 2);
    float mt = -INFINITY;
    for (int s = 0; s < p.splits; ++s) mt = fmaxf(mt, part[s * (D + 2) + D]);
    float lt = 0.0f;
    float acc[D / 32] = {};
    for (int s = 0; s < p.splits; ++s) {
        const float ms = part[s * (D + 2) + D];
        if (ms == -INFINITY) continue;
        const float w = ex2_approx(ms - mt);
        lt += w * part[s * (D + 2) + D + 1];
#pragma unroll
        for (int i = 0; i < D / 32; ++i) acc[i] += w * part[s * (D + 2) + lane + 32 * i];
    }
    const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
    __nv_bfloat16* o = p.out + (size_t)bh * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) o[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
}

template <int D>
cudaError_t launch_d(const DecodeLaunch& a)
{
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.k = static_cast<const __nv_bfloat16*>(a.k);
    p.v = static_cast<const __nv_bfloat16*>(a.v);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.kv_lens = a.kv_lens;
    p.partial = static_cast<float*>(a.workspace);
    p.B = a.B;
    p.h = a.h;
    p.n_max = a.n_max;
    p.splits = a.splits;
    p.chunk = a.chunk;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err_word = a.err_word;
    decode_split_kernel<D><<<dim3(a.splits, a.h, a.B), kThreads, 0, a.stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int bh = a.B * a.h;
    decode_combine_kernel<D><<<(bh + 3) / 4, 128, 0, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

void decode_split_plan(int B, int h, int n_max, int* splits, int* chunk)
{
    // Enough CTAs to cover the SMs about four times, keys in chunks of >= 256.
    const long long bh = (long long)B * h;
    long long s = (4LL * 152 + bh - 1) / bh;
    const long long max_s = (n_max + 255) / 256;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    if (s > 65535) s = 65535;
    int c = static_cast<int>((n_max + s - 1) / s);
    c = (c + 63) / 64 * 64;
    *chunk = c;
    *splits = (n_max + c - 1) / c;
}

cudaError_t launch_attn_decode(const DecodeLaunch& a)
{
    if (a.d == 64) return launch_d<64>(a);
    if (a.d == 128) return launch_d<128>(a);
    return launch_d<256>(a);
}

}  // namespace hattn
