// Sinusoidal positional encoding added to scaled embeddings (elementwise,
// HBM-bound): out[b,t,2i] = s*emb[b,t,2i] + sin(pos*w_i), out[b,t,2i+1] =
// s*emb[b,t,2i+1] + cos(pos*w_i), pos = pos0 + t, w_i = 10000^(-2i/d_model)
// ("做法 · Attention Is All You Need", §去掉循环，因而须补回顺序; the embedding
// is multiplied by sqrt(d_model) before the addition per "读懂 Attention Is All
// You Need", §没有循环，模型怎样知道词序？).
//
// Layout of the work: the encoding depends on (t, i) only, so a thread owns
// kPairs adjacent frequencies i of one position t, computes their sin/cos once,
// and applies them to a chunk of kBatchInFlight batch rows at that position
// (grid z walks the chunks); the chunk's loads are all issued before any is
// used, so each SM keeps enough bytes in flight to cover the HBM latency.
// Consecutive threads cover consecutive 16-byte pieces of a row (coalesced).
// The grid is one wave of resident CTAs and each thread walks positions with a
// grid stride, so the last, partial pass over positions is a small share.
//
// Accuracy without per-element fp64: the angle pos * w_i reaches tens of
// thousands of radians, where a plain fp32 product is off by ~1e-3 rad. The
// constant c_i = w_i / (2 pi) (turns per position) is formed in fp64 once and
// split into fp32 hi + lo. Positions are integers below 2^24, exact in fp32, so
//   pos * hi = p + e   exactly (p rounded, e = fma(pos, hi, -p)),
//   p - rint(p)        exact,
// and the fraction of a turn f = (p - rint(p)) + (e + pos * lo) lies in about
// [-1/2, 1/2] with an absolute error of a few 2^-25. sin/cos of 2 pi f, an
// angle in [-pi, pi], use the hardware approximations, whose absolute error on
// that range is about 2^-21.4; the total stays below 1e-6 absolute.
#include <cuda_bf16.h>

#include "internal.h"

namespace hattn {
namespace {

constexpr int kThreads = 256;
constexpr int kBatchInFlight = 8;

// kPairs consecutive (even, odd) element pairs of one row: 2 * kPairs values.
template <typename T, int kPairs>
struct Vec {
    static constexpr int kBytes = 2 * kPairs * (int)sizeof(T);
    static_assert(kBytes % 4 == 0 && (kBytes <= 16 || kBytes % 16 == 0), "vector size");
    static constexpr int kWords = kBytes / 4;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const T* p)
    {
        if constexpr (kBytes >= 16) {
#pragma unroll
            for (int j = 0; j < kBytes / 16; ++j) {
                const uint4 v = reinterpret_cast<const uint4*>(p)[j];
                w[4 * j] = v.x, w[4 * j + 1] = v.y, w[4 * j + 2] = v.z, w[4 * j + 3] = v.w;
            }
        } else if constexpr (kBytes == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            w[0] = v.x, w[1] = v.y;
        } else {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        }
    }
    __device__ __forceinline__ void store(T* p) const
    {
        if constexpr (kBytes >= 16) {
#pragma unroll
            for (int j = 0; j < kBytes / 16; ++j)
                reinterpret_cast<uint4*>(p)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        } else if constexpr (kBytes == 8) {
            *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        } else {
            *reinterpret_cast<uint32_t*>(p) = w[0];
        }
    }
    // Value e (0 .. 2*kPairs-1) as fp32, and its replacement by x.
    __device__ __forceinline__ float get(int e) const
    {
        if constexpr (sizeof(T) == 4) return __uint_as_float(w[e]);
        else return __uint_as_float((e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
    }
    __device__ __forceinline__ void set_pair(int j, float a, float b)
    {
        if constexpr (sizeof(T) == 4) {
            w[2 * j] = __float_as_uint(a);
            w[2 * j + 1] = __float_as_uint(b);
        } else {
            const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
            w[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
    }
};

template <typename T, int kPairs>
__global__ void __launch_bounds__(kThreads)
    pos_encoding_kernel(const T* emb, T* out, int B, int n, int half_d, int cols_per_block,
                        float emb_scale, int pos0, double log2_w_step)
{
    const int i0 = (blockIdx.x * cols_per_block + threadIdx.x % cols_per_block) * kPairs;
    if (i0 >= half_d) return;
    const int t_per_block = kThreads / cols_per_block;
    const float two_pi = 6.283185307179586f;
    // Turns per position of each owned frequency, 10000^(-2i/d_model) / (2 pi),
    // as an fp32 hi + lo pair.
    float hi[kPairs], lo[kPairs];
#pragma unroll
    for (int j = 0; j < kPairs; ++j) {
        const double c = exp2(log2_w_step * (i0 + j)) * 0.15915494309189535;
        hi[j] = static_cast<float>(c);
        lo[j] = static_cast<float>(c - static_cast<double>(hi[j]));
    }
    const size_t row_elems = 2 * (size_t)half_d;
    const size_t batch_stride = (size_t)n * row_elems;
    for (int t = blockIdx.y * t_per_block + threadIdx.x / cols_per_block; t < n;
         t += gridDim.y * t_per_block) {
        const float pos = static_cast<float>(pos0 + t);
        float sn[kPairs], cs[kPairs];
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            const float p = pos * hi[j];
            const float e = fmaf(pos, hi[j], -p);
            const float f = (p - rintf(p)) + fmaf(pos, lo[j], e);
            const float ang = two_pi * f;
            sn[j] = __sinf(ang);
            cs[j] = __cosf(ang);
        }
        const size_t at = (size_t)t * row_elems + 2 * (size_t)i0;
        for (int b0 = blockIdx.z * kBatchInFlight; b0 < B; b0 += gridDim.z * kBatchInFlight) {
            Vec<T, kPairs> v[kBatchInFlight];
#pragma unroll
            for (int u = 0; u < kBatchInFlight; ++u) {
#pragma unroll
                for (int k = 0; k < Vec<T, kPairs>::kWords; ++k) v[u].w[k] = 0u;
                if (emb && b0 + u < B) v[u].load(emb + (size_t)(b0 + u) * batch_stride + at);
            }
#pragma unroll
            for (int u = 0; u < kBatchInFlight; ++u) {
                if (b0 + u >= B) break;
#pragma unroll
                for (int j = 0; j < kPairs; ++j)
                    v[u].set_pair(j, fmaf(emb_scale, v[u].get(2 * j), sn[j]),
                                  fmaf(emb_scale, v[u].get(2 * j + 1), cs[j]));
                v[u].store(out + (size_t)(b0 + u) * batch_stride + at);
            }
        }
    }
}

template <typename T, int kPairs>
cudaError_t launch_typed(const void* emb, void* out, int B, int n, int d_model, float emb_scale,
                         int pos0, cudaStream_t stream)
{
    const int half_d = d_model / 2;
    const int col_threads = (half_d + kPairs - 1) / kPairs;
    int cols = 32;
    while (cols < col_threads && cols < kThreads) cols *= 2;
    const int t_per_block = kThreads / cols;
    const int gx = (col_threads + cols - 1) / cols;
    long long gy = (n + t_per_block - 1) / t_per_block;
    // One wave of resident CTAs in all.
    static const int resident = [] {
        int dev = 0, sms = 0, per_sm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pos_encoding_kernel<T, kPairs>,
                                                      kThreads, 0);
        return (sms > 0 ? sms : 152) * (per_sm > 0 ? per_sm : 1);
    }();
    long long gz = (B + kBatchInFlight - 1) / kBatchInFlight;
    if (gz > 65535) gz = 65535;
    const long long cap = (resident + gx * gz - 1) / (gx * gz);
    if (gy > cap) gy = cap;
    if (gy > 65535) gy = 65535;
    // 10000^(-2i/d) = 2^(i * (-log2(10000) / (d/2)))
    const double step = -13.287712379549449 / half_d;
    pos_encoding_kernel<T, kPairs><<<dim3(gx, (unsigned)gy, (unsigned)gz), kThreads, 0, stream>>>(
        static_cast<const T*>(emb), static_cast<T*>(out), B, n, half_d, cols, emb_scale, pos0,
        step);
    return cudaGetLastError();
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

cudaError_t launch_pos_encoding(const void* emb, void* out, int dtype, int B, int n, int d_model,
                                float emb_scale, int pos0, cudaStream_t stream)
{
    // Four pairs per thread (16- or 32-byte accesses) when every row start is
    // 16-byte aligned; one pair otherwise.
    const bool wide = (d_model % 8 == 0) && aligned(out, 16) && (!emb || aligned(emb, 16));
    if (dtype == HATTN_F32)
        return wide ? launch_typed<float, 4>(emb, out, B, n, d_model, emb_scale, pos0, stream)
                    : launch_typed<float, 1>(emb, out, B, n, d_model, emb_scale, pos0, stream);
    return wide ? launch_typed<__nv_bfloat16, 4>(emb, out, B, n, d_model, emb_scale, pos0, stream)
                : launch_typed<__nv_bfloat16, 1>(emb, out, B, n, d_model, emb_scale, pos0, stream);
}

}  // namespace hattn
