// Sinusoidal positional encoding added to scaled embeddings (elementwise,
// HBM-bound): out[b,t,2i] = s*emb[b,t,2i] + sin(pos*w_i), out[b,t,2i+1] =
// s*emb[b,t,2i+1] + cos(pos*w_i), pos = pos0 + t, w_i = 10000^(-2i/d_model)
// ("做法 · Attention Is All You Need", §去掉循环，因而须补回顺序; the embedding
// is multiplied by sqrt(d_model) before the addition per "读懂 Attention Is All
// You Need", §没有循环，模型怎样知道词序？).
//
// Two kernels. Problems of 16 MB or more whose rows are 16-byte multiples at
// 16-byte aligned addresses take the bulk-copy path below (83 % of the measured
// HBM copy bandwidth on B=16 n=8192 d_model=512 bf16, against 66 % for the
// register path). Otherwise, the register path:
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

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 256;
constexpr int kBatchInFlight = 8;

// sin and cos of 2 pi (pos * (hi + lo)) mod 1 turn (see the accuracy note above).
__device__ __forceinline__ void pe_sincos(float pos, float hi, float lo, float& sn, float& cs)
{
    const float p = pos * hi;
    const float e = fmaf(pos, hi, -p);
    const float f = (p - rintf(p)) + fmaf(pos, lo, e);
    const float ang = 6.283185307179586f * f;
    sn = __sinf(ang);
    cs = __cosf(ang);
}

// Turns per position of frequency i, 10000^(-2i/d_model) / (2 pi), as fp32 hi + lo.
__device__ __forceinline__ void pe_turns(double log2_w_step, int i, float& hi, float& lo)
{
    const double c = exp2(log2_w_step * i) * 0.15915494309189535;
    hi = static_cast<float>(c);
    lo = static_cast<float>(c - static_cast<double>(hi));
}

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
    // Turns per position of each owned frequency, 10000^(-2i/d_model) / (2 pi),
    // as an fp32 hi + lo pair.
    float hi[kPairs], lo[kPairs];
#pragma unroll
    for (int j = 0; j < kPairs; ++j) pe_turns(log2_w_step, i0 + j, hi[j], lo[j]);
    const size_t row_elems = 2 * (size_t)half_d;
    const size_t batch_stride = (size_t)n * row_elems;
    for (int t = blockIdx.y * t_per_block + threadIdx.x / cols_per_block; t < n;
         t += gridDim.y * t_per_block) {
        const float pos = static_cast<float>(pos0 + t);
        float sn[kPairs], cs[kPairs];
#pragma unroll
        for (int j = 0; j < kPairs; ++j) pe_sincos(pos, hi[j], lo[j], sn[j], cs[j]);
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

// ---------------------------------------------------------------- bulk-copy path
//
// Rows of 16-byte multiples at 16-byte aligned addresses stream through shared
// memory by bulk copies instead: a persistent CTA (one per SM) walks chunks of
// R positions x Bc batch rows (each batch row's R rows are contiguous, one copy
// each) through a 4-stage ring of 48 KB stages. Warp 0 moves the data: it loads a stage, and
// once the other 31 warps report the chunk computed (an mbarrier, no block-wide
// barrier) stores it back and refills the stage two chunks ahead after the
// stores out of it have been read. The compute warps compute sin/cos once per
// (position, frequency) of the chunk and apply them to its Bc batch rows in
// place. Two chunks of loads stay in flight per SM, without registers holding them.
constexpr int kBulkStages = 4;
constexpr int kBulkThreads = 1024;
constexpr uint32_t kBulkStageBytes = 48 * 1024;
constexpr int kBulkMaxHalfD = 2048;  // turn table of half_d (hi, lo) pairs: 16 KB

struct BulkShape {
    int B, n, half_d;
    uint32_t row_bytes;
    int R, Bc;         // positions and batch rows per chunk
    int b_groups;      // ceil(B / Bc)
    int chunks;        // ceil(n / R) * b_groups
};

template <typename T>
__global__ void __launch_bounds__(kBulkThreads, 1)
    pos_encoding_bulk_kernel(const T* emb, T* out, const BulkShape sh, float emb_scale, int pos0,
                             double log2_w_step, int* err_word)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    float2* turns = reinterpret_cast<float2*>(smem + kBulkStages * kBulkStageBytes);
    const uint32_t bar0 = smem_u32(turns + kBulkMaxHalfD);
    // ready(s): the stage's chunk landed (or, without loads, the stage is free);
    // computed(s): every compute warp finished the stage's chunk.
    auto ready = [&](int st) { return bar0 + 8u * st; };
    auto computed = [&](int st) { return bar0 + 8u * (kBulkStages + st); };
    const uint32_t stage0 = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    constexpr int kComputeWarps = kBulkThreads / 32 - 1;  // warp 0 moves the data
    const bool load = emb != nullptr;

    for (int i = tid; i < sh.half_d; i += kBulkThreads) pe_turns(log2_w_step, i, turns[i].x, turns[i].y);
    if (tid == 0) {
        for (int st = 0; st < kBulkStages; ++st) {
            mbar_init(ready(st), 1);
            mbar_init(computed(st), kComputeWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    struct Chunk {
        int t0, rows, b0, bcnt;
    };
    auto chunk_of = [&](int k) {
        const int c = blockIdx.x + k * gridDim.x;
        const int tc = c / sh.b_groups, bg = c - tc * sh.b_groups;
        Chunk ch;
        ch.t0 = tc * sh.R;
        ch.rows = min(sh.R, sh.n - ch.t0);
        ch.b0 = bg * sh.Bc;
        ch.bcnt = min(sh.Bc, sh.B - ch.b0);
        return ch;
    };
    const int mine = sh.chunks > static_cast<int>(blockIdx.x)
                         ? (sh.chunks - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                         : 0;
    const size_t batch_stride = (size_t)sh.n * 2 * sh.half_d;
    // Stage layout: batch row b of the chunk at b * R * row_bytes, its R rows contiguous.
    auto gaddr = [&](const Chunk& ch, int b) { return (size_t)(ch.b0 + b) * batch_stride + (size_t)ch.t0 * 2 * sh.half_d; };
    auto saddr = [&](int st, int b) { return stage0 + st * kBulkStageBytes + b * sh.R * sh.row_bytes; };

    if (warp == 0) {
        if (lane == 0) {
            // Marks stage k % 3 ready for chunk k: loads it, or (without loads) just
            // releases it to the compute warps.
            auto fill = [&](int k) {
                const Chunk ch = chunk_of(k);
                const int st = k % kBulkStages;
                if (!load) {
                    mbar_arrive(ready(st));
                    return;
                }
                const uint32_t bytes = static_cast<uint32_t>(ch.rows) * sh.row_bytes;
                mbar_arrive_expect_tx(ready(st), bytes * static_cast<uint32_t>(ch.bcnt));
                for (int b = 0; b < ch.bcnt; ++b) bulk_load(saddr(st, b), emb + gaddr(ch, b), bytes, ready(st));
            };
            int filled = 0;
            for (; filled < min(mine, kBulkStages - 1); ++filled) fill(filled);
            int k = 0;
            for (; k < mine; ++k) {
                const int st = k % kBulkStages;
                if (!mbar_wait(computed(st), (k / kBulkStages) & 1)) break;
                const Chunk ch = chunk_of(k);
                const uint32_t bytes = static_cast<uint32_t>(ch.rows) * sh.row_bytes;
                for (int b = 0; b < ch.bcnt; ++b) bulk_store(out + gaddr(ch, b), saddr(st, b), bytes);
                bulk_commit_group();
                // The stage of chunk k + 2 held chunk k - 1, whose stores must have read it.
                if (filled < mine) {
                    bulk_wait_group_read_1();
                    fill(filled++);
                }
            }
            if (k < mine) raise_device_error(err_word, HATTN_ETIMEOUT);
            bulk_wait_group_all();
            // Loads of chunks never stored (only after a wait gave up) must land.
            for (int j = k; load && j < filled; ++j)
                if (!mbar_wait(ready(j % kBulkStages), (j / kBulkStages) & 1)) raise_device_error(err_word, HATTN_ETIMEOUT);
        }
        __syncwarp();
        return;
    }

    // Compute warps: a thread takes one 16-byte piece of a row (kP frequency pairs)
    // at one position and applies its sin/cos to that piece of every batch row.
    constexpr int kP = 8 / static_cast<int>(sizeof(T));
    const int pieces = sh.half_d / kP;
    const int ctid = tid - 32;
    for (int k = 0; k < mine; ++k) {
        const Chunk ch = chunk_of(k);
        const int st = k % kBulkStages;
        uint8_t* stage = smem + st * kBulkStageBytes;
        if (!__all_sync(0xffffffffu, mbar_wait(ready(st), (k / kBulkStages) & 1))) {
            if (lane == 0) raise_device_error(err_word, HATTN_ETIMEOUT);
            break;
        }
        for (int q = ctid; q < ch.rows * pieces; q += kComputeWarps * 32) {
            const int r = q / pieces, i0 = (q - r * pieces) * kP;
            float sn[kP], cs[kP];
#pragma unroll
            for (int j = 0; j < kP; ++j)
                pe_sincos(static_cast<float>(pos0 + ch.t0 + r), turns[i0 + j].x, turns[i0 + j].y, sn[j], cs[j]);
            uint8_t* piece = stage + r * sh.row_bytes + 2 * i0 * sizeof(T);
            for (int b = 0; b < ch.bcnt; ++b) {
                uint4* e = reinterpret_cast<uint4*>(piece + (size_t)b * sh.R * sh.row_bytes);
                const uint4 v = load ? *e : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < kP; ++j) {
                    if constexpr (sizeof(T) == 4) {
                        o[2 * j] = __float_as_uint(fmaf(emb_scale, __uint_as_float(w[2 * j]), sn[j]));
                        o[2 * j + 1] = __float_as_uint(fmaf(emb_scale, __uint_as_float(w[2 * j + 1]), cs[j]));
                    } else {
                        const __nv_bfloat162 x = __floats2bfloat162_rn(fmaf(emb_scale, __uint_as_float(w[j] << 16), sn[j]),
                                                                       fmaf(emb_scale, __uint_as_float(w[j] & 0xffff0000u), cs[j]));
                        o[j] = *reinterpret_cast<const uint32_t*>(&x);
                    }
                }
                *e = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        // This thread's writes become visible to the bulk stores; one arrival per warp.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(computed(st));
    }
}

template <typename T>
size_t bulk_smem_bytes()
{
    return kBulkStages * kBulkStageBytes + kBulkMaxHalfD * sizeof(float2) + 16 * kBulkStages + 128;
}

// The bulk path's chunk shape, or false when a row does not fit a stage, the
// turn table is too small, or the problem is too small to fill the SMs.
bool bulk_shape(int B, int n, int d_model, size_t esize, BulkShape* sh)
{
    const size_t row_bytes = (size_t)d_model * esize;
    if (row_bytes % 16 != 0 || row_bytes > kBulkStageBytes || d_model / 2 > kBulkMaxHalfD) return false;
    sh->B = B;
    sh->n = n;
    sh->half_d = d_model / 2;
    sh->row_bytes = static_cast<uint32_t>(row_bytes);
    sh->Bc = static_cast<int>(std::min<size_t>(B, kBulkStageBytes / row_bytes));
    sh->R = static_cast<int>(std::max<size_t>(1, std::min<size_t>(n, kBulkStageBytes / (sh->Bc * row_bytes))));
    sh->b_groups = (B + sh->Bc - 1) / sh->Bc;
    const long long chunks = (long long)((n + sh->R - 1) / sh->R) * sh->b_groups;
    if (chunks > 0x7fffffffLL) return false;
    sh->chunks = static_cast<int>(chunks);
    return true;
}

template <typename T>
cudaError_t launch_bulk(const void* emb, void* out, const BulkShape& sh, float emb_scale, int pos0,
                        int* err_word, cudaStream_t stream)
{
    const size_t smem = bulk_smem_bytes<T>();
    cudaError_t e = cudaFuncSetAttribute(pos_encoding_bulk_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 152;
    const int grid = std::min(sh.chunks, sms);
    const double step = -13.287712379549449 / sh.half_d;  // log2 of 10000^(-1/(d/2))
    pos_encoding_bulk_kernel<T><<<grid, kBulkThreads, smem, stream>>>(
        static_cast<const T*>(emb), static_cast<T*>(out), sh, emb_scale, pos0, step, err_word);
    return cudaGetLastError();
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
                                float emb_scale, int pos0, int* err_word, cudaStream_t stream)
{
    // Bulk copies through shared memory when every row is a 16-byte multiple at
    // 16-byte aligned addresses and the problem (>= 16 MB, a chunk per SM) is
    // large enough for the ring to run full.
    const size_t esize = dtype == HATTN_F32 ? 4 : 2;
    BulkShape sh;
    if (aligned(out, 16) && (!emb || aligned(emb, 16)) && bulk_shape(B, n, d_model, esize, &sh) &&
        (double)B * n * d_model * esize >= 16.0 * (1 << 20) && sh.chunks >= 152) {
        return dtype == HATTN_F32 ? launch_bulk<float>(emb, out, sh, emb_scale, pos0, err_word, stream)
                                  : launch_bulk<__nv_bfloat16>(emb, out, sh, emb_scale, pos0, err_word, stream);
    }
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
