// Tensor-core GEMMs of the post-norm MHA sublayer (bf16 operands, fp32
// accumulation in TMEM), for sm_103a.
//
//   proj_gemm:    C = A . W for up to three independent problems in one launch
//                 (Q = x_q Wq, K = x_kv Wk, V = x_kv Wv). C is row-major
//                 [M, h*d], which is already the [B, n, h, d] layout the
//                 attention kernel reads (heads concatenated along features).
//                 An optional per-column bias and ReLU make the same kernel the
//                 first layer of the feed-forward sublayer, max(0, x W1 + b1).
//   outproj_ln:   y = LayerNorm(x + A . Wo [+ b]) * gamma + beta, one CTA per 128 rows
//                 holding the whole d_model-wide row in TMEM, so the residual
//                 add, the mean/variance and the normalisation run in the
//                 epilogue on fp32 values and y is rounded to bf16 once.
//
// Operands arrive by TMA with 128-byte swizzle: A as 128-row x 64-column
// K-major boxes, W ([K][N] row-major, i.e. N-major) as 64-row x 64-column
// boxes. Warp 0 issues the copies, warp 1 (one thread) the tcgen05 MMAs, and
// warps 2-5 run the epilogue; thread r of the epilogue owns output row r (TMEM
// lane r). All mbarrier waits are bounded.
//
// Sources: the projections Q = X W^Q etc. ([hex4c59 "读懂 Attention Is All You
// Need", §Q、K、V 是三种计算角色]), W^O after the concatenated heads
// (§多头注意力让一次读取有多组投影), LayerNorm(x + F(x)) (§Add & Norm 里究竟
// 发生了什么？); the feed-forward sublayer LayerNorm(x + max(0, x W1 + b1) W2 + b2)
// ([devpress "【深度学习】Transformer（Attention Is All You Need）", §2.3]).
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 192;
constexpr int kWarpLoad = 0;
constexpr int kWarpMma = 1;
constexpr uint32_t kABoxBytes = 128 * 64 * 2;  // A box: 128 rows x 64 columns
constexpr uint32_t kWBoxBytes = 64 * 64 * 2;   // W box: 64 rows x 64 columns

// ------------------------------------------------------------------ shared pieces

struct Ring {
    uint32_t full0, empty0, acc, slot;
};

__device__ __forceinline__ void gemm_setup(uint32_t sbar, int stages, uint32_t* tmem_slot,
                                           uint32_t tmem_cols, int warp)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(sbar + 8u * s, 1);             // full
            mbar_init(sbar + 8u * (stages + s), 1);  // empty
        }
        mbar_init(sbar + 8u * (2 * stages), 1);  // accumulator ready
        mbar_init(sbar + 8u * (2 * stages + 1), 1);  // drain
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ __forceinline__ void gemm_teardown(uint32_t tmem, uint32_t cols, int warp)
{
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, cols);
    }
}

// ------------------------------------------------------------------ projection GEMM

constexpr int kProjBN = 128;
constexpr int kProjStages = 3;
constexpr uint32_t kProjStageBytes = kABoxBytes + 2 * kWBoxBytes;
constexpr int kProjOffBar = kProjStages * kProjStageBytes;
constexpr int kProjSmem = kProjOffBar + 8 * (2 * kProjStages + 2) + 16 + 1024;
constexpr uint32_t kProjIdesc = idesc_bf16_f32(128, kProjBN, false, true);

struct ProjParams {
    void* c[3];
    const float* bias[3];
    int relu[3];
    int M[3], N[3];
    int K;
    int tiles_n[3];
    int tile_start[4];
    int* err_word;
};

__global__ void __launch_bounds__(kThreads, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                     const __grid_constant__ CUtensorMap a2, const __grid_constant__ CUtensorMap w0,
                     const __grid_constant__ CUtensorMap w1, const __grid_constant__ CUtensorMap w2,
                     const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sbar = sbase + kProjOffBar;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kProjOffBar + 8 * (2 * kProjStages + 2));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int tile = blockIdx.x;
    const int prob = tile < p.tile_start[1] ? 0 : (tile < p.tile_start[2] ? 1 : 2);
    const int local = tile - p.tile_start[prob];
    const int tm = local / p.tiles_n[prob], tn = local % p.tiles_n[prob];
    const CUtensorMap* am = prob == 0 ? &a0 : (prob == 1 ? &a1 : &a2);
    const CUtensorMap* wm = prob == 0 ? &w0 : (prob == 1 ? &w1 : &w2);
    const int kblocks = p.K / 64;

    gemm_setup(sbar, kProjStages, tmem_slot, kProjBN, warp);
    const uint32_t tmem = *tmem_slot;
    const uint32_t bar_acc = sbar + 8u * (2 * kProjStages);
    const uint32_t bar_drain = bar_acc + 8u;

    if (warp == kWarpLoad) {
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kProjStages;
                const uint32_t ph = (kb / kProjStages) & 1;
                if (!mbar_wait(sbar + 8u * (kProjStages + s), ph ^ 1)) { ok = false; break; }
                const uint32_t full = sbar + 8u * s;
                const uint32_t st = sbase + s * kProjStageBytes;
                mbar_arrive_expect_tx(full, kProjStageBytes);
                tma_load_2d(st, am, full, kb * 64, tm * 128);
                tma_load_2d(st + kABoxBytes, wm, full, tn * kProjBN, kb * 64);
                tma_load_2d(st + kABoxBytes + kWBoxBytes, wm, full, tn * kProjBN + 64, kb * 64);
                ++issued;
            }
            if (!ok) raise_device_error(p.err_word, HATTN_ETIMEOUT);
            for (int kb = max(0, issued - kProjStages); kb < issued; ++kb)
                mbar_wait(sbar + 8u * (kb % kProjStages), (kb / kProjStages) & 1);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kProjStages;
                const uint32_t ph = (kb / kProjStages) & 1;
                if (!mbar_wait(sbar + 8u * s, ph)) { ok = false; break; }
                tc_fence_after();
                const uint32_t st = sbase + s * kProjStageBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem, sdesc_sw128(st + ks * 32, 16, 1024),
                           sdesc_sw128(st + kABoxBytes + ks * 2048, kWBoxBytes, 1024), kProjIdesc,
                           (kb > 0 || ks > 0) ? 1u : 0u);
                mma_commit(sbar + 8u * (kProjStages + s));
            }
            if (ok) mma_commit(bar_acc);
            else raise_device_error(p.err_word, HATTN_ETIMEOUT);
            mma_commit(bar_drain);
            mbar_wait(bar_drain, 0);
        }
        __syncwarp();
    } else {
        const int wq = warp % 4;
        const int row = tm * 128 + wq * 32 + lane;
        bool got = mbar_wait(bar_acc, 0);
        if (__all_sync(0xffffffffu, got)) {
            tc_fence_after();
            __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(p.c[prob]) + (size_t)row * p.N[prob];
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
            const float* bias = p.bias[prob];
            const bool relu = p.relu[prob] != 0;
#pragma unroll
            for (int c = 0; c < kProjBN / 32; ++c) {
                uint32_t acc[32];
                tmem_ld_x32(lane_base + 32 * c, acc);
                const int col = tn * kProjBN + 32 * c;
                if (bias && col < p.N[prob]) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float v = __uint_as_float(acc[i]) + __ldg(bias + col + i);
                        if (relu) v = fmaxf(v, 0.0f);
                        acc[i] = __float_as_uint(v);
                    }
                } else if (relu) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] = __float_as_uint(fmaxf(__uint_as_float(acc[i]), 0.0f));
                }
                if (row < p.M[prob] && col < p.N[prob]) {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            w[i] = pack_bf16x2(__uint_as_float(acc[8 * v4 + 2 * i]),
                                               __uint_as_float(acc[8 * v4 + 2 * i + 1]));
                        st_global_v4(crow + col + 8 * v4, w[0], w[1], w[2], w[3]);
                    }
                }
            }
        } else {
            raise_device_error(p.err_word, HATTN_ETIMEOUT);
        }
    }
    gemm_teardown(tmem, kProjBN, warp);
}

// ------------------------------------------------------------------ out-projection + LayerNorm

constexpr int kLnMaxN = 512;
constexpr int kLnStages = 2;
constexpr uint32_t kLnStageBytes = kABoxBytes + (kLnMaxN / 64) * kWBoxBytes;
constexpr int kLnOffBar = kLnStages * kLnStageBytes;
constexpr int kLnSmem = kLnOffBar + 8 * (2 * kLnStages + 2) + 16 + 1024;

struct LnParams {
    const __nv_bfloat16* x;
    const float* bias;
    const float* gamma;
    const float* beta;
    float eps;
    __nv_bfloat16* y;
    int M, N, K;
    int* err_word;
};

__global__ void __launch_bounds__(kThreads, 1)
    outproj_ln_kernel(const __grid_constant__ CUtensorMap am, const __grid_constant__ CUtensorMap wm,
                      const LnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sbar = sbase + kLnOffBar;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kLnOffBar + 8 * (2 * kLnStages + 2));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tm = blockIdx.x;
    const int kblocks = p.K / 64;
    const int nboxes = p.N / 64;
    const uint32_t stage_tx = kABoxBytes + nboxes * kWBoxBytes;

    gemm_setup(sbar, kLnStages, tmem_slot, 512, warp);
    const uint32_t tmem = *tmem_slot;
    const uint32_t bar_acc = sbar + 8u * (2 * kLnStages);
    const uint32_t bar_drain = bar_acc + 8u;

    if (warp == kWarpLoad) {
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kLnStages;
                const uint32_t ph = (kb / kLnStages) & 1;
                if (!mbar_wait(sbar + 8u * (kLnStages + s), ph ^ 1)) { ok = false; break; }
                const uint32_t full = sbar + 8u * s;
                const uint32_t st = sbase + s * kLnStageBytes;
                mbar_arrive_expect_tx(full, stage_tx);
                tma_load_2d(st, &am, full, kb * 64, tm * 128);
                for (int x = 0; x < nboxes; ++x)
                    tma_load_2d(st + kABoxBytes + x * kWBoxBytes, &wm, full, x * 64, kb * 64);
                ++issued;
            }
            if (!ok) raise_device_error(p.err_word, HATTN_ETIMEOUT);
            for (int kb = max(0, issued - kLnStages); kb < issued; ++kb)
                mbar_wait(sbar + 8u * (kb % kLnStages), (kb / kLnStages) & 1);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kLnStages;
                const uint32_t ph = (kb / kLnStages) & 1;
                if (!mbar_wait(sbar + 8u * s, ph)) { ok = false; break; }
                tc_fence_after();
                const uint32_t st = sbase + s * kLnStageBytes;
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a_desc = sdesc_sw128(st + ks * 32, 16, 1024);
                    for (int n0 = 0; n0 < p.N; n0 += 256) {
                        const int nn = min(256, p.N - n0);
                        const uint32_t b_addr = st + kABoxBytes + (n0 / 64) * kWBoxBytes + ks * 2048;
                        mma_ss(tmem + n0, a_desc, sdesc_sw128(b_addr, kWBoxBytes, 1024),
                               idesc_bf16_f32(128, nn, false, true), (kb > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                mma_commit(sbar + 8u * (kLnStages + s));
            }
            if (ok) mma_commit(bar_acc);
            else raise_device_error(p.err_word, HATTN_ETIMEOUT);
            mma_commit(bar_drain);
            mbar_wait(bar_drain, 0);
        }
        __syncwarp();
    } else {
        const int wq = warp % 4;
        const int row = tm * 128 + wq * 32 + lane;
        const bool valid = row < p.M;
        bool got = mbar_wait(bar_acc, 0);
        if (__all_sync(0xffffffffu, got)) {
            tc_fence_after();
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
            const __nv_bfloat16* xrow = p.x + (size_t)row * p.N;
            const int nchunks = p.N / 32;
            // Pass 1: z = acc + x (kept in TMEM), row sum.
            float sum = 0.0f;
            for (int c = 0; c < nchunks; ++c) {
                uint32_t z[32];
                tmem_ld_x32(lane_base + 32 * c, z);
                uint4 xv[4] = {};
                if (valid) {
                    const uint4* src = reinterpret_cast<const uint4*>(xrow + 32 * c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) xv[v4] = src[v4];
                }
                const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(xv);
                if (p.bias) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        z[i] = __float_as_uint(__uint_as_float(z[i]) + __ldg(p.bias + 32 * c + i));
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float zi = __uint_as_float(z[i]) + __bfloat162float(xb[i]);
                    sum += zi;
                    z[i] = __float_as_uint(zi);
                }
                tmem_st_x32(lane_base + 32 * c, z);
            }
            tmem_st_wait();
            const float mean = sum / static_cast<float>(p.N);
            // Pass 2: biased variance about the mean.
            float var = 0.0f;
            for (int c = 0; c < nchunks; ++c) {
                uint32_t z[32];
                tmem_ld_x32(lane_base + 32 * c, z);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float dz = __uint_as_float(z[i]) - mean;
                    var = fmaf(dz, dz, var);
                }
            }
            const float rstd = 1.0f / sqrtf(var / static_cast<float>(p.N) + p.eps);
            // Pass 3: normalise, scale, shift, round once to bf16.
            __nv_bfloat16* yrow = p.y + (size_t)row * p.N;
            for (int c = 0; c < nchunks; ++c) {
                uint32_t z[32];
                tmem_ld_x32(lane_base + 32 * c, z);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int col = 32 * c + 2 * i;
                    const float y0 = (__uint_as_float(z[2 * i]) - mean) * rstd * __ldg(p.gamma + col) +
                                     __ldg(p.beta + col);
                    const float y1 = (__uint_as_float(z[2 * i + 1]) - mean) * rstd *
                                         __ldg(p.gamma + col + 1) + __ldg(p.beta + col + 1);
                    w[i] = pack_bf16x2(y0, y1);
                }
                if (valid) {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        st_global_v4(yrow + 32 * c + 8 * v4, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                                     w[4 * v4 + 3]);
                }
            }
        } else {
            raise_device_error(p.err_word, HATTN_ETIMEOUT);
        }
    }
    gemm_teardown(tmem, 512, warp);
}

}  // namespace

cudaError_t launch_proj_gemm(const ProjProblem* problems, int count, cudaStream_t stream,
                             int* err_word)
{
    if (count < 1 || count > 3) return cudaErrorInvalidValue;
    ProjParams p{};
    p.K = problems[0].K;
    p.err_word = err_word;
    p.tile_start[0] = 0;
    for (int i = 0; i < 3; ++i) {
        const ProjProblem& pr = problems[i < count ? i : count - 1];
        if (pr.K != p.K || pr.K % 64 != 0 || pr.N % 64 != 0) return cudaErrorInvalidValue;
        p.c[i] = pr.c;
        p.bias[i] = pr.bias;
        p.relu[i] = pr.relu ? 1 : 0;
        p.M[i] = pr.M;
        p.N[i] = pr.N;
        p.tiles_n[i] = (pr.N + kProjBN - 1) / kProjBN;
        const int tiles = i < count ? ((pr.M + 127) / 128) * p.tiles_n[i] : 0;
        p.tile_start[i + 1] = p.tile_start[i] + tiles;
    }
    cudaError_t e = cudaFuncSetAttribute(proj_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem);
    if (e != cudaSuccess) return e;
    const ProjProblem& q0 = problems[0];
    const ProjProblem& q1 = problems[count > 1 ? 1 : 0];
    const ProjProblem& q2 = problems[count > 2 ? 2 : 0];
    proj_gemm_kernel<<<p.tile_start[3], kThreads, kProjSmem, stream>>>(q0.a, q1.a, q2.a, q0.w,
                                                                      q1.w, q2.w, p);
    return cudaGetLastError();
}

cudaError_t launch_outproj_ln(const OutProjLnArgs& a, cudaStream_t stream, int* err_word)
{
    if (a.N % 64 != 0 || a.N > kLnMaxN || a.K % 64 != 0) return cudaErrorInvalidValue;
    LnParams p;
    p.x = static_cast<const __nv_bfloat16*>(a.x);
    p.bias = a.bias;
    p.gamma = a.gamma;
    p.beta = a.beta;
    p.eps = a.eps;
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.err_word = err_word;
    cudaError_t e = cudaFuncSetAttribute(outproj_ln_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kLnSmem);
    if (e != cudaSuccess) return e;
    outproj_ln_kernel<<<(a.M + 127) / 128, kThreads, kLnSmem, stream>>>(a.a, a.wo, p);
    return cudaGetLastError();
}

}  // namespace hattn
