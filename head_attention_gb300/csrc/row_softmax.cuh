// Per-row pieces of the streaming softmax shared by the tensor-core attention
// kernels: a thread owns one query row (one TMEM lane) and 128 raw scores q.k_j
// of one key block in registers.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"

namespace hattn {

// p = 2^(s * c - m) for the 128 scores of this thread's row, packed to bf16 and
// stored into 64 TMEM columns from p_taddr; the fp32 sum goes to acc. With
// kMax, the row max of the raw scores is computed alongside (on the ALU pipe,
// while the exponentials occupy MUFU and FMA) and returned.
template <bool kMax>
__device__ __forceinline__ float exp_block(const uint32_t (&sr)[128], uint64_t c2, uint64_t nm2,
                                           uint64_t (&acc)[4], uint32_t p_taddr)
{
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = 32 * q + 2 * i;
            const uint64_t x2 =
                fma_f32x2(f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nm2);
            float t0, t1;
            f32x2_split(x2, t0, t1);
            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            acc[i & 3] = add_f32x2(acc[i & 3], f32x2(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st_x16(p_taddr + 16 * q, pk);
        if (kMax) {
            const uint32_t* v = sr + 32 * q;
            float g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t* v8 = v + 8 * k;
                g[k] = max3f(max3f(__uint_as_float(v8[0]), __uint_as_float(v8[1]), __uint_as_float(v8[2])),
                             max3f(__uint_as_float(v8[3]), __uint_as_float(v8[4]), __uint_as_float(v8[5])),
                             fmaxf(__uint_as_float(v8[6]), __uint_as_float(v8[7])));
            }
            mx = max3f(mx, max3f(g[0], g[1], g[2]), g[3]);
        }
    }
    return mx;
}

// Row max of the 128 raw scores (a tree of independent 3-input maxima).
__device__ __forceinline__ float row_max(const uint32_t (&sr)[128])
{
    float part[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) {
        const uint32_t* v8 = sr + 8 * g;
        const float a = max3f(__uint_as_float(v8[0]), __uint_as_float(v8[1]), __uint_as_float(v8[2]));
        const float e = max3f(__uint_as_float(v8[3]), __uint_as_float(v8[4]), __uint_as_float(v8[5]));
        part[g] = max3f(a, e, fmaxf(__uint_as_float(v8[6]), __uint_as_float(v8[7])));
    }
#pragma unroll
    for (int g = 0; g < 5; ++g) part[g] = max3f(part[g], part[g + 5], part[g + 10]);
    return max3f(max3f(part[0], part[1], part[2]), part[3], fmaxf(part[4], part[15]));
}

}  // namespace hattn
