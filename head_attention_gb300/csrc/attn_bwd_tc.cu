// Tensor-core attention backward for sm_103a (bf16 in/out, fp32 accumulation,
// d_k == d_v == D in {64, 128}, scale > 0).
//
// The gradients of sum(dO * O), O = softmax(scale Q K^T [masked]) V, per (b, h):
//   P = 2^(scale log2(e) Q K^T - lse2)   (lse2: the forward's log-sum-exp in base 2)
//   dP = dO V^T,  dS = P (dP - D),  D_t = dO_t . O_t
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K
// Training sends the loss gradient back through the attention weights
// ("读懂 Attention Is All You Need", §参数是怎样学出来的？); these are the chain
// rule applied to the forward (§六步算完一行注意力).
//
// Two CTA kinds in one grid, no atomics, both with 10 warps: warp 0 issues the
// TMA copies, warp 1 (one thread) the tcgen05 MMAs and owns TMEM (the control
// warps come first because the warp schedulers favour lower-numbered ready
// warps); row warps 2-9: warp w owns TMEM lanes 32 (w % 4) .. + 31 (one row
// each: a key in the first kernel, a query in the second), and warps 2-5 and
// 6-9 take the two halves of each block's 128 columns.
//
//   key_grads_tc:   a CTA keeps one 128-key block of K and V in shared memory
//                   and streams 128-query blocks of Q, dO, lse2 and D through a
//                   2-stage (D = 128) / 3-stage (D = 64) ring. Per block: S^T = K Q^T and dP^T = V dO^T (SS
//                   MMAs into TMEM); the row warps form P^T and dS^T, written back
//                   to TMEM as bf16 over S^T and dP^T; then dV += P^T dO and
//                   dK += dS^T Q (TS MMAs). TMEM: S^T | dP^T | dV | dK.
//                   Each block runs as two halves of 64 queries (N = 64 MMAs,
//                   one handoff per half), pipelined: the row warps of half 1
//                   work on block i while the tensor pipe runs half 0's dV/dK of
//                   block i and half 0's S^T/dP^T of block i + 1.
//   query_grads_tc: a CTA keeps one 128-query block of Q and dO and streams
//                   128-key blocks of K and V. Per block: S = Q K^T, dP = dO V^T,
//                   dS (bf16, over S), dQ += dS K. TMEM: S | dP | dQ. The same
//                   pipeline over halves of 64 keys.
// Causal: blocks entirely above the diagonal are skipped; key padding: key
// blocks at or past key_lens[b] are skipped, the last one masked. All waits are
// bounded; a wait that gives up raises HATTN_ETIMEOUT, and the CTA drains its
// copies and MMAs before it frees TMEM.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 320;
constexpr int kWarpLoad = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpRow0 = 2;  // row warps 2-9
constexpr int kRowWarps = 8;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // 128 rows x 64 bf16 columns
// Ring depth: three stages where they fit (D = 64), else two.
template <int D>
constexpr int kStages = D == 64 ? 3 : 2;

template <int D>
struct Tile {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBytes = 128 * D * 2;
    static constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, false, false);
    static constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, false, true);
};

// The 64-row half h of a K-major 128-row tile starts 8 row groups (8 KB) in.
constexpr uint32_t kHalfRowsBytes = 64 * 128;

// X_h = A . B_h^T over the D columns, B_h the 64-row half h of a K-major tile
// (into 64 TMEM columns from d_tmem): one column half of a block, so the row
// warps of that half can start while the other half is multiplied.
template <int D>
__device__ __forceinline__ void mma_abt_half(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, int h)
{
    const uint64_t bh = b_desc + ((h * kHalfRowsBytes) >> 4);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = ((ks / 4) * kBoxBytes + (ks % 4) * 32) >> 4;
        mma_ss(d_tmem, a_desc + off, bh + off, Tile<D>::kIdescHalf, ks > 0 ? 1u : 0u);
    }
}

// Acc (+)= X_h . T_h over the column half h of X (128 x 128 bf16 in TMEM) and
// the matching rows 64 h .. 64 h + 63 of a 128-row tile T used MN-major (its D
// columns are the output columns). X's column pairs are packed in two runs of
// 32 TMEM columns, at x_tmem (X columns 0-63) and x_tmem + 64 (X columns
// 64-127): each half is written by its own row warps inside the columns they
// have already read.
template <int D>
__device__ __forceinline__ void mma_xt_half(uint32_t d_tmem, uint32_t x_tmem, uint64_t t_desc, int h,
                                            bool accumulate)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int ks = 4 * h + k;
        mma_ts(d_tmem, x_tmem + h * 64 + k * 8, t_desc + ((ks * 2048) >> 4), Tile<D>::kIdescAcc,
               (accumulate || ks > 0) ? 1u : 0u);
    }
}

struct BwdTcParams {
    int B, h, n_q, n_k, nqp;  // nqp: n_q rounded up to 128 (row stride of lse2 / dsum)
    int mask_kind;
    float scale, scale_log2;
    const int32_t* key_lens;
    const float* lse2;  // [B, h, nqp], minus the base-2 log-sum-exp of scale*q.k (-inf past n_q)
    const float* dsum;  // [B, h, nqp], -D = -(dO . O) (0 past n_q)
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int* err_word;
};

__device__ __forceinline__ void store_row(__nv_bfloat16* dst, uint32_t tmem_row, int ncols, float mul,
                                          bool valid)
{
    for (int c = 0; c < ncols; c += 32) {
        uint32_t v[32];
        tmem_ld_x32(tmem_row + c, v);
        if (valid) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                st_global_v4(dst + c + 8 * v4,
                             pack_bf16x2(mul * __uint_as_float(v[8 * v4]), mul * __uint_as_float(v[8 * v4 + 1])),
                             pack_bf16x2(mul * __uint_as_float(v[8 * v4 + 2]), mul * __uint_as_float(v[8 * v4 + 3])),
                             pack_bf16x2(mul * __uint_as_float(v[8 * v4 + 4]), mul * __uint_as_float(v[8 * v4 + 5])),
                             pack_bf16x2(mul * __uint_as_float(v[8 * v4 + 6]), mul * __uint_as_float(v[8 * v4 + 7])));
        }
    }
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* dst, int ncols)
{
    for (int c = 0; c < ncols; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
}

// ------------------------------------------------------------------ dK, dV

template <int D>
struct KCfg {
    using T = Tile<D>;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = T::kBytes;
    static constexpr int kOffStage = 2 * T::kBytes;  // stage s: Q, dO, lse2[128], D[128]
    static constexpr int kStageBytes = 2 * T::kBytes + 1024;
    static constexpr int kOffBar = kOffStage + kStages<D> * kStageBytes;
    // kBarS + h: S^T and dP^T of query half h ready; kBarP + h: its P^T and dS^T written.
    static constexpr int kBarKV = 0, kBarFull = 1, kBarEmpty = 1 + kStages<D>, kBarS = 1 + 2 * kStages<D>,
                         kBarP = kBarS + 2, kBarO = kBarP + 2, kBarDrain = kBarO + 1,
                         kNumBars = kBarDrain + 1;
    static constexpr int kOffSlot = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffSlot + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
};

// CTA `cta` of the key-gradient work: key block kblk = cta / (B h) of head
// cta % (B h) (with the causal mask, low key blocks meet the most query blocks).
template <int D>
__device__ __forceinline__ void key_grads_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                             const CUtensorMap& tm_v, const CUtensorMap& tm_g,
                                             const BwdTcParams& p, int cta)
{
    using C = KCfg<D>;
    using T = Tile<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffSlot);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int kblk = cta / (p.B * p.h);
    const int bh = cta % (p.B * p.h);
    const int b = bh / p.h, head = bh % p.h;
    const int key0 = kblk * 128;
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;
    const int kv_len = (p.mask_kind & HATTN_MASK_KEY_PADDING) ? p.key_lens[b] : p.n_k;
    const size_t row_elems = (size_t)p.h * D;

    if (kv_len < 1 || kv_len > p.n_k) {
        if (threadIdx.x < 128 && key0 + threadIdx.x < p.n_k) {
            const size_t off = ((size_t)b * p.n_k + key0 + threadIdx.x) * row_elems + (size_t)head * D;
            zero_row(p.dk + off, D);
            zero_row(p.dv + off, D);
        }
        if (threadIdx.x == 0) raise_device_error(p.err_word, HATTN_EKEYLEN);
        return;
    }
    // Query blocks this key block meets: causal starts at the diagonal block.
    const int n_qblk = (p.n_q + 127) / 128;
    const int qb_first = causal ? kblk : 0;
    const int nblk = key0 < kv_len ? max(0, n_qblk - qb_first) : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarKV), 1);
        for (int s = 0; s < kStages<D>; ++s) {
            mbar_init(bar(C::kBarFull + s), 1);
            mbar_init(bar(C::kBarEmpty + s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(C::kBarS + h), 1);
            mbar_init(bar(C::kBarP + h), kRowWarps / 2);
        }
        mbar_init(bar(C::kBarO), 1);
        mbar_init(bar(C::kBarDrain), 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpLoad) {
        if (lane == 0 && nblk > 0) {
            mbar_arrive_expect_tx(bar(C::kBarKV), 2 * T::kBytes);
            for (int x = 0; x < T::kBoxes; ++x) {
                tma_load_4d(sbase + C::kOffK + x * kBoxBytes, &tm_k, bar(C::kBarKV), x * 64, head, key0, b);
                tma_load_4d(sbase + C::kOffV + x * kBoxBytes, &tm_v, bar(C::kBarKV), x * 64, head, key0, b);
            }
            const float* lse_row = p.lse2 + ((size_t)b * p.h + head) * p.nqp;
            const float* d_row = p.dsum + ((size_t)b * p.h + head) * p.nqp;
            int issued = 0;
            for (int i = 0; i < nblk; ++i) {
                const int s = i % kStages<D>;
                if (!mbar_wait(bar(C::kBarEmpty + s), ((i / kStages<D>) & 1) ^ 1)) {
                    raise_device_error(p.err_word, HATTN_ETIMEOUT);
                    break;
                }
                const int q0 = (qb_first + i) * 128;
                const uint32_t st = sbase + C::kOffStage + s * C::kStageBytes;
                mbar_arrive_expect_tx(bar(C::kBarFull + s), 2 * T::kBytes + 1024);
                for (int x = 0; x < T::kBoxes; ++x) {
                    tma_load_4d(st + x * kBoxBytes, &tm_q, bar(C::kBarFull + s), x * 64, head, q0, b);
                    tma_load_4d(st + T::kBytes + x * kBoxBytes, &tm_g, bar(C::kBarFull + s), x * 64, head, q0, b);
                }
                bulk_load(st + 2 * T::kBytes, lse_row + q0, 512, bar(C::kBarFull + s));
                bulk_load(st + 2 * T::kBytes + 512, d_row + q0, 512, bar(C::kBarFull + s));
                ++issued;
            }
            // Every copy this CTA started must land before the CTA may exit.
            mbar_wait(bar(C::kBarKV), 0);
            for (int i = max(0, issued - kStages<D>); i < issued; ++i)
                mbar_wait(bar(C::kBarFull + i % kStages<D>), (i / kStages<D>) & 1);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0 && nblk > 0) {
            const uint64_t k_desc = sdesc_sw128(sbase + C::kOffK, 16, 1024);
            const uint64_t v_desc = sdesc_sw128(sbase + C::kOffV, 16, 1024);
            auto stage = [&](int i) { return sbase + C::kOffStage + (i % kStages<D>) * C::kStageBytes; };
            // S^T = K Q^T and dP^T = V dO^T for the queries of half h of block i.
            auto issue_sdp = [&](int i, int h) {
                const uint32_t st = stage(i);
                mma_abt_half<D>(tmem + C::kColS + 64 * h, k_desc, sdesc_sw128(st, 16, 1024), h);
                mma_abt_half<D>(tmem + C::kColDP + 64 * h, v_desc, sdesc_sw128(st + T::kBytes, 16, 1024), h);
                mma_commit(bar(C::kBarS + h));
            };
            // dV += P^T dO and dK += dS^T Q over the queries of half h (Q / dO used MN-major).
            auto issue_acc = [&](int i, int h) {
                const uint32_t st = stage(i);
                mma_xt_half<D>(tmem + C::kColDV, tmem + C::kColS, sdesc_sw128(st + T::kBytes, kBoxBytes, 1024), h, i > 0);
                mma_xt_half<D>(tmem + C::kColDK, tmem + C::kColDP, sdesc_sw128(st, kBoxBytes, 1024), h, i > 0);
            };
            // Two-stage pipeline over the query halves of each block: while the row
            // warps of half 1 work on block i, the tensor pipe runs half 0's dV/dK of
            // block i and half 0's S^T/dP^T of block i + 1. Each S^T/dP^T half
            // overwrites TMEM columns whose P^T/dS^T were read by MMAs issued before it.
            bool ok = mbar_wait(bar(C::kBarKV), 0) && mbar_wait(bar(C::kBarFull), 0);
            if (ok) {
                tc_fence_after();
                issue_sdp(0, 0);
                issue_sdp(0, 1);
            }
            for (int i = 0; ok && i < nblk; ++i) {
                const bool next = i + 1 < nblk;
                if (!mbar_wait(bar(C::kBarP), i & 1)) { ok = false; break; }
                tc_fence_after();
                issue_acc(i, 0);
                if (next) {
                    const int s1 = (i + 1) % kStages<D>;
                    if (!mbar_wait(bar(C::kBarFull + s1), ((i + 1) / kStages<D>) & 1)) { ok = false; break; }
                    tc_fence_after();
                    issue_sdp(i + 1, 0);
                }
                if (!mbar_wait(bar(C::kBarP + 1), i & 1)) { ok = false; break; }
                tc_fence_after();
                issue_acc(i, 1);
                mma_commit(bar(C::kBarEmpty + i % kStages<D>));
                if (next) issue_sdp(i + 1, 1);
            }
            if (ok) mma_commit(bar(C::kBarO));
            else raise_device_error(p.err_word, HATTN_ETIMEOUT);
            mma_commit(bar(C::kBarDrain));
            mbar_wait(bar(C::kBarDrain), 0);
        }
        __syncwarp();
    } else {
        // Row warps: warp w owns keys key0 + 32 (w % 4) .. + 31 (the TMEM lanes of
        // its quadrant) and query columns [64 half, 64 half + 64) of each block.
        const int quad = warp % 4, half = (warp - kWarpRow0) / 4;
        const int r = quad * 32 + lane;
        const int key = key0 + r;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const bool key_ok = key < kv_len;
        const size_t off = ((size_t)b * p.n_k + key) * row_elems + (size_t)head * D;
        const uint64_t c2 = f32x2(p.scale_log2, p.scale_log2);
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            const int s = i % kStages<D>;
            const int q0 = (qb_first + i) * 128;
            if (ok) {
                const bool got = mbar_wait(bar(C::kBarFull + s), (i / kStages<D>) & 1) &&
                                 mbar_wait(bar(C::kBarS + half), i & 1);
                ok = __all_sync(0xffffffffu, got);
            }
            if (!ok) continue;
            tc_fence_after();
            // Per query column: -lse2 and -D of this stage (16-byte broadcast reads).
            const float* nlse_s = reinterpret_cast<const float*>(smem + C::kOffStage + s * C::kStageBytes + 2 * T::kBytes) + 64 * half;
            const float* nd_s = nlse_s + 128;
            // Keys at or past the length, or after every query of the block (causal), see nothing.
            const bool row_live = key_ok && !(causal && key > q0 + 127);
            const bool diag = causal && key0 + 127 > q0;  // this block straddles the diagonal
            // Without the diagonal or the query tail, no element of the block is masked.
            const bool plain = !diag && q0 + 127 < p.n_q;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const uint32_t col = 64 * half + 32 * c;  // this chunk's first S^T / dP^T column
                uint32_t sv[32], pv[32];
                tmem_ld_x32(lane_base + C::kColS + col, sv);
                tmem_ld_x32(lane_base + C::kColDP + col, pv);
                uint32_t pk[16], dk[16];
                if (plain) {
                    const float4* l4 = reinterpret_cast<const float4*>(nlse_s + 32 * c);
                    const float4* d4 = reinterpret_cast<const float4*>(nd_s + 32 * c);
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 L = l4[e4], Dn = d4[e4];
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int e = 4 * e4 + 2 * h2;
                            const uint64_t x2 = fma_f32x2(f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2,
                                                          h2 ? f32x2(L.z, L.w) : f32x2(L.x, L.y));
                            float x0, x1;
                            f32x2_split(x2, x0, x1);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            const uint64_t t2 = add_f32x2(f32x2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])),
                                                          h2 ? f32x2(Dn.z, Dn.w) : f32x2(Dn.x, Dn.y));
                            float t0, t1;
                            f32x2_split(t2, t0, t1);
                            pk[e / 2] = pack_bf16x2(p0, p1);
                            dk[e / 2] = pack_bf16x2(p0 * t0, p1 * t1);
                        }
                    }
                    if (!row_live) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pk[e] = dk[e] = 0u;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float pr[2], ds[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int q = q0 + col + e + u;
                            const bool vis = row_live && q < p.n_q && !(diag && key > q);
                            const float x = fmaf(__uint_as_float(sv[e + u]), p.scale_log2, nlse_s[32 * c + e + u]);
                            pr[u] = vis ? ex2_approx(x) : 0.0f;
                            ds[u] = pr[u] * (__uint_as_float(pv[e + u]) + nd_s[32 * c + e + u]);
                        }
                        pk[e / 2] = pack_bf16x2(pr[0], pr[1]);
                        dk[e / 2] = pack_bf16x2(ds[0], ds[1]);
                    }
                }
                // bf16 P^T over S^T's columns [64 half + 16 c, + 16), dS^T over dP^T's:
                // columns this warp has already read.
                tmem_st_x16(lane_base + C::kColS + 64 * half + 16 * c, pk);
                tmem_st_x16(lane_base + C::kColDP + 64 * half + 16 * c, dk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarP + half));
        }
        // Each warp of the quadrant stores half of the D columns of dV and dK.
        constexpr int kHalfD = D / 2;
        if (nblk == 0) {
            if (key < p.n_k) {
                zero_row(p.dk + off + kHalfD * half, kHalfD);
                zero_row(p.dv + off + kHalfD * half, kHalfD);
            }
        } else if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarO), 0));
            if (ok) {
                tc_fence_after();
                store_row(p.dv + off + kHalfD * half, lane_base + C::kColDV + kHalfD * half, kHalfD, 1.0f, key < p.n_k);
                store_row(p.dk + off + kHalfD * half, lane_base + C::kColDK + kHalfD * half, kHalfD, p.scale, key < p.n_k);
            }
        }
        if (!ok) raise_device_error(p.err_word, HATTN_ETIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ dQ

template <int D>
struct QCfg {
    using T = Tile<D>;
    static constexpr int kOffQ = 0;
    static constexpr int kOffG = T::kBytes;
    static constexpr int kOffStage = 2 * T::kBytes;  // stage s: K, V
    static constexpr int kStageBytes = 2 * T::kBytes;
    static constexpr int kOffBar = kOffStage + kStages<D> * kStageBytes;
    // kBarS + h: S and dP of key half h ready; kBarP + h: its dS written.
    static constexpr int kBarQG = 0, kBarFull = 1, kBarEmpty = 1 + kStages<D>, kBarS = 1 + 2 * kStages<D>,
                         kBarP = kBarS + 2, kBarO = kBarP + 2, kBarDrain = kBarO + 1,
                         kNumBars = kBarDrain + 1;
    static constexpr int kOffSlot = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffSlot + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
};

// CTA `cta` of the query-gradient work: query block n_qblk - 1 - cta / (B h)
// of head cta % (B h) (with the causal mask, high query blocks meet the most key blocks).
template <int D>
__device__ __forceinline__ void query_grads_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                               const CUtensorMap& tm_v, const CUtensorMap& tm_g,
                                               const BwdTcParams& p, int cta)
{
    using C = QCfg<D>;
    using T = Tile<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffSlot);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int n_qblk = (p.n_q + 127) / 128;
    const int qblk = n_qblk - 1 - cta / (p.B * p.h);
    const int bh = cta % (p.B * p.h);
    const int b = bh / p.h, head = bh % p.h;
    const int q0 = qblk * 128;
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;
    const int kv_len = (p.mask_kind & HATTN_MASK_KEY_PADDING) ? p.key_lens[b] : p.n_k;
    const size_t row_elems = (size_t)p.h * D;

    if (kv_len < 1 || kv_len > p.n_k) {
        if (threadIdx.x < 128 && q0 + threadIdx.x < p.n_q)
            zero_row(p.dq + ((size_t)b * p.n_q + q0 + threadIdx.x) * row_elems + (size_t)head * D, D);
        return;  // the key-gradient kernel raises the error
    }
    int nblk = (kv_len + 127) / 128;
    if (causal) nblk = min(nblk, qblk + 1);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarQG), 1);
        for (int s = 0; s < kStages<D>; ++s) {
            mbar_init(bar(C::kBarFull + s), 1);
            mbar_init(bar(C::kBarEmpty + s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(C::kBarS + h), 1);
            mbar_init(bar(C::kBarP + h), kRowWarps / 2);
        }
        mbar_init(bar(C::kBarO), 1);
        mbar_init(bar(C::kBarDrain), 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpLoad) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::kBarQG), 2 * T::kBytes);
            for (int x = 0; x < T::kBoxes; ++x) {
                tma_load_4d(sbase + C::kOffQ + x * kBoxBytes, &tm_q, bar(C::kBarQG), x * 64, head, q0, b);
                tma_load_4d(sbase + C::kOffG + x * kBoxBytes, &tm_g, bar(C::kBarQG), x * 64, head, q0, b);
            }
            int issued = 0;
            for (int j = 0; j < nblk; ++j) {
                const int s = j % kStages<D>;
                if (!mbar_wait(bar(C::kBarEmpty + s), ((j / kStages<D>) & 1) ^ 1)) {
                    raise_device_error(p.err_word, HATTN_ETIMEOUT);
                    break;
                }
                const uint32_t st = sbase + C::kOffStage + s * C::kStageBytes;
                mbar_arrive_expect_tx(bar(C::kBarFull + s), 2 * T::kBytes);
                for (int x = 0; x < T::kBoxes; ++x) {
                    tma_load_4d(st + x * kBoxBytes, &tm_k, bar(C::kBarFull + s), x * 64, head, j * 128, b);
                    tma_load_4d(st + T::kBytes + x * kBoxBytes, &tm_v, bar(C::kBarFull + s), x * 64, head, j * 128, b);
                }
                ++issued;
            }
            mbar_wait(bar(C::kBarQG), 0);
            for (int j = max(0, issued - kStages<D>); j < issued; ++j)
                mbar_wait(bar(C::kBarFull + j % kStages<D>), (j / kStages<D>) & 1);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            const uint64_t q_desc = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
            const uint64_t g_desc = sdesc_sw128(sbase + C::kOffG, 16, 1024);
            auto stage = [&](int j) { return sbase + C::kOffStage + (j % kStages<D>) * C::kStageBytes; };
            // S = Q K^T and dP = dO V^T for the keys of half h of block j.
            auto issue_sdp = [&](int j, int h) {
                const uint32_t st = stage(j);
                mma_abt_half<D>(tmem + C::kColS + 64 * h, q_desc, sdesc_sw128(st, 16, 1024), h);
                mma_abt_half<D>(tmem + C::kColDP + 64 * h, g_desc, sdesc_sw128(st + T::kBytes, 16, 1024), h);
                mma_commit(bar(C::kBarS + h));
            };
            // The same two-stage pipeline over key halves as the key-gradient CTAs.
            bool ok = mbar_wait(bar(C::kBarQG), 0) && (nblk == 0 || mbar_wait(bar(C::kBarFull), 0));
            if (ok && nblk > 0) {
                tc_fence_after();
                issue_sdp(0, 0);
                issue_sdp(0, 1);
            }
            for (int j = 0; ok && j < nblk; ++j) {
                const bool next = j + 1 < nblk;
                const uint32_t st = stage(j);
                if (!mbar_wait(bar(C::kBarP), j & 1)) { ok = false; break; }
                tc_fence_after();
                mma_xt_half<D>(tmem + C::kColDQ, tmem + C::kColS, sdesc_sw128(st, kBoxBytes, 1024), 0, j > 0);
                if (next) {
                    const int s1 = (j + 1) % kStages<D>;
                    if (!mbar_wait(bar(C::kBarFull + s1), ((j + 1) / kStages<D>) & 1)) { ok = false; break; }
                    tc_fence_after();
                    issue_sdp(j + 1, 0);
                }
                if (!mbar_wait(bar(C::kBarP + 1), j & 1)) { ok = false; break; }
                tc_fence_after();
                mma_xt_half<D>(tmem + C::kColDQ, tmem + C::kColS, sdesc_sw128(st, kBoxBytes, 1024), 1, j > 0);
                mma_commit(bar(C::kBarEmpty + j % kStages<D>));
                if (next) issue_sdp(j + 1, 1);
            }
            if (ok) mma_commit(bar(C::kBarO));
            else raise_device_error(p.err_word, HATTN_ETIMEOUT);
            mma_commit(bar(C::kBarDrain));
            mbar_wait(bar(C::kBarDrain), 0);
        }
        __syncwarp();
    } else {
        // Row warps: warp w owns queries q0 + 32 (w % 4) .. + 31 and key columns
        // [64 half, 64 half + 64) of each block.
        const int quad = warp % 4, half = (warp - kWarpRow0) / 4;
        const int r = quad * 32 + lane;
        const int q = q0 + r;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float nlse2 = q < p.n_q ? p.lse2[((size_t)b * p.h + head) * p.nqp + q] : 0.0f;  // -lse2
        const float nd = q < p.n_q ? p.dsum[((size_t)b * p.h + head) * p.nqp + q] : 0.0f;     // -D
        const uint64_t c2 = f32x2(p.scale_log2, p.scale_log2);
        const uint64_t nl2 = f32x2(nlse2, nlse2), nd2 = f32x2(nd, nd);
        const bool row_ok = q < p.n_q;
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            const int k0 = j * 128;
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarS + half), j & 1));
            if (!ok) continue;
            tc_fence_after();
            const bool edge = (k0 + 128 > kv_len) || (causal && k0 + 127 > q0);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const uint32_t col = 64 * half + 32 * c;
                uint32_t sv[32], pv[32];
                tmem_ld_x32(lane_base + C::kColS + col, sv);
                tmem_ld_x32(lane_base + C::kColDP + col, pv);
                uint32_t dk[16];
                if (!edge) {
                    // No key of the block is masked, so the packed path needs no per-element
                    // test (a query row past n_q is zeroed whole).
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const uint64_t x2 = fma_f32x2(f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nl2);
                        float x0, x1;
                        f32x2_split(x2, x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        const uint64_t t2 = add_f32x2(f32x2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), nd2);
                        float t0, t1;
                        f32x2_split(t2, t0, t1);
                        dk[e / 2] = pack_bf16x2(row_ok ? p0 * t0 : 0.0f, row_ok ? p1 * t1 : 0.0f);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float ds[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int key = k0 + col + e + u;
                            const bool vis = row_ok && !(key >= kv_len || (causal && key > q));
                            const float x = fmaf(__uint_as_float(sv[e + u]), p.scale_log2, nlse2);
                            const float pr = vis ? ex2_approx(x) : 0.0f;
                            ds[u] = pr * (__uint_as_float(pv[e + u]) + nd);
                        }
                        dk[e / 2] = pack_bf16x2(ds[0], ds[1]);
                    }
                }
                // bf16 dS over S's columns [64 half + 16 c, + 16), already read.
                tmem_st_x16(lane_base + C::kColS + 64 * half + 16 * c, dk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarP + half));
        }
        constexpr int kHalfD = D / 2;
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarO), 0));
            if (ok) {
                tc_fence_after();
                store_row(p.dq + ((size_t)b * p.n_q + q) * row_elems + (size_t)head * D + kHalfD * half,
                          lane_base + C::kColDQ + kHalfD * half, kHalfD, p.scale, row_ok);
            }
        }
        if (!ok) raise_device_error(p.err_word, HATTN_ETIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Both gradient computations in one grid: the query-gradient CTAs first, then
// the key-gradient CTAs, so the tail of one overlaps the other.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    grads_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                    const BwdTcParams p, int q_ctas)
{
    if (static_cast<int>(blockIdx.x) < q_ctas) query_grads_tc<D>(tm_q, tm_k, tm_v, tm_g, p, blockIdx.x);
    else key_grads_tc<D>(tm_q, tm_k, tm_v, tm_g, p, blockIdx.x - q_ctas);
}

template <int D>
cudaError_t launch_d(const AttnBwdArgs& a, const AttnMaps& m, const CUtensorMap& tm_g)
{
    BwdTcParams p;
    p.B = a.B;
    p.h = a.h;
    p.n_q = a.n_q;
    p.n_k = a.n_k;
    p.nqp = (a.n_q + 127) / 128 * 128;
    p.mask_kind = a.mask_kind;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.key_lens = a.key_lens;
    p.lse2 = a.lse2;
    p.dsum = a.dsum;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.err_word = a.err_word;
    const long long kctas = (long long)a.B * a.h * ((a.n_k + 127) / 128);
    const long long qctas = (long long)a.B * a.h * ((a.n_q + 127) / 128);
    if (kctas + qctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = KCfg<D>::kSmemBytes > QCfg<D>::kSmemBytes ? KCfg<D>::kSmemBytes : QCfg<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(grads_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    grads_tc_kernel<D><<<(unsigned)(kctas + qctas), kThreads, smem, a.stream>>>(m.q, m.k, m.v, tm_g, p,
                                                                               static_cast<int>(qctas));
    return cudaGetLastError();
}

}  // namespace

bool attn_bwd_tc_supported(const AttnBwdArgs& a)
{
    return a.dtype == HATTN_BF16 && a.d_k == a.d_v && (a.d_k == 64 || a.d_k == 128) && a.scale > 0.0f;
}

cudaError_t launch_attn_bwd_tc(const AttnBwdArgs& a, const AttnMaps& maps, const CUtensorMap& tm_dout)
{
    return a.d_k == 64 ? launch_d<64>(a, maps, tm_dout) : launch_d<128>(a, maps, tm_dout);
}

}  // namespace hattn
