// Tensor-core attention forward for short sequences on sm_103a: bf16 in/out,
// fp32 accumulation, n_q <= 128 query rows, and n_k <= 256 keys at
// d_k == d_v == 64 or n_k <= 128 at d_k == d_v == 128.
//
// What it computes is the scaled dot-product attention of the pages on
// "Attention Is All You Need" (hex4c59 §把所有位置合并，就是那条核心公式), with
// the decoder's causal mask and the cross-attention key padding (hex4c59
// §掩码必须在 softmax 之前生效, §解码器有两种读取): these are the short,
// per-sentence uses, where a head's whole key range fits one or two 128-key
// blocks and the time goes to latency (launch, one DRAM round trip, a chain of
// dependent steps), not to bandwidth or tensor throughput.
//
// How. One CTA of four warps per (b, i) head, a straight-line chain without a
// work loop or a ring: thread r owns query row r (TMEM lane r).
//   1. Thread 0 prefetches the head's tiles into L2 while the previous kernel
//      may still run, then (past the grid dependency) issues every TMA load the
//      head may need at once (Q and both key blocks' K and V, before the key
//      length is read), so one DRAM round trip covers them all.
//   2. Thread 0 issues S_j = Q K_j^T (tcgen05, M = 128, N = 128) for every
//      block into TMEM columns [128 j, 128 j + 128).
//   3. The whole row is visible at once, so the softmax takes two passes over
//      the scores instead of a running max: the exact row max first (masked
//      keys at -inf; one compare per score against a per-row limit), then
//      p = 2^(s * scale * log2(e) - m), summed in fp32 and stored to TMEM as
//      bf16 (P_0 over S_0's first 64 columns, P_1 over S_1's).
//   4. Thread 0 issues O = sum_j P_j V_j (TS MMAs, P from TMEM, V from shared
//      memory) into columns [64, 64 + d), i.e. over S_0's second half, which
//      no thread reads any more.
//   5. O / l is packed to bf16. At d = 64 each thread stores its 128-byte row
//      directly; at d = 128 the tile goes into the (no longer needed) Q tile in
//      shared memory, in the 128-byte swizzled layout of the output tensor map,
//      and leaves as one TMA store per 64-column box (rows past n_q clipped by
//      the map).
// TMEM: 128 columns at d = 64 with one key block (up to four CTAs per SM),
// 256 otherwise. Every mbarrier wait is bounded (HATTN_ETIMEOUT on give-up).
// A key length outside [1, n_k] zeroes the head's output and raises
// HATTN_EKEYLEN.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "row_softmax.cuh"

namespace hattn {
namespace {

constexpr int kShortThreads = 128;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column bf16 box

template <int D, int NKB>
struct ShortCfg {
    static_assert((D == 64 && (NKB == 1 || NKB == 2)) || (D == 128 && NKB == 1), "short shapes");
    static constexpr int kBoxes = D / 64;
    static constexpr uint32_t kTileBytes = 128u * D * 2u;
    static constexpr uint32_t kOffQ = 0;  // Q, then the output staging tile
    static constexpr uint32_t kOffK = kOffQ + kTileBytes;
    static constexpr uint32_t kOffV = kOffK + NKB * kTileBytes;
    static constexpr uint32_t kOffBar = kOffV + NKB * kTileBytes;
    // barriers
    static constexpr int kBarQK0 = 0;  // Q and K_0 landed
    static constexpr int kBarK1 = 1;   // K_1 landed
    static constexpr int kBarV0 = 2;
    static constexpr int kBarV1 = 3;
    static constexpr int kBarS = 4;      // every S_j complete
    static constexpr int kBarP = 5;      // P written (one arrival per warp)
    static constexpr int kBarO = 6;      // O complete
    static constexpr int kBarDrain = 7;  // the issued MMAs complete (failure path)
    static constexpr int kNumBars = 8;
    static constexpr uint32_t kOffSlot = kOffBar + 8 * kNumBars;  // TMEM base address
    static constexpr uint32_t kSmemBytes = kOffSlot + 16 + 1024;  // slack to align to 1024 B
    static constexpr uint32_t kTmemCols = (D == 64 && NKB == 1) ? 128u : 256u;
    static constexpr uint32_t kColP1 = 128;  // P_1 over S_1's first half
    static constexpr uint32_t kColO = 64;    // O over S_0's second half
    static_assert(kColO + D <= kTmemCols, "TMEM columns");
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct ShortParams {
    int h, n_q, n_k;
    int mask_kind;
    float scale_log2;
    const int32_t* key_lens;
    float* lse;  // optional [B, h, n_q]
    int* err_word;
    __nv_bfloat16* out;  // [B, n_q, h, D]
};

// Up to three CTAs per SM with one key block at d = 64 (128 TMEM columns each),
// two otherwise (256 columns).
template <int D, int NKB>
__global__ void __launch_bounds__(kShortThreads, (D == 64 && NKB == 1) ? 3 : 2)
    attn_short_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const ShortParams p)
{
    using C = ShortCfg<D, NKB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kOffBar;
    auto bar = [&](int i) { return bar0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffSlot);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, r = threadIdx.x;
    const int b = blockIdx.x / p.h, head = blockIdx.x % p.h;
    const bool leader = threadIdx.x == 0;

    if (leader) {
        mbar_init(bar(C::kBarQK0), 1);
        mbar_init(bar(C::kBarK1), 1);
        mbar_init(bar(C::kBarV0), 1);
        mbar_init(bar(C::kBarV1), 1);
        mbar_init(bar(C::kBarS), 1);
        mbar_init(bar(C::kBarP), 4);
        mbar_init(bar(C::kBarO), 1);
        mbar_init(bar(C::kBarDrain), 1);
        fence_barrier_init();
        prefetch_tmap(&tm_o);
    }
    // 1. Every load goes out first, before the TMEM allocation and the CTA-wide
    // barrier (only this thread uses the barriers it just initialised), and before
    // the key length is known: waiting for it would put a DRAM round trip in front
    // of block 1's loads, and the bandwidth a block past the key length wastes is
    // cheaper than that latency. The inputs may come from the previous kernel
    // (programmatic dependent launch), so the grid dependency is waited for first.
    const bool two_blocks = NKB == 2 && p.n_k > 128;
    // While the previous kernel may still run (programmatic dependent launch), this
    // head's tiles are only prefetched into L2: inputs that are already in memory
    // then arrive from L2 once the dependency is met, and inputs the previous kernel
    // is still writing are simply read again (L2 holds the latest values).
    if (leader) {
        for (int x = 0; x < C::kBoxes; ++x) {
            tma_prefetch_4d(&tm_q, 64 * x, head, 0, b);
            tma_prefetch_4d(&tm_k, 64 * x, head, 0, b);
            tma_prefetch_4d(&tm_v, 64 * x, head, 0, b);
            if (two_blocks) {
                tma_prefetch_4d(&tm_k, 64 * x, head, 128, b);
                tma_prefetch_4d(&tm_v, 64 * x, head, 128, b);
            }
        }
    }
    griddep_wait();
    if (leader) {
        mbar_arrive_expect_tx(bar(C::kBarQK0), 2 * C::kTileBytes);
        for (int x = 0; x < C::kBoxes; ++x) {
            tma_load_4d(sbase + C::kOffQ + x * kBoxBytes, &tm_q, bar(C::kBarQK0), 64 * x, head, 0, b);
            tma_load_4d(sbase + C::kOffK + x * kBoxBytes, &tm_k, bar(C::kBarQK0), 64 * x, head, 0, b);
        }
        if (two_blocks) {
            mbar_arrive_expect_tx(bar(C::kBarK1), C::kTileBytes);
            for (int x = 0; x < C::kBoxes; ++x)
                tma_load_4d(sbase + C::kOffK + C::kTileBytes + x * kBoxBytes, &tm_k, bar(C::kBarK1),
                            64 * x, head, 128, b);
        }
        mbar_arrive_expect_tx(bar(C::kBarV0), C::kTileBytes);
        for (int x = 0; x < C::kBoxes; ++x)
            tma_load_4d(sbase + C::kOffV + x * kBoxBytes, &tm_v, bar(C::kBarV0), 64 * x, head, 0, b);
        if (two_blocks) {
            mbar_arrive_expect_tx(bar(C::kBarV1), C::kTileBytes);
            for (int x = 0; x < C::kBoxes; ++x)
                tma_load_4d(sbase + C::kOffV + C::kTileBytes + x * kBoxBytes, &tm_v, bar(C::kBarV1),
                            64 * x, head, 128, b);
        }
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_launch_dependents();
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;
    const int kv_len = (p.mask_kind & HATTN_MASK_KEY_PADDING) ? p.key_lens[b] : p.n_k;
    const bool valid = kv_len >= 1 && kv_len <= p.n_k;
    const int nblk = valid ? (NKB == 2 && kv_len > 128 ? 2 : 1) : 0;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);

    // 2. S_j for every block that holds valid keys.
    bool ctl_ok = true;
    if (leader) {
        if (nblk > 0) {
            const uint64_t q_desc = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
            for (int j = 0; j < nblk && ctl_ok; ++j) {
                ctl_ok = mbar_wait(bar(j == 0 ? C::kBarQK0 : C::kBarK1), 0);
                if (!ctl_ok) break;
                tc_fence_after();
                const uint64_t k_desc = sdesc_sw128(sbase + C::kOffK + j * C::kTileBytes, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t off = ((ks / 4) * kBoxBytes + (ks % 4) * 32) >> 4;
                    mma_ss(tmem + 128u * j, q_desc + off, k_desc + off, C::kIdescS, ks > 0 ? 1u : 0u);
                }
            }
            if (ctl_ok) mma_commit(bar(C::kBarS));
        }
    }
    __syncwarp();

    // 3. Softmax over the whole row: exact max, then the exponentials.
    float m = -INFINITY, l = 0.0f;
    bool ok = ctl_ok;
    if (nblk > 0) {
        const bool got = mbar_wait(bar(C::kBarS), 0);
        ok = __all_sync(0xffffffffu, got);
        if (ok) {
            tc_fence_after();
            // Key j is visible iff j < lim: inside the key length and, when causal,
            // not after this row (top-left aligned; causal implies n_q == n_k <= 128).
            const int lim = min(kv_len, causal ? r + 1 : kv_len);
            const uint64_t c2 = f32x2(p.scale_log2, p.scale_log2);
            uint64_t acc[4] = {0, 0, 0, 0};
            uint32_t sr[128];
            tmem_ld_x128(lane_base, sr);
#pragma unroll
            for (int i = 0; i < 128; ++i)
                if (i >= lim) sr[i] = __float_as_uint(-INFINITY);
            float mx = row_max(sr);
            if (NKB == 2 && nblk == 2) {
                // Block 1 stays in registers: its max, then its exponentials; block 0
                // is read again for its own (its columns are not written before).
                tmem_ld_x128(lane_base + 128, sr);
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i + 128 >= lim) sr[i] = __float_as_uint(-INFINITY);
                mx = fmaxf(mx, row_max(sr));
                m = mx * p.scale_log2;
                exp_block<false>(sr, c2, f32x2(-m, -m), acc, lane_base + C::kColP1);
                tmem_ld_x128(lane_base, sr);
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= lim) sr[i] = __float_as_uint(-INFINITY);
            } else {
                m = mx * p.scale_log2;
            }
            exp_block<false>(sr, c2, f32x2(-m, -m), acc, lane_base);
            float a0, a1;
            f32x2_split(add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3])), a0, a1);
            l = a0 + a1;
            tmem_st_wait();
            tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarP));
    }

    // 4. O = sum_j P_j V_j.
    if (leader && nblk > 0 && ctl_ok) {
        ctl_ok = mbar_wait(bar(C::kBarP), 0) && mbar_wait(bar(C::kBarV0), 0) &&
                 (nblk < 2 || mbar_wait(bar(C::kBarV1), 0));
        if (ctl_ok) {
            tc_fence_after();
            for (int j = 0; j < nblk; ++j) {
                const uint64_t v_desc =
                    sdesc_sw128(sbase + C::kOffV + j * C::kTileBytes, kBoxBytes, 1024);
                const uint32_t p_tmem = tmem + (j == 0 ? 0u : C::kColP1);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ts(tmem + C::kColO, p_tmem + ks * 8, v_desc + ((ks * 2048) >> 4), C::kIdescPV,
                           (j > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(bar(C::kBarO));
        }
    }
    __syncwarp();
    if (nblk > 0 && ok) {
        const bool got = mbar_wait(bar(C::kBarO), 0);
        ok = __all_sync(0xffffffffu, got);
    }
    if (leader) {
        // Every copy this CTA started has landed (they normally have) before the Q
        // tile is overwritten or the CTA exits; every MMA it issued has completed.
        mbar_wait(bar(C::kBarQK0), 0);
        mbar_wait(bar(C::kBarV0), 0);
        if (two_blocks) {
            mbar_wait(bar(C::kBarK1), 0);
            mbar_wait(bar(C::kBarV1), 0);
        }
        mma_commit(bar(C::kBarDrain));
        mbar_wait(bar(C::kBarDrain), 0);
        if (!valid) raise_device_error(p.err_word, HATTN_EKEYLEN);
        if (!ctl_ok) raise_device_error(p.err_word, HATTN_ETIMEOUT);
    }
    if (nblk > 0 && !ok && lane == 0) raise_device_error(p.err_word, HATTN_ETIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // 5. O / l (zeros for an invalid key length). At D = 64 each thread stores its
    // own 128-byte output row with 16-byte global stores (whole sectors, nothing to
    // wait for before the CTA exits): measured 4 % faster on the decoder workload
    // than the staged TMA store. At D = 128 (256-byte rows) the staged tile and one
    // TMA store per box measured 3.5 % faster, so it keeps them.
    constexpr bool kDirect = D == 64;
    const bool have = nblk > 0 && ok;
    const float inv = have ? 1.0f / l : 0.0f;
    uint8_t* yrow = smem + C::kOffQ + r * 128;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        if (have) {
            tmem_ld_x32(lane_base + C::kColO + 32 * q, o);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if constexpr (kDirect) {
            if (r < p.n_q) {
                __nv_bfloat16* orow = p.out + (((size_t)b * p.n_q + r) * p.h + head) * D;
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    st_global_v4(orow + 32 * q + 8 * v4,
                                 pack_bf16x2(__uint_as_float(o[8 * v4]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv),
                                 pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv),
                                 pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv),
                                 pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv));
            }
        } else {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
                const int kc = (q % 2) * 4 + v4;  // 16-byte chunk within the box row
                *reinterpret_cast<uint4*>(yrow + (q / 2) * kBoxBytes + ((kc ^ (r & 7)) * 16)) =
                    make_uint4(pack_bf16x2(__uint_as_float(o[8 * v4]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv),
                               pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv),
                               pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv),
                               pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv));
            }
        }
    }
    // Natural-log log-sum-exp of the scaled scores: the exponentials ran in base 2
    // on s * scale * log2(e) with the row max m, so ln sum = (m + log2 l) ln 2.
    if (p.lse && r < p.n_q)
        p.lse[((size_t)b * p.h + head) * p.n_q + r] =
            have ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    if constexpr (!kDirect) fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (!kDirect && leader) {
        for (int x = 0; x < C::kBoxes; ++x)
            tma_store_4d(&tm_o, sbase + C::kOffQ + x * kBoxBytes, 64 * x, head, 0, b);
        bulk_commit_group();
        bulk_wait_group_read_all();  // the tile is read out before shared memory is released
    }
    __syncwarp();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, int NKB>
cudaError_t launch_short(const AttnArgs& a, const AttnMaps& m)
{
    using C = ShortCfg<D, NKB>;
    const long long grid = (long long)a.B * a.h;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(attn_short_kernel<D, NKB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    ShortParams p;
    p.h = a.h;
    p.n_q = a.n_q;
    p.n_k = a.n_k;
    p.mask_kind = a.mask_kind;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.key_lens = a.key_lens;
    p.lse = a.lse;
    p.err_word = a.err_word;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kShortThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_short_kernel<D, NKB>, m.q, m.k, m.v, m.o, p);
}

}  // namespace

// The short kernel runs every head from scratch; the persistent kernel overlaps one
// head's loads with another's compute, which pays once each SM has many heads to
// run. Measured on GB300 (back-to-back steps, inputs from HBM): with one key block
// one CTA per head was 12-20 % faster at 256, 1024 and 2048 heads (13.5 per SM);
// with two it was even at 512 heads and 19 % slower at 1024 (6.7 per SM).
bool attn_short_supported(const AttnArgs& a)
{
    if (!attn_tc_supported(a) || a.n_q > 128) return false;
    const bool one_block = a.n_k <= 128;
    if (!(one_block || (a.d_k == 64 && a.n_k <= 256))) return false;
    const long long heads = (long long)a.B * a.h;
    return heads <= (long long)sm_count() * (one_block ? 16 : 3);
}

cudaError_t launch_attn_short(const AttnArgs& a, const AttnMaps& maps)
{
    if (a.d_k == 128) return launch_short<128, 1>(a, maps);
    return a.n_k <= 128 ? launch_short<64, 1>(a, maps) : launch_short<64, 2>(a, maps);
}

}  // namespace hattn
