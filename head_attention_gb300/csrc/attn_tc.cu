// Tensor-core attention forward for sm_103a (bf16 in/out, fp32 accumulation,
// d_k == d_v == D in {64, 128}).
//
// What it computes: for every (batch b, head i, query t)
//     out[b,t,i,:] = sum_j softmax_j(scale * q.k_j) v_j     (visible keys j only)
// — the scaled dot-product attention of the explanatory pages on "Attention
// Is All You Need" (hex4c59 §把所有位置合并，就是那条核心公式; masks per
// §掩码必须在 softmax 之前生效).
//
// How (one CTA = one (b, i) and 256 consecutive query rows = two 128-row tiles):
//   warp 8      TMA producer: loads the two Q tiles once, then streams K_j and
//               V_j (128 keys each) through a ring of shared-memory stages.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, and
//               O_t += P_t V_j with P_t read from TMEM; completion is reported
//               through tcgen05.commit onto mbarriers.
//   warps 0-3   softmax of tile 0, warps 4-7 softmax of tile 1: thread r owns
//               query row r (TMEM lane r), so the row max and row sum are
//               thread-local. Streaming softmax in base 2: running max m, sum l,
//               p = 2^(s*scale*log2e - m), P written back to TMEM as bf16 over
//               the first half of S's columns. O is rescaled only when the
//               max grows by more than 2^8 (the final 1/l uses the same stale
//               max, so the result is unchanged; p stays <= 2^8).
//   The issue order S_0(j), S_1(j), then per tile PV_t(j) followed at once by
//   S_t(j+1) lets one tile's softmax overlap the other tile's MMAs.
//   Causal: key blocks above the diagonal are never loaded or multiplied; only
//   the diagonal block is masked element-wise. Key padding: blocks at or past
//   key_lens[b] are skipped; the last block is masked column-wise.
//   Epilogue: O / l packed to bf16, 16-byte stores into [B, n_q, h, D].
//
// TMEM columns: tile t holds S at [256t, 256t+128) and O at [256t+128, 256t+128+D).
// Every mbarrier wait is bounded; on a timeout the CTA records HATTN_ETIMEOUT in
// the device error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 320;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kRowsPerCta = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column bf16 box

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    // barrier indices
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kStages;
    static constexpr int kBarVFull = kBarKEmpty + kStages;
    static constexpr int kBarVEmpty = kBarVFull + kStages;
    static constexpr int kBarS = kBarVEmpty + kStages;  // 2
    static constexpr int kBarP = kBarS + 2;             // 2
    static constexpr int kBarO = kBarP + 2;             // 2
    static constexpr int kBarDrain = kBarO + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffSlot = kOffBar + 8 * kNumBars;  // TMEM base address + abort flag
    static constexpr int kSmemUsed = kOffSlot + 16;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct TcParams {
    int B, h, n_q, n_k;
    int mask_kind;
    float scale_log2;
    int n_pairs;
    const int32_t* key_lens;
    __nv_bfloat16* out;
    int* err_word;
};

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem)
{
    using C = Cfg<D>;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        // 16-element K step: box (ks / 4), 32-byte offset inside the swizzled 128-byte row.
        const uint32_t off = (ks / 4) * kBoxBytes + (ks % 4) * 32;
        mma_ss(d_tmem, sdesc_sw128(q_smem + off, 16, 1024), sdesc_sw128(k_smem + off, 16, 1024),
               C::kIdescS, ks > 0 ? 1u : 0u);
    }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate)
{
    using C = Cfg<D>;
#pragma unroll
    for (int ks = 0; ks < 128 / 16; ++ks) {
        // 16 keys = 16 rows of the V tile (2 swizzle atoms of 8 rows); P columns hold bf16 pairs.
        mma_ts(d_tmem, p_tmem + ks * 8, sdesc_sw128(v_smem + ks * 2048, kBoxBytes, 1024),
               C::kIdescPV, (accumulate || ks > 0) ? 1u : 0u);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const TcParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffSlot + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;

    // ---- work unit: heaviest causal rows first
    const int bh_count = p.B * p.h;
    int pair = blockIdx.x / bh_count;
    const int bh = blockIdx.x % bh_count;
    if (causal) pair = p.n_pairs - 1 - pair;
    const int b = bh / p.h, head = bh % p.h;
    const int row0_0 = pair * kRowsPerCta, row0_1 = row0_0 + 128;

    int kv_len = p.n_k;
    if (p.mask_kind & HATTN_MASK_KEY_PADDING) kv_len = p.key_lens[b];
    if (kv_len < 1 || kv_len > p.n_k) {
        if (threadIdx.x < 256) {
            const int row = (threadIdx.x < 128 ? row0_0 : row0_1) + threadIdx.x % 128;
            if (row < p.n_q) {
                __nv_bfloat16* orow = p.out + (((size_t)b * p.n_q + row) * p.h + head) * D;
                for (int c = 0; c < D; c += 8) st_global_v4(orow + c, 0u, 0u, 0u, 0u);
            }
        }
        if (threadIdx.x == 0) raise_device_error(p.err_word, HATTN_EKEYLEN);
        return;
    }
    const int kv_blocks = (kv_len + 127) / 128;
    auto blocks_for = [&](int r0) {
        if (r0 >= p.n_q) return 0;
        return causal ? min(kv_blocks, r0 / 128 + 1) : kv_blocks;
    };
    const int nblk_0 = blocks_for(row0_0), nblk_1 = blocks_for(row0_1);
    const int nblk_max = max(nblk_0, nblk_1);

    // ---- setup
    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarQ), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKEmpty + s), 1);
            mbar_init(bar(C::kBarVFull + s), 1);
            mbar_init(bar(C::kBarVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::kBarS + t), 1);
            mbar_init(bar(C::kBarP + t), 128);
            mbar_init(bar(C::kBarO + t), 1);
        }
        mbar_init(bar(C::kBarDrain), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto give_up = [&]() {
        *abort_flag = 1;
        raise_device_error(p.err_word, HATTN_ETIMEOUT);
    };

    if (warp == kWarpLoad) {
        // ================================================================ TMA producer
        if (lane == 0) {
            const int n_tiles = nblk_1 > 0 ? 2 : 1;
            mbar_arrive_expect_tx(bar(C::kBarQ), n_tiles * C::kTileBytes);
            for (int t = 0; t < n_tiles; ++t)
                for (int x = 0; x < C::kBoxes; ++x)
                    tma_load_4d(sbase + C::kOffQ + t * C::kTileBytes + x * kBoxBytes, &tm_q,
                                bar(C::kBarQ), x * 64, head, t ? row0_1 : row0_0, b);
            int k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int j = 0; j < nblk_max; ++j) {
                const int s = j % C::kStages;
                const uint32_t ph = (j / C::kStages) & 1;
                if (*abort_flag || !mbar_wait(bar(C::kBarKEmpty + s), ph ^ 1)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(C::kBarKFull + s), C::kTileBytes);
                for (int x = 0; x < C::kBoxes; ++x)
                    tma_load_4d(sbase + C::kOffK + s * C::kTileBytes + x * kBoxBytes, &tm_k,
                                bar(C::kBarKFull + s), x * 64, head, j * 128, b);
                ++k_issued;
                if (*abort_flag || !mbar_wait(bar(C::kBarVEmpty + s), ph ^ 1)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(C::kBarVFull + s), C::kTileBytes);
                for (int x = 0; x < C::kBoxes; ++x)
                    tma_load_4d(sbase + C::kOffV + s * C::kTileBytes + x * kBoxBytes, &tm_v,
                                bar(C::kBarVFull + s), x * 64, head, j * 128, b);
                ++v_issued;
            }
            if (!ok) give_up();
            // Every copy this CTA started must land before the CTA may exit.
            mbar_wait(bar(C::kBarQ), 0);
            for (int j = max(0, k_issued - C::kStages); j < k_issued; ++j)
                mbar_wait(bar(C::kBarKFull + j % C::kStages), (j / C::kStages) & 1);
            for (int j = max(0, v_issued - C::kStages); j < v_issued; ++j)
                mbar_wait(bar(C::kBarVFull + j % C::kStages), (j / C::kStages) & 1);
        }
    } else if (warp == kWarpMma) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t sQ0 = sbase + C::kOffQ, sQ1 = sQ0 + C::kTileBytes;
            auto sK = [&](int s) { return sbase + C::kOffK + s * C::kTileBytes; };
            auto sV = [&](int s) { return sbase + C::kOffV + s * C::kTileBytes; };
            bool ok = mbar_wait(bar(C::kBarQ), 0) && mbar_wait(bar(C::kBarKFull), 0);
            if (ok) {
                tc_fence_after();
                if (nblk_0 > 0) {
                    issue_qk<D>(tmem, sQ0, sK(0));
                    mma_commit(bar(C::kBarS));
                }
                if (nblk_1 > 0) {
                    issue_qk<D>(tmem + 256, sQ1, sK(0));
                    mma_commit(bar(C::kBarS + 1));
                }
                mma_commit(bar(C::kBarKEmpty));
            }
            // PV of tile t for block j, then at once S of tile t for block j + 1.
            auto tile_step = [&](int t, int nb, uint32_t sQ, int j, int s, int s1) -> bool {
                if (j >= nb) return true;
                if (*abort_flag || !mbar_wait(bar(C::kBarP + t), j & 1)) return false;
                tc_fence_after();
                issue_pv<D>(tmem + 256 * t + 128, tmem + 256 * t, sV(s), j > 0);
                if (j == nb - 1) mma_commit(bar(C::kBarO + t));
                if (j + 1 < nb) {
                    issue_qk<D>(tmem + 256 * t, sQ, sK(s1));
                    mma_commit(bar(C::kBarS + t));
                }
                return true;
            };
            for (int j = 0; ok && j < nblk_max; ++j) {
                const int s = j % C::kStages, s1 = (j + 1) % C::kStages;
                const uint32_t ph = (j / C::kStages) & 1, ph1 = ((j + 1) / C::kStages) & 1;
                const bool next = j + 1 < nblk_max;
                if (!mbar_wait(bar(C::kBarVFull + s), ph)) { ok = false; break; }
                if (next && !mbar_wait(bar(C::kBarKFull + s1), ph1)) { ok = false; break; }
                tc_fence_after();
                if (!tile_step(0, nblk_0, sQ0, j, s, s1) || !tile_step(1, nblk_1, sQ1, j, s, s1)) {
                    ok = false;
                    break;
                }
                mma_commit(bar(C::kBarVEmpty + s));
                if (next) mma_commit(bar(C::kBarKEmpty + s1));
            }
            if (!ok) give_up();
            // All issued MMAs must complete before TMEM is released.
            mma_commit(bar(C::kBarDrain));
            mbar_wait(bar(C::kBarDrain), 0);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax + epilogue
        const int t = warp / 4;
        const int wq = warp % 4;
        const int r = wq * 32 + lane;
        const int my_row0 = t ? row0_1 : row0_0;
        const int row = my_row0 + r;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t cS = 256u * t, cO = 256u * t + 128u;
        const int nb = t ? nblk_1 : nblk_0;
        float m_used = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            bool got = mbar_wait(bar(C::kBarS + t), j & 1);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc_fence_after();
            float x[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t raw[32];
                tmem_ld_x32(lane_base + cS + 32 * c, raw);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(raw[i]) * p.scale_log2;
            }
            const int kbase = j * 128;
            const bool need_mask = (kbase + 128 > kv_len) || (causal && kbase + 127 > my_row0);
            if (need_mask) {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    const int kj = kbase + i;
                    const bool visible = (kj < kv_len) && !(causal && kj > row);
                    if (!visible) x[i] = -INFINITY;
                }
            }
            float mx = x[0];
#pragma unroll
            for (int i = 1; i < 128; ++i) mx = fmaxf(mx, x[i]);
            const float m_new = fmaxf(m_used, mx);
            const bool grow = m_new > m_used + kRescaleLog2;
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t o[16];
                    tmem_ld_x16(lane_base + cO + 16 * c, o);
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_x16(lane_base + cO + 16 * c, o);
                }
                l *= alpha;
            }
            if (grow) m_used = m_new;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ex2_approx(x[32 * c + 2 * i] - m_used);
                    const float p1 = ex2_approx(x[32 * c + 2 * i + 1] - m_used);
                    l += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st_x16(lane_base + cS + 16 * c, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(C::kBarP + t));
        }
        if (nb > 0 && ok) {
            bool got = mbar_wait(bar(C::kBarO + t), 0);
            ok = __all_sync(0xffffffffu, got);
        }
        if (!ok) {
            give_up();
        } else if (nb > 0) {
            tc_fence_after();
            const float inv = 1.0f / l;
            __nv_bfloat16* orow = p.out + (((size_t)b * p.n_q + row) * p.h + head) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + cO + 32 * c, o);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv,
                                        __uint_as_float(o[2 * i + 1]) * inv);
                if (row < p.n_q) {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        st_global_v4(orow + 32 * c + 8 * v4, pk[4 * v4], pk[4 * v4 + 1],
                                     pk[4 * v4 + 2], pk[4 * v4 + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const AttnMaps& m)
{
    using C = Cfg<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    TcParams p;
    p.B = a.B;
    p.h = a.h;
    p.n_q = a.n_q;
    p.n_k = a.n_k;
    p.mask_kind = a.mask_kind;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.n_pairs = (a.n_q + kRowsPerCta - 1) / kRowsPerCta;
    p.key_lens = a.key_lens;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.err_word = a.err_word;
    const long long units = (long long)p.n_pairs * a.B * a.h;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    attn_tc_kernel<D><<<dim3((unsigned)units), kThreads, C::kSmemBytes, a.stream>>>(m.q, m.k, m.v, p);
    return cudaGetLastError();
}

}  // namespace

bool attn_tc_supported(const AttnArgs& a)
{
    return a.dtype == HATTN_BF16 && a.d_k == a.d_v && (a.d_k == 64 || a.d_k == 128);
}

cudaError_t launch_attn_tc(const AttnArgs& a, const AttnMaps& maps)
{
    return a.d_k == 64 ? launch_d<64>(a, maps) : launch_d<128>(a, maps);
}

}  // namespace hattn
