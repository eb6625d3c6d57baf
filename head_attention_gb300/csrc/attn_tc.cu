// Tensor-core attention forward for sm_103a (bf16 in/out, fp32 accumulation,
// d_k == d_v == D in {64, 128}, scale > 0).
//
// What it computes: for every (batch b, head i, query t)
//     out[b,t,i,:] = sum_j softmax_j(scale * q.k_j) v_j     (visible keys j only)
// — the scaled dot-product attention of the explanatory pages on "Attention
// Is All You Need" (hex4c59 §把所有位置合并，就是那条核心公式; masks per
// §掩码必须在 softmax 之前生效).
//
// How. A persistent kernel: one CTA per SM loops over work units, a unit being
// one (b, i) and 256 consecutive query rows = two 128-row tiles (when n_q <= 128,
// two (b, i) heads instead, one per tile, each with its own K/V stream). Units are
// ordered in groups of heads whose K/V take at most a quarter of L2 together,
// heaviest causal rows first within a group; for causal problems the host assigns units to
// CTAs by greedy list scheduling on their block counts (a table passed with
// the launch), otherwise CTAs take them in a snake order. All barrier phases
// run on across units, so a CTA pays its set-up once, the next unit's Q tile
// is loaded as soon as the previous unit's last S MMA of that tile retired,
// and a tile's epilogue overlaps its first S MMA of the next unit.
// 12 warps in three warpgroups; a register split gives the softmax warps 208
// registers and the control warps 72. The control warps come first: the warp
// schedulers favour lower-numbered warps among the ready ones, and an MMA
// issuer that waits behind a busy softmax warp for issue slots delays the
// tensor pipe (measured: 7% at D=64, 3% at D=128).
//   warp 0      TMA: the unit's Q tiles, then K_j (128 keys) through a
//               3-stage (D=128) / 7-stage (D=64) shared-memory ring.
//   warp 2      TMA: V_j through a 2-stage (D=128) / 5-stage (D=64) ring. K
//               runs one block ahead of V because S(j+1) precedes PV(j) (D=64)
//               or follows it at once (D=128).
//   warps 1, 3  MMA issuers, one thread per tile: S_t = Q_t K_j^T into TMEM,
//               then per block PV_t(j) (O_t += P_t V_j, P_t read from TMEM)
//               and S_t(j+1). Completion is reported by tcgen05.commit onto
//               mbarriers. With one issuer per tile, a tile whose P is ready
//               never waits behind the other tile's MMA issue, and one tile's
//               softmax overlaps the other tile's MMAs. Nothing but the MMAs
//               sits between P(j) and S(j+1) (D = 128): K(j+1) is waited for
//               before P(j), and the commits that release buffers follow S(j+1).
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1; at D = 128
//               they take turns on the exponentials (two named barriers), so
//               that the MUFU work of one tile overlaps the MMAs of the other
//               (at D = 64 they run freely). Thread r owns
//               query row r (TMEM lane r), so the row max and row sum are
//               thread-local. Streaming softmax in base 2: running max m and
//               sum l, p = 2^(s*scale*log2e - m), P stored back to TMEM as bf16.
//               The exponentials of a block use the running max while the
//               block's own max is computed alongside; O is rescaled (and the
//               block redone) only when a row's max grows by more than 2^8. The
//               final 1/l uses the same max as the numerator, so the result is
//               unchanged; p <= 2^8.
//   Causal: key blocks above the diagonal are never loaded or multiplied; only
//   the diagonal block is masked element-wise. Key padding: blocks at or past
//   key_lens[b] are skipped and the last block is masked column-wise.
//   Epilogue (softmax warps): O / l packed to bf16, 16-byte stores into
//   [B, n_q, h, D].
//
// TMEM columns (tile t owns [256t, 256t+256)): D = 128: S at +0, P over S's
// first 64 columns, O at +128; S(j+1) then waits for PV(j). D = 64: S at +0,
// P at +128, O at +192; S(j+1) is computed as soon as the softmax has read
// S(j) out, while block j's exponentials run.
// Every mbarrier wait is bounded; on a timeout the CTA records HATTN_ETIMEOUT in
// the device error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <queue>
#include <type_traits>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"
#include "row_softmax.cuh"

namespace hattn {
namespace {

constexpr int kThreads = 384;
constexpr int kWarpLoadK = 0;
constexpr int kWarpMma0 = 1;   // MMA issuer of tile 0 (also owns the TMEM allocation)
constexpr int kWarpLoadV = 2;
constexpr int kWarpMma1 = 3;   // MMA issuer of tile 1
constexpr int kWarpSoftmax0 = 4;  // warps 4-7 softmax of tile 0, 8-11 of tile 1
// Launched at 168 registers per thread (384 x 168 = 64512 of the SM's 65536).
constexpr int kRegsSoftmax = 208;
constexpr int kRegsControl = 72;
static_assert(256 * kRegsSoftmax + 128 * kRegsControl <= kThreads * 168, "register split");

// Named barriers that make the two softmax warpgroups take turns on the
// exponentials (barrier 0 is __syncthreads): tile 0 waits on kTurn0, tile 1 on kTurn1.
constexpr uint32_t kTurn0 = 1, kTurn1 = 2;

constexpr int kRowsPerCta = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column bf16 box

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kKStages = (D == 128) ? 3 : 7;
    static constexpr int kVStages = (D == 128) ? 2 : 5;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    // barrier indices
    static constexpr int kBarQFull = 0;   // 2: Q_t landed
    static constexpr int kBarQEmpty = 2;  // 2: the unit's last S MMA of tile t retired
    static constexpr int kBarKFull = 4;
    static constexpr int kBarKEmpty = kBarKFull + kKStages;
    static constexpr int kBarVFull = kBarKEmpty + kKStages;
    static constexpr int kBarVEmpty = kBarVFull + kVStages;
    static constexpr int kBarS = kBarVEmpty + kVStages;  // 2: S_t ready
    static constexpr int kBarP = kBarS + 2;              // 2: P_t written (one arrival per warp)
    static constexpr int kBarO = kBarP + 2;              // 2: final O_t ready
    static constexpr int kBarDrain = kBarO + 2;  // 2: one per issuer
    // Separate P columns only: S_t read out of TMEM (one arrival per warp), and
    // PV_t(j) retired for a block that is not the tile's last.
    static constexpr int kBarSFree = kBarDrain + 2;
    static constexpr int kBarPVDone = kBarSFree + 2;
    static constexpr int kNumBars = kBarPVDone + 2;
    // TMEM columns inside a tile's 256. With D = 64 P gets columns of its own
    // (S 128 + P 64 + O 64), so S(j+1) can be computed while block j's
    // exponentials run; with D = 128 P is written over the first half of S.
    static constexpr bool kSepP = (D == 64);
    static constexpr uint32_t kColP = kSepP ? 128u : 0u;
    static constexpr uint32_t kColO = kSepP ? 192u : 128u;
    static_assert(kColO + D <= 256, "TMEM columns of a tile");
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
    int n_pairs;      // 256-row query pairs per (b, i)
    int units;        // B * h * n_pairs
    int group_heads;  // heads per L2 group in the unit order
    int issuers;      // 2 when any unit has a second tile, else 1
    const int32_t* key_lens;
    __nv_bfloat16* out;
    float* lse;  // optional [B, h, n_q]
    int* err_word;
};

// Units of every CTA, computed on the host (greedy list scheduling on the
// units' block counts) and passed by value with the launch: CTA c takes the
// unit slots list[first[c] .. first[c + 1]) in that (ascending) order.
constexpr int kTableUnits = 4096;
constexpr int kTableCtas = 256;
struct SchedTable {
    uint16_t first[kTableCtas + 1];
    uint16_t list[kTableUnits];
};
struct SchedSnake {};
// Query rows that fit one tile (n_q <= 128): a unit's two tiles take two (b, i)
// heads, units in snake order. A type of its own, so that the other launches
// compile without the paired bookkeeping.
struct SchedPaired {};
template <class Sched>
constexpr bool kPaired = std::is_same<Sched, SchedPaired>::value;

// Whether the two tiles' softmax warpgroups take turns on the exponentials, so
// that one tile's exponentials overlap the other tile's MMAs. Measured on GB300:
// at D = 128 the turns are worth 16 % on the long causal workload. At D = 64 (P in
// columns of its own, MMAs half as long) they cost 5.5 % on the long causal
// workload (table schedule) and gain 2 % on the MHA sublayer (n = 512, snake
// order) and on cross-attention (paired heads).
template <int D, class Sched>
constexpr bool kPingPong = D == 128 || !std::is_same<Sched, SchedTable>::value;

// Per-CTA state shared by the role functions; the unit fields are rewritten
// by unit_setup for every unit.
struct Cta {
    uint32_t sbase;       // shared-memory base (1024-aligned)
    uint32_t bar0;        // address of barrier 0
    uint32_t tmem;        // TMEM base address
    uint32_t abort_flag;  // shared address of the word set when any wait gave up
    bool causal;
    // Per tile: the (b, i) head, its first query row, its key blocks (0: tile
    // absent), its key length and whether that is within [1, n_k]. Both tiles
    // share one head except in paired units.
    int b[2], head[2];
    int row0[2];
    int nblk[2];
    int nblk_max;
    int kv_len[2];
    bool valid[2];
    __device__ uint32_t bar(int i) const { return bar0 + 8u * i; }
    __device__ bool aborted() const { return ld_volatile_shared(abort_flag) != 0u; }
};

// Walks this CTA's unit slots in increasing order.
template <bool kTable>
struct UnitIter {
    int pos = -1, end = 0;
    template <class Sched>
    __device__ __forceinline__ int next(const TcParams& p, const Sched& sch)
    {
        if constexpr (kTable) {
            if (pos < 0) {
                pos = sch.first[blockIdx.x];
                end = sch.first[blockIdx.x + 1];
            }
            return pos < end ? static_cast<int>(sch.list[pos++]) : -1;
        } else {
            if (pos < 0) pos = 0;
            // Snake: round r takes slots [r * grid, (r + 1) * grid), reversed on odd rounds.
            const long long r = pos++;
            const long long slot = r * gridDim.x + ((r & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
            return slot < p.units ? static_cast<int>(slot) : -1;
        }
    }
};

// Unit order: groups of group_heads (b, i) heads; within a group, query pairs
// from the heaviest (causal: the last rows) down, heads inner.
// The per-unit fields of Cta, decoded from a unit slot.
struct UnitInfo {
    int b[2], head[2], row0[2], nblk[2], kv_len[2];
    bool valid[2];
};

template <bool kPairedUnit>
__device__ __forceinline__ UnitInfo unit_decode(const TcParams& p, bool causal, int slot)
{
    UnitInfo u;
    if constexpr (kPairedUnit) {
        // Tile t takes head 2 slot + t (absent past the last head), all its n_q <= 128
        // query rows in one tile.
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int bh = 2 * slot + t;
            const bool present = bh < p.B * p.h;
            u.b[t] = present ? bh / p.h : 0;
            u.head[t] = present ? bh % p.h : 0;
            u.row0[t] = 0;
            u.kv_len[t] = (p.mask_kind & HATTN_MASK_KEY_PADDING) ? p.key_lens[u.b[t]] : p.n_k;
            u.valid[t] = !present || (u.kv_len[t] >= 1 && u.kv_len[t] <= p.n_k);
            const int kv_blocks = (u.kv_len[t] + 127) / 128;
            u.nblk[t] = (present && u.valid[t]) ? (causal ? min(kv_blocks, 1) : kv_blocks) : 0;
        }
        return u;
    }
    const int per_group = p.group_heads * p.n_pairs;
    const int g = slot / per_group;
    const int w = slot - g * per_group;
    const int heads_here = min(p.group_heads, p.B * p.h - g * p.group_heads);
    const int pi = w / heads_here;
    const int bh = g * p.group_heads + (w - pi * heads_here);
    const int pair = causal ? p.n_pairs - 1 - pi : pi;
    const int b = bh / p.h, head = bh % p.h;
    const int kv_len = (p.mask_kind & HATTN_MASK_KEY_PADDING) ? p.key_lens[b] : p.n_k;
    const bool valid = kv_len >= 1 && kv_len <= p.n_k;
    const int kv_blocks = (kv_len + 127) / 128;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        u.b[t] = b;
        u.head[t] = head;
        u.row0[t] = pair * kRowsPerCta + 128 * t;
        u.kv_len[t] = kv_len;
        u.valid[t] = valid;
        if (!valid || u.row0[t] >= p.n_q) u.nblk[t] = 0;
        else u.nblk[t] = causal ? min(kv_blocks, u.row0[t] / 128 + 1) : kv_blocks;
    }
    return u;
}

__device__ __forceinline__ void unit_apply(Cta& c, const UnitInfo& u)
{
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        c.b[t] = u.b[t];
        c.head[t] = u.head[t];
        c.row0[t] = u.row0[t];
        c.kv_len[t] = u.kv_len[t];
        c.valid[t] = u.valid[t];
        c.nblk[t] = u.nblk[t];
    }
    c.nblk_max = max(u.nblk[0], u.nblk[1]);
}

template <class Sched>
__device__ __forceinline__ void unit_setup(Cta& c, const TcParams& p, int slot)
{
    unit_apply(c, unit_decode<kPaired<Sched>>(p, c.causal, slot));
}

// The unit slots of this CTA with the next one decoded ahead: a role calls
// prefetch() where it waits anyway (so the integer divisions, the key-length
// load and the rarely run code behind them leave its critical path) and
// advance() at its unit boundary. A role keeps only its View of a unit (the
// fewest live registers). Measured on the cross-attention workload, decoding
// at the boundary kept the MMA issuer ~1.5k cycles per unit from its next S MMA.
template <bool kTable, class View>
struct Ahead {
    UnitIter<kTable> it;
    int slot = -2;  // -2: the next slot is not fetched yet; -1: no more units
    View info;
    template <class Sched>
    __device__ __forceinline__ void prefetch(const TcParams& p, const Sched& sch, bool causal, int t)
    {
        if (slot != -2) return;
        slot = it.next(p, sch);
        if (slot >= 0) info = View::of(unit_decode<kPaired<Sched>>(p, causal, slot), t);
    }
    template <class Sched>
    __device__ __forceinline__ bool advance(View& v, const TcParams& p, const Sched& sch, bool causal, int t)
    {
        prefetch(p, sch, causal, t);
        if (slot < 0) return false;
        v = info;
        slot = -2;
        return true;
    }
};

// The MMA issuer's view: the key blocks of both tiles.
struct BlockCounts {
    int n0, n1;
    __device__ __forceinline__ static BlockCounts of(const UnitInfo& u, int) { return {u.nblk[0], u.nblk[1]}; }
};

__device__ __forceinline__ void give_up(const Cta& c, int* err_word)
{
    st_volatile_shared(c.abort_flag, 1u);
    raise_device_error(err_word, HATTN_ETIMEOUT);
}

// The MMA issue loops run on warps that share their SM sub-partition with busy
// softmax warps, so each MMA costs as few instructions as possible: shared-memory
// descriptors are built once per operand tile and stepped by adding the K-step
// offset (in 16-byte units) to the start-address field.

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc)
{
    using C = Cfg<D>;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        // 16-element K step: box (ks / 4), 32-byte offset inside the swizzled 128-byte row.
        const uint64_t off = ((ks / 4) * kBoxBytes + (ks % 4) * 32) >> 4;
        mma_ss(d_tmem, q_desc + off, k_desc + off, C::kIdescS, ks > 0 ? 1u : 0u);
    }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate)
{
    using C = Cfg<D>;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        // 16 keys = 16 rows of the V tile (2 swizzle atoms of 8 rows); P columns hold bf16 pairs.
        mma_ts(d_tmem, p_tmem + ks * 8, v_desc + ((ks * 2048) >> 4), C::kIdescPV,
               (accumulate || ks > 0) ? 1u : 0u);
    }
}

// ---------------------------------------------------------------- TMA producers

template <int D, bool kTable, class Sched>
__device__ void produce_qk(Cta c, const TcParams& p, const Sched& sch, const CUtensorMap* tm_q,
                           const CUtensorMap* tm_k)
{
    using C = Cfg<D>;
    uint32_t kc = 0;    // K blocks issued so far (ring position)
    int qn[2] = {0, 0};  // Q tiles issued so far, per tile
    bool ok = true;
    UnitIter<kTable> it;
    for (int slot; ok && (slot = it.next(p, sch)) >= 0;) {
        if (c.aborted()) break;
        unit_setup<Sched>(c, p, slot);
        for (int t = 0; t < 2 && ok; ++t) {
            if (c.nblk[t] == 0) continue;
            // The previous unit's S MMAs of this tile must have finished reading Q_t.
            if (qn[t] > 0 && !mbar_wait(c.bar(C::kBarQEmpty + t), (qn[t] - 1) & 1)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(c.bar(C::kBarQFull + t), C::kTileBytes);
            for (int x = 0; x < C::kBoxes; ++x)
                tma_load_4d(c.sbase + C::kOffQ + t * C::kTileBytes + x * kBoxBytes, tm_q,
                            c.bar(C::kBarQFull + t), x * 64, c.head[t], c.row0[t], c.b[t]);
            ++qn[t];
        }
        // K_j of the unit's head (paired units: K_j of tile 0's head, then of tile 1's,
        // for the tiles that multiply block j), in the order the issuers consume them.
        for (int j = 0; ok && j < c.nblk_max; ++j) {
            for (int t = 0; ok && t < 2; ++t) {
                if (kPaired<Sched> ? j >= c.nblk[t] : t > 0) continue;
                const uint32_t s = kc % C::kKStages;
                if (c.aborted() || !mbar_wait(c.bar(C::kBarKEmpty + s), ((kc / C::kKStages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(c.bar(C::kBarKFull + s), C::kTileBytes);
                for (int x = 0; x < C::kBoxes; ++x)
                    tma_load_4d(c.sbase + C::kOffK + s * C::kTileBytes + x * kBoxBytes, tm_k,
                                c.bar(C::kBarKFull + s), x * 64, c.head[t], j * 128, c.b[t]);
                ++kc;
            }
        }
    }
    if (!ok) give_up(c, p.err_word);
    // Every copy this CTA started must land before the CTA may exit.
    for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) mbar_wait(c.bar(C::kBarQFull + t), (qn[t] - 1) & 1);
    for (uint32_t i = kc > (uint32_t)C::kKStages ? kc - C::kKStages : 0u; i < kc; ++i)
        mbar_wait(c.bar(C::kBarKFull + i % C::kKStages), (i / C::kKStages) & 1);
}

template <int D, bool kTable, class Sched>
__device__ void produce_v(Cta c, const TcParams& p, const Sched& sch, const CUtensorMap* tm_v)
{
    using C = Cfg<D>;
    uint32_t vc = 0;
    bool ok = true;
    UnitIter<kTable> it;
    for (int slot; ok && (slot = it.next(p, sch)) >= 0;) {
        if (c.aborted()) break;
        unit_setup<Sched>(c, p, slot);
        for (int j = 0; ok && j < c.nblk_max; ++j) {
            for (int t = 0; ok && t < 2; ++t) {
                if (kPaired<Sched> ? j >= c.nblk[t] : t > 0) continue;
                const uint32_t s = vc % C::kVStages;
                if (c.aborted() || !mbar_wait(c.bar(C::kBarVEmpty + s), ((vc / C::kVStages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(c.bar(C::kBarVFull + s), C::kTileBytes);
                for (int x = 0; x < C::kBoxes; ++x)
                    tma_load_4d(c.sbase + C::kOffV + s * C::kTileBytes + x * kBoxBytes, tm_v,
                                c.bar(C::kBarVFull + s), x * 64, c.head[t], j * 128, c.b[t]);
                ++vc;
            }
        }
    }
    if (!ok) give_up(c, p.err_word);
    for (uint32_t i = vc > (uint32_t)C::kVStages ? vc - C::kVStages : 0u; i < vc; ++i)
        mbar_wait(c.bar(C::kBarVFull + i % C::kVStages), (i / C::kVStages) & 1);
}

// ---------------------------------------------------------------- MMA issuers

// Issues every MMA of tile t (one thread), unit after unit. The K/V "empty"
// barriers expect one arrival per issuer and block: a block this tile does not
// multiply is released by a plain arrive once its copy has landed (so the
// arrival belongs to the phase of that block). After the unit's last S MMA of
// the tile, a commit onto the tile's Q-empty barrier lets the producer load
// the next unit's Q tile.
template <int D, bool kTable, class Sched>
__device__ void issue_tile_mmas(Cta c, const TcParams& p, const Sched& sch, int t)
{
    using C = Cfg<D>;
    const uint32_t tS = c.tmem + 256u * t, tP = tS + C::kColP, tO = tS + C::kColO;
    // K-major Q/K tiles: SBO = 1024 (8-row groups); MN-major V: LBO = one 64-column box.
    const uint64_t q_desc = sdesc_sw128(c.sbase + C::kOffQ + t * C::kTileBytes, 16, 1024);
    const uint64_t k_desc0 = sdesc_sw128(c.sbase + C::kOffK, 16, 1024);
    const uint64_t v_desc0 = sdesc_sw128(c.sbase + C::kOffV, kBoxBytes, 1024);
    auto kdesc = [&](uint32_t s) { return k_desc0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4); };
    auto vdesc = [&](uint32_t s) { return v_desc0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4); };

    uint32_t kc = 0, vc = 0, pc = 0, qn = 0;  // K / V blocks, P handoffs, Q tiles so far
    uint32_t sfc = 0;                         // S read-outs waited for (separate P only)
    bool ok = true;
    Ahead<kTable, BlockCounts> units;
    BlockCounts u;
    while (ok && units.advance(u, p, sch, c.causal, t)) {
        if (c.aborted()) {
            ok = false;
            break;
        }
        const int n0 = u.n0, n1 = u.n1;
        const int nb = t ? n1 : n0;
        // Rounds this issuer walks: every block of a shared unit (releasing the ones
        // its tile does not multiply), only its own blocks in a paired unit.
        const int R = kPaired<Sched> ? nb : max(n0, n1);
        // The unit's K/V ring entries, and the position of this tile's block j among
        // them (paired units: block j of tile 0, then of tile 1, for the tiles that have it).
        const uint32_t entries = static_cast<uint32_t>(kPaired<Sched> ? n0 + n1 : max(n0, n1));
        auto pos = [&](int j) -> uint32_t {
            if constexpr (!kPaired<Sched>) return static_cast<uint32_t>(j);
            return static_cast<uint32_t>(min(j, n0) + min(j, n1) + ((t == 1 && j < n0) ? 1 : 0));
        };
        if (R == 0) {
            kc += entries;
            vc += entries;
            continue;
        }
        if (nb > 0) {
            if (!mbar_wait(c.bar(C::kBarQFull + t), qn & 1)) { ok = false; break; }
            ++qn;
        }
        {
            const uint32_t k0 = kc + pos(0);
            const uint32_t s = k0 % C::kKStages;
            if (!mbar_wait(c.bar(C::kBarKFull + s), (k0 / C::kKStages) & 1)) { ok = false; break; }
            if (nb > 0) {
                tc_fence_after();
                issue_qk<D>(tS, q_desc, kdesc(s));
                mma_commit(c.bar(C::kBarS + t));
                mma_commit(c.bar(C::kBarKEmpty + s));
                if (nb == 1) mma_commit(c.bar(C::kBarQEmpty + t));
            } else {
                mbar_arrive(c.bar(C::kBarKEmpty + s));
            }
        }
        units.prefetch(p, sch, c.causal, t);  // while this unit's blocks are waited for
        for (int j = 0; ok && j < R; ++j) {
            const uint32_t vi = vc + pos(j), ki = kc + pos(j + 1);
            const uint32_t sv = vi % C::kVStages, phv = (vi / C::kVStages) & 1;
            const uint32_t sk1 = ki % C::kKStages, phk1 = (ki / C::kKStages) & 1;
            const bool has_next = j + 1 < R;
            if constexpr (C::kSepP) {
                // S(j+1) first: it only needs the softmax to have read S(j) out of TMEM.
                if (has_next) {
                    if (!mbar_wait(c.bar(C::kBarKFull + sk1), phk1)) { ok = false; break; }
                    if (j + 1 < nb) {
                        if (c.aborted() || !mbar_wait(c.bar(C::kBarSFree + t), sfc & 1)) { ok = false; break; }
                        ++sfc;
                        tc_fence_after();
                        issue_qk<D>(tS, q_desc, kdesc(sk1));
                        mma_commit(c.bar(C::kBarS + t));
                        mma_commit(c.bar(C::kBarKEmpty + sk1));
                        if (j + 1 == nb - 1) mma_commit(c.bar(C::kBarQEmpty + t));
                    } else {
                        mbar_arrive(c.bar(C::kBarKEmpty + sk1));
                    }
                }
                if (!mbar_wait(c.bar(C::kBarVFull + sv), phv)) { ok = false; break; }
                if (j < nb) {
                    if (c.aborted() || !mbar_wait(c.bar(C::kBarP + t), pc & 1)) { ok = false; break; }
                    ++pc;
                    tc_fence_after();
                    issue_pv<D>(tO, tP, vdesc(sv), j > 0);
                    mma_commit(c.bar(j == nb - 1 ? C::kBarO + t : C::kBarPVDone + t));
                    mma_commit(c.bar(C::kBarVEmpty + sv));
                } else {
                    mbar_arrive(c.bar(C::kBarVEmpty + sv));
                }
                continue;
            }
            if (!mbar_wait(c.bar(C::kBarVFull + sv), phv)) { ok = false; break; }
            if (j < nb) {
                // K(j+1) has normally landed long before P(j) is written; waiting for it
                // first keeps the wait off the path from P(j) to S(j+1).
                if (has_next && !mbar_wait(c.bar(C::kBarKFull + sk1), phk1)) { ok = false; break; }
                if (c.aborted() || !mbar_wait(c.bar(C::kBarP + t), pc & 1)) { ok = false; break; }
                ++pc;
                tc_fence_after();
                issue_pv<D>(tO, tS, vdesc(sv), j > 0);
                // S(j+1) right behind PV(j); the commits that only release buffers follow it.
                if (has_next && j + 1 < nb) {
                    issue_qk<D>(tS, q_desc, kdesc(sk1));
                    mma_commit(c.bar(C::kBarS + t));
                    mma_commit(c.bar(C::kBarKEmpty + sk1));
                    if (j + 1 == nb - 1) mma_commit(c.bar(C::kBarQEmpty + t));
                } else if (has_next) {
                    mbar_arrive(c.bar(C::kBarKEmpty + sk1));
                }
                if (j == nb - 1) mma_commit(c.bar(C::kBarO + t));
                mma_commit(c.bar(C::kBarVEmpty + sv));
            } else {
                mbar_arrive(c.bar(C::kBarVEmpty + sv));
                if (has_next) {
                    if (!mbar_wait(c.bar(C::kBarKFull + sk1), phk1)) { ok = false; break; }
                    mbar_arrive(c.bar(C::kBarKEmpty + sk1));
                }
            }
        }
        kc += entries;
        vc += entries;
    }
    if (!ok) give_up(c, p.err_word);
    // All issued MMAs must complete before TMEM is released.
    mma_commit(c.bar(C::kBarDrain + t));
    mbar_wait(c.bar(C::kBarDrain + t), 0);
}

// ---------------------------------------------------------------- softmax + epilogue

// One tile's view of a unit, all that its softmax warps keep (fewer live
// registers next to the 128 scores of a row than the whole unit).
struct TileUnit {
    int b, head, row0, nb, R, kv_len;
    bool valid;
    __device__ __forceinline__ static TileUnit of(const UnitInfo& u, int t);
};

__device__ __forceinline__ TileUnit TileUnit::of(const UnitInfo& u, int t)
{
    TileUnit v;
    v.b = t ? u.b[1] : u.b[0];
    v.head = t ? u.head[1] : u.head[0];
    v.row0 = t ? u.row0[1] : u.row0[0];
    v.nb = t ? u.nblk[1] : u.nblk[0];
    v.R = max(u.nblk[0], u.nblk[1]);
    v.kv_len = t ? u.kv_len[1] : u.kv_len[0];
    v.valid = t ? u.valid[1] : u.valid[0];
    return v;
}

template <int D, bool kTable, bool kLse, class Sched>
__device__ void softmax_tile(Cta c, const TcParams& p, const Sched& sch, int t, int wq, int lane)
{
    using C = Cfg<D>;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = c.tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t cS = 256u * t, cP = cS + C::kColP, cO = cS + C::kColO;
    const uint32_t my_turn = t ? kTurn1 : kTurn0, other_turn = t ? kTurn0 : kTurn1;
    uint32_t sc = 0, oc = 0;  // S blocks and O results waited for so far
    uint32_t pvc = 0;         // PV retirements waited for (separate P only)
    bool ok = true;
    Ahead<kTable, TileUnit> units;
    TileUnit u;
    while (units.advance(u, p, sch, c.causal, t)) {
        const int my_row0 = u.row0;
        const int row = my_row0 + r;
        const int my_b = u.b, my_head = u.head;
        const int kv_len = u.kv_len;
        if (!u.valid) {
            // Key length outside [1, n_k]: this tile's rows are zero and the error is
            // raised. The tile has no blocks, so it still takes the unit's rounds (the
            // other tile of a paired unit may have work) without doing any.
            __nv_bfloat16* orow = p.out + (((size_t)my_b * p.n_q + row) * p.h + my_head) * D;
            if (row < p.n_q) {
                for (int k = 0; k < D; k += 8) st_global_v4(orow + k, 0u, 0u, 0u, 0u);
                if constexpr (kLse) p.lse[((size_t)my_b * p.h + my_head) * p.n_q + row] = -INFINITY;
            }
            if (r == 0) raise_device_error(p.err_word, HATTN_EKEYLEN);
        }
        const int nb = u.nb, R = u.R;
        units.prefetch(p, sch, c.causal, t);  // while S(0) is waited for
        float m_used = -INFINITY, l = 0.0f;
        // Turn protocol over the unit's R rounds (every round is taken, with or
        // without work, so both warpgroups pass the named barriers the same number
        // of times): tile 0 waits for its turn, works, hands the turn over; tile 1
        // hands tile 0 the first turn, then waits, works, and hands it back
        // (except after the last round).
        if (kPingPong<D, Sched> && t == 1 && R > 0) named_arrive(kTurn0, 256);
        for (int j = 0; j < R; ++j) {
            ok = __all_sync(0xffffffffu, ok && !c.aborted());
            const bool work = ok && j < nb;
            uint32_t sr[128];  // raw scores q.k of this row for keys kbase .. kbase + 127
            const int kbase = j * 128;
            const bool need_mask = (kbase + 128 > kv_len) || (c.causal && kbase + 127 > my_row0);
            if (work) {
                const bool got = mbar_wait(c.bar(C::kBarS + t), sc & 1);
                ++sc;
                ok = __all_sync(0xffffffffu, got);
            }
            if (work && ok) {
                tc_fence_after();
                tmem_ld_x128(lane_base + cS, sr);
                if constexpr (C::kSepP) {
                    // S is in registers: the issuer may overwrite it with S(j+1).
                    if (j + 1 < nb) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(c.bar(C::kBarSFree + t));
                    }
                }
                if (need_mask) {
                    // Key kbase + i is visible iff i < lim (inside the key length and,
                    // when causal, not after this row): one compare per score.
                    const int lim = min(kv_len, c.causal ? row + 1 : kv_len) - kbase;
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i >= lim) sr[i] = __float_as_uint(-INFINITY);
                }
                // The first block sets the running max before its exponentials.
                if (j == 0) m_used = row_max(sr) * p.scale_log2;
            }
            if (kPingPong<D, Sched>) named_sync(my_turn, 256);
            if constexpr (C::kSepP) {
                // PV(j-1) must have read P before it is overwritten (and O must be
                // complete before a rescale).
                if (work && ok && j > 0) {
                    const bool got = mbar_wait(c.bar(C::kBarPVDone + t), pvc & 1);
                    ++pvc;
                    ok = __all_sync(0xffffffffu, got);
                    tc_fence_after();
                }
            }
            if (work && ok) {
                // p = 2^(s * scale * log2(e) - m) with the running max m (scale > 0, so
                // the max of scale * s is scale * max s). After the first block the
                // block's own max is found alongside the exponentials; a row whose max
                // grows by more than 2^8 (rare) rescales O and l and redoes the block.
                const uint64_t c2 = f32x2(p.scale_log2, p.scale_log2);
                uint64_t acc[4] = {0, 0, 0, 0};
                const float mx = exp_block<true>(sr, c2, f32x2(-m_used, -m_used), acc, lane_base + cP) *
                                 p.scale_log2;
                const bool grow = j > 0 && mx > m_used + kRescaleLog2;
                if (__any_sync(0xffffffffu, grow)) {
                    const float m_new = grow ? mx : m_used;
                    const float alpha = ex2_approx(m_used - m_new);  // 1 where the max is kept
#pragma unroll
                    for (int q = 0; q < D / 16; ++q) {
                        uint32_t o[16];
                        tmem_ld_x16(lane_base + cO + 16 * q, o);  // PV up to block j-1 is complete
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st_x16(lane_base + cO + 16 * q, o);
                    }
                    l *= alpha;
                    m_used = m_new;
                    acc[0] = acc[1] = acc[2] = acc[3] = 0;
                    exp_block<false>(sr, c2, f32x2(-m_used, -m_used), acc, lane_base + cP);
                }
                if (kPingPong<D, Sched> && (t == 0 || j + 1 < R)) named_arrive(other_turn, 256);
                float a0, a1;
                f32x2_split(add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3])), a0, a1);
                l += a0 + a1;
                // Each thread's TMEM stores are complete and fenced before the warp
                // synchronises; one arrival per warp (128 single-thread arrivals on one
                // barrier word would serialise).
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(c.bar(C::kBarP + t));
            } else if (kPingPong<D, Sched> && (t == 0 || j + 1 < R)) {
                named_arrive(other_turn, 256);
            }
        }
        if (nb == 0 || !ok) continue;
        {
            const bool got = mbar_wait(c.bar(C::kBarO + t), oc & 1);
            ++oc;
            ok = __all_sync(0xffffffffu, got);
        }
        if (!ok) continue;
        tc_fence_after();
        // O is in registers after the loads below; the next unit's first PV of this
        // tile (which overwrites O) waits for this warpgroup's next P handoff.
        const float inv = 1.0f / l;
        __nv_bfloat16* orow = p.out + (((size_t)my_b * p.n_q + row) * p.h + my_head) * D;
        // Natural-log log-sum-exp of the scaled scores: the exponentials ran in base 2
        // on s * scale * log2(e) with the running max m, so ln sum = (m + log2 l) ln 2.
        if constexpr (kLse) {
            if (row < p.n_q)
                p.lse[((size_t)my_b * p.h + my_head) * p.n_q + row] = (m_used + log2f(l)) * 0.6931471805599453f;
        }
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld_x32(lane_base + cO + 32 * q, o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            if (row < p.n_q) {
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    st_global_v4(orow + 32 * q + 8 * v4, pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                 pk[4 * v4 + 3]);
            }
        }
    }
    if (!ok) give_up(c, p.err_word);
}

// Before the grid dependency: the first unit's Q tiles and the K and V of its
// first two key blocks into L2 (tma_prefetch_4d: only L2 is warmed, so inputs the
// previous kernel still writes are read again later). The key length is taken as
// n_k here, since key_lens may be an output of the previous kernel too.
template <int D, bool kTable, class Sched>
__device__ void prefetch_first_unit(const TcParams& p, const Sched& sch, bool causal, const CUtensorMap* tm_q,
                                    const CUtensorMap* tm_k, const CUtensorMap* tm_v)
{
    using C = Cfg<D>;
    UnitIter<kTable> it;
    const int slot = it.next(p, sch);
    if (slot < 0) return;
    TcParams q = p;
    q.mask_kind &= ~HATTN_MASK_KEY_PADDING;
    const UnitInfo u = unit_decode<kPaired<Sched>>(q, causal, slot);
    for (int t = 0; t < 2; ++t) {
        if (u.nblk[t] == 0) continue;
        for (int x = 0; x < C::kBoxes; ++x) tma_prefetch_4d(tm_q, x * 64, u.head[t], u.row0[t], u.b[t]);
        // A shared unit's tiles read the same K and V: tile 0 prefetches them.
        if (!kPaired<Sched> && t > 0) continue;
        const int nb = min(kPaired<Sched> ? u.nblk[t] : max(u.nblk[0], u.nblk[1]), 2);
        for (int j = 0; j < nb; ++j)
            for (int x = 0; x < C::kBoxes; ++x) {
                tma_prefetch_4d(tm_k, x * 64, u.head[t], j * 128, u.b[t]);
                tma_prefetch_4d(tm_v, x * 64, u.head[t], j * 128, u.b[t]);
            }
    }
}

// ---------------------------------------------------------------- kernel

template <int D, bool kTable, bool kLse, class Sched>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const TcParams p,
                   const __grid_constant__ Sched sch)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffSlot);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    Cta c;
    c.sbase = smem_u32(smem);
    c.bar0 = c.sbase + C::kOffBar;
    c.abort_flag = c.sbase + C::kOffSlot + 4;
    c.causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(c.bar(C::kBarQFull + t), 1);
            mbar_init(c.bar(C::kBarQEmpty + t), 1);
        }
        // A K/V entry is released by every issuer of a shared unit, by its own
        // tile's issuer alone in a paired unit.
        const uint32_t releases = kPaired<Sched> ? 1u : static_cast<uint32_t>(p.issuers);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(c.bar(C::kBarKFull + s), 1);
            mbar_init(c.bar(C::kBarKEmpty + s), releases);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(c.bar(C::kBarVFull + s), 1);
            mbar_init(c.bar(C::kBarVEmpty + s), releases);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(c.bar(C::kBarS + t), 1);
            mbar_init(c.bar(C::kBarP + t), 4);
            mbar_init(c.bar(C::kBarO + t), 1);
            mbar_init(c.bar(C::kBarSFree + t), 4);
            mbar_init(c.bar(C::kBarPVDone + t), 1);
        }
        mbar_init(c.bar(C::kBarDrain), 1);
        mbar_init(c.bar(C::kBarDrain + 1), 1);
        st_volatile_shared(c.abort_flag, 0u);
        fence_barrier_init();
    }
    if (warp == kWarpMma0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kWarpLoadK && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        // Measured: paired units (n_q <= 128, one or two key blocks each) gain ~9 % from
        // it on the cross-attention workload; long units lose ~1 % (the duplicate
        // requests delay the real loads where the tiles are too many to hide anyway).
        if (kPaired<Sched>) prefetch_first_unit<D, kTable>(p, sch, c.causal, &tm_q, &tm_k, &tm_v);
    }
    if (warp == kWarpLoadV && lane == 0) prefetch_tmap(&tm_v);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tmem_slot;
    // Set-up above overlaps the previous kernel's tail; its outputs are read below.
    griddep_wait();
    griddep_launch_dependents();

    if (warp < kWarpSoftmax0) {
        regs_dec<kRegsControl>();
        if (lane == 0) {
            if (warp == kWarpLoadK) produce_qk<D, kTable>(c, p, sch, &tm_q, &tm_k);
            else if (warp == kWarpLoadV) produce_v<D, kTable>(c, p, sch, &tm_v);
            else if (warp == kWarpMma0) issue_tile_mmas<D, kTable>(c, p, sch, 0);
            else if (warp == kWarpMma1 && p.issuers == 2) issue_tile_mmas<D, kTable>(c, p, sch, 1);
        }
        __syncwarp();
    } else {
        regs_inc<kRegsSoftmax>();
        softmax_tile<D, kTable, kLse>(c, p, sch, (warp - kWarpSoftmax0) / 4, warp % 4, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma0) {
        tc_fence_after();
        tmem_dealloc(c.tmem, 512);
    }
}

// Greedy list scheduling of the unit slots (in their order) onto `grid` CTAs,
// each unit costing its key-block count per tile plus a fixed per-unit
// overhead; the owner table is cached per shape.
std::shared_ptr<const SchedTable> greedy_table(const TcParams& p, int grid)
{
    struct Key {
        int B, h, n_q, n_k, mask, grid, group;
        bool operator==(const Key& o) const
        {
            return B == o.B && h == o.h && n_q == o.n_q && n_k == o.n_k && mask == o.mask &&
                   grid == o.grid && group == o.group;
        }
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, std::shared_ptr<const SchedTable>>> cache;
    const Key key{p.B, p.h, p.n_q, p.n_k, p.mask_kind, grid, p.group_heads};
    std::lock_guard<std::mutex> lock(mu);
    for (auto& e : cache)
        if (e.first == key) return e.second;
    std::vector<int> owner(p.units);
    using Load = std::pair<long long, int>;  // (accumulated cost, cta)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int i = 0; i < grid; ++i) heap.push({0, i});
    const int kv_blocks = (p.n_k + 127) / 128;
    const bool causal = (p.mask_kind & HATTN_MASK_CAUSAL) != 0;
    const int per_group = p.group_heads * p.n_pairs;
    const int BH = p.B * p.h;
    constexpr long long kUnitOverhead = 2;  // in key blocks
    for (int slot = 0; slot < p.units; ++slot) {
        const int g = slot / per_group;
        const int w = slot - g * per_group;
        const int heads_here = std::min(p.group_heads, BH - g * p.group_heads);
        const int pi = w / heads_here;
        const int pair = causal ? p.n_pairs - 1 - pi : pi;
        long long cost = kUnitOverhead;
        for (int t = 0; t < 2; ++t) {
            const int row0 = pair * kRowsPerCta + 128 * t;
            if (row0 < p.n_q) cost += causal ? std::min(kv_blocks, row0 / 128 + 1) : kv_blocks;
        }
        Load top = heap.top();
        heap.pop();
        owner[slot] = top.second;
        heap.push({top.first + cost, top.second});
    }
    auto tab = std::make_shared<SchedTable>();
    std::memset(tab.get(), 0, sizeof(SchedTable));
    std::vector<int> count(grid + 1, 0);
    for (int slot = 0; slot < p.units; ++slot) ++count[owner[slot] + 1];
    for (int i = 0; i < grid; ++i) count[i + 1] += count[i];
    for (int i = 0; i <= kTableCtas; ++i) tab->first[i] = static_cast<uint16_t>(count[std::min(i, grid)]);
    std::vector<int> fill(count.begin(), count.end() - 1);
    for (int slot = 0; slot < p.units; ++slot) tab->list[fill[owner[slot]]++] = static_cast<uint16_t>(slot);
    if (cache.size() >= 64) cache.clear();
    cache.emplace_back(key, tab);
    return tab;
}

template <int D, bool kTable, bool kLse, class Sched>
cudaError_t launch_kernel_lse(const AttnArgs& a, const AttnMaps& m, const TcParams& p, int grid,
                              const Sched& sch)
{
    using C = Cfg<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, kTable, kLse, Sched>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, kTable, kLse, Sched>, m.q, m.k, m.v, p, sch);
}

// The log-sum-exp output is a separate instantiation, so the plain forward's
// softmax code (and its register allocation) does not carry it.
template <int D, bool kTable, class Sched>
cudaError_t launch_kernel(const AttnArgs& a, const AttnMaps& m, const TcParams& p, int grid,
                          const Sched& sch)
{
    if (p.lse) return launch_kernel_lse<D, kTable, true>(a, m, p, grid, sch);
    return launch_kernel_lse<D, kTable, false>(a, m, p, grid, sch);
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const AttnMaps& m)
{
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
    p.lse = a.lse;
    p.err_word = a.err_word;
    // Query rows that fit one tile: a unit's two tiles take two heads.
    const bool paired = a.n_q <= 128;
    p.issuers = (a.n_q > 128 || (paired && (long long)a.B * a.h > 1)) ? 2 : 1;
    const long long units = paired ? ((long long)a.B * a.h + 1) / 2 : (long long)p.n_pairs * a.B * a.h;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.units = static_cast<int>(units);
    // Heads per group: their K and V together take at most ~32 MB of the 129 MB L2
    // (measured on the long causal d = 128 workload at B = 2: DRAM reads 1.35x the
    // input bytes with 64 MB groups, 1.00x with 32 MB or 16 MB, at the same speed).
    const long long kv_head_bytes = 4LL * a.n_k * D;
    long long g = (32LL << 20) / kv_head_bytes;
    g = std::max(1LL, std::min(g, (long long)a.B * a.h));
    p.group_heads = static_cast<int>(g);
    const int grid = static_cast<int>(std::min<long long>(units, std::min(sm_count(), kTableCtas)));
    const bool causal = (a.mask_kind & HATTN_MASK_CAUSAL) != 0;
    if (paired) return launch_kernel<D, false>(a, m, p, grid, SchedPaired{});
    if (causal && units > grid && units <= kTableUnits) {
        const std::shared_ptr<const SchedTable> tab = greedy_table(p, grid);
        return launch_kernel<D, true>(a, m, p, grid, *tab);
    }
    return launch_kernel<D, false>(a, m, p, grid, SchedSnake{});
}

}  // namespace

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 152;
    return n;
}

bool attn_tc_supported(const AttnArgs& a)
{
    return a.dtype == HATTN_BF16 && a.d_k == a.d_v && (a.d_k == 64 || a.d_k == 128) &&
           a.scale > 0.0f;
}

cudaError_t launch_attn_tc(const AttnArgs& a, const AttnMaps& maps)
{
    return a.d_k == 64 ? launch_d<64>(a, maps) : launch_d<128>(a, maps);
}

}  // namespace hattn
