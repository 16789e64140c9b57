// dQ of backward attention on sm_103a tensor cores: the dQ loop of "Backward 구현" in
// "Triton 06: Flash Attention v2" (after the Delta preprocess).  A CTA owns one block of 128
// query rows (Q_i and dO_i resident in shared memory, the row's base-2 LSE and Delta in
// registers) and sweeps the key blocks j it sees, accumulating in Tensor Memory:
//   S = Q_i K_j^T,  dP = dO_i V_j^T                    (tcgen05, N = 128, operands in smem)
//   P = exp2(c S - L2_i),  dS = P o (dP - Delta_i)     (elementwise warpgroups)
//   acc += dS K_j                                        (tcgen05, dS from TMEM)
// and dQ_i = scale * acc.  S and P are recomputed ("Flash Attention IO-awareness principle",
// recomputation); nothing N x N reaches device memory and there are no atomics.
//
// Roles (18 warps): warps 0-15 elementwise, warpgroup h owning key columns [32h, 32h+32) of
// every block (thread = query row = TMEM lane); warp 16 TMA producer; warp 17 TMEM allocator
// and MMA issuer (whole warp, one elected lane issues).
//
// TMEM: one S buffer, two dP buffers, the accumulator.  The bf16 dS of block j overwrites the
// dP buffer it came from (j % 2), so the S buffer is free as soon as the elementwise warps have
// loaded S(j) into registers, and dP(j+2) can be issued as soon as acc(j) has been queued.
// Issue order, block j (tcgen05.mma operations of one CTA execute in issue order, so a
// product that overwrites a buffer runs after the one that reads it):
//   wait dS(j) | acc += dS(j) K_j | dP(j+2) -> dP buffer j % 2 | wait S(j+1) loaded |
//   S(j+2) -> S buffer
// While the elementwise warps work on block j+1 (S(j+1) and dP(j+1) were issued a block
// earlier) the pipe runs acc(j), dP(j+2), S(j+2): three 128x128x128 products of cover.  Each
// streamed tile is issued about two blocks before its first use, which hides the ~1 us latency
// of a TMA load under full load: K_j is read by S(j) and last by acc(j) (3-stage ring), V_j by
// dP(j) only (2 stages).
// TMEM columns: S [0, 128), dP buffers [128, 256) and [256, 384), acc [384, 384 + d).
// Within a dP buffer, warpgroup h's dS (16 columns of bf16 pairs) lands at [32h, 32h + 16),
// the first half of the columns it loaded itself.
#include <type_traits>

#include "fa_common.cuh"
#include "tc_ptx.cuh"

namespace fa {

template <int D>
struct DqCfg {
    static constexpr int PANELS = D / 64;
    static constexpr int PANEL_BYTES = 128 * 128;            // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;  // 128 rows x D bf16
    static constexpr int KSTAGES = 3;
    static constexpr int VSTAGES = 2;
    static constexpr int SMEM_BYTES = (2 + KSTAGES + VSTAGES) * TILE_BYTES + 1024;
    // Elementwise warpgroups: warpgroup h owns key columns [COLS h, COLS h + COLS) of every
    // block.  Nothing in the elementwise pass reduces across columns (L2 and Delta are known per
    // row), so the columns split across warpgroups with no exchange.  Four warpgroups (four
    // elementwise warps per sub-partition) measured 1.3 % faster than two at B1 H32 N32000 d128
    // causal and 1.8 % for the d = 64 backward.
    static constexpr int EW = 4;
    static constexpr int EW_WARPS = 4 * EW;
    static constexpr int COLS = 128 / EW;         // key columns per warpgroup
    static constexpr int ACC_COLS = D / EW;       // accumulator columns each warpgroup stores
    static constexpr int WARP_TMA = EW_WARPS, WARP_MMA = EW_WARPS + 1;
    static constexpr int THREADS = 32 * (EW_WARPS + 2);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_ACC = 384;  // dP buffer b at COL_DP + 128 b
};

// TMEM column (relative to a dP buffer) of the bf16 pairs of keys [16 ks, 16 ks + 16): warpgroup
// h writes the pairs of its COLS keys over the first COLS / 2 of the columns it loaded.
template <int COLS>
__host__ __device__ constexpr uint32_t dq_ds_col(int ks)
{
    return static_cast<uint32_t>(COLS * ((16 * ks) / COLS) + ((16 * ks) % COLS) / 2);
}

// D/16 k-steps of a 128 x 128 product of two K-major 128-row tiles, the first overwriting.
template <int D, int PANEL>
__device__ __forceinline__ void dq_issue_nt(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks / 4) * PANEL + (ks % 4) * 32;
        mma_ss_w(d_tmem, sdesc_adv(adesc, off), sdesc_adv(bdesc, off), idesc, ks > 0 ? 1u : 0u);
    }
}

// One work tile: query block qb of (sequence b, query head h_q), for tile index `id` of the launch
// grid, in the order of tile_order: within a head the last query blocks (most key blocks under
// the causal mask) rank first.
struct DqTile {
    SeqRows sr;
    int q0, q1;        // query rows [q0, q1) of the sequence
    int qhead, khead;  // head indices of the query-side and key-side tensors
    int shift;         // bottom-right causal alignment (nk - nq), 0 in the square layout
    int n_it;          // key blocks [0, n_it) are seen by some query of the block
    bool valid;        // the block holds at least one query of its sequence
};

template <int MODE>
__device__ __forceinline__ DqTile dq_tile(const BwdParams& p, int id)
{
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);
    constexpr bool general = mode_general(MODE);
    const int qblk_max = (L.Nq + 127) / 128;
    int bhead, rank;
    tile_order(id, L.B * L.H, qblk_max, L.order_group, bhead, rank);
    const int b = bhead / L.H, h_q = bhead % L.H;
    const int qb = qblk_max - 1 - rank;
    DqTile t;
    t.sr = seq_rows<packed>(L, b);
    const int nq = t.sr.nq, nk = t.sr.nk;
    t.q0 = qb * 128;
    t.q1 = min(nq, t.q0 + 128);
    t.valid = t.q0 < nq;
    t.qhead = q_head_index<packed>(L, b, h_q);
    t.khead = k_head_index<packed>(L, b, general ? h_q / (L.H / L.Hkv) : h_q);
    t.shift = general ? nk - nq : 0;
    int n = (nk + 127) / 128;
    if (p.causal) {
        const int kend = min(nk, t.q1 + t.shift);
        n = kend > 0 ? (kend + 127) / 128 : 0;
    }
    t.n_it = t.valid ? n : 0;
    return t;
}

template <int D, int MODE>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1)
    fa_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const BwdParams p,
                        int wait_first)
{
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sG = sQ + C::TILE_BYTES;
    uint8_t* sK = sG + C::TILE_BYTES;                  // KSTAGES tiles
    uint8_t* sV = sK + C::KSTAGES * C::TILE_BYTES;     // VSTAGES tiles

    __shared__ __align__(8) uint64_t bar_res;    // Q_i and dO_i of a tile landed
    __shared__ __align__(8) uint64_t bar_qfree;  // every S and dP product of a tile has run
    __shared__ __align__(8) uint64_t bar_kfull[C::KSTAGES];
    __shared__ __align__(8) uint64_t bar_kempty[C::KSTAGES];
    __shared__ __align__(8) uint64_t bar_vfull[C::VSTAGES];
    __shared__ __align__(8) uint64_t bar_vempty[C::VSTAGES];
    __shared__ __align__(8) uint64_t bar_s;      // S of the next block landed
    __shared__ __align__(8) uint64_t bar_sfree;  // every elementwise warp loaded S
    __shared__ __align__(8) uint64_t bar_dp[2];  // dP landed in dP buffer b
    // every elementwise warp wrote its dS of a block of parity b (and read its S, dP): bar_e[b].
    // Both products of block j + 1 are issued before the MMA warp waits for dS(j), so a single
    // barrier could complete twice before that wait; per parity it cannot (block j + 2's dP is
    // issued only after the wait).
    __shared__ __align__(8) uint64_t bar_e[2];
    __shared__ __align__(8) uint64_t bar_acc;   // accumulator of a tile final
    __shared__ __align__(8) uint64_t bar_drain;
    // Tile queue: the producer warp takes further tiles from the launch grid by cluster launch
    // control and publishes their indices (-1: none left) in a two-slot queue.
    __shared__ __align__(16) __int128 clc_resp;
    __shared__ __align__(8) uint64_t bar_clc;        // cancellation response landed
    __shared__ __align__(8) uint64_t bar_tfull[2];   // tile index published
    __shared__ __align__(8) uint64_t bar_tempty[2];  // tile index read by every other warp
    __shared__ int tile_ids[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);  // tensors stored token by token

    if (threadIdx.x == 0) {
        mbar_init(&bar_res, 1);
        mbar_init(&bar_qfree, 1);
        for (int s = 0; s < C::KSTAGES; ++s) {
            mbar_init(&bar_kfull[s], 1);
            mbar_init(&bar_kempty[s], 1);
        }
        for (int s = 0; s < C::VSTAGES; ++s) {
            mbar_init(&bar_vfull[s], 1);
            mbar_init(&bar_vempty[s], 1);
        }
        mbar_init(&bar_s, 1);
        mbar_init(&bar_sfree, C::EW_WARPS);  // one elected arrive per elementwise warp
        mbar_init(&bar_dp[0], 1);
        mbar_init(&bar_dp[1], 1);
        mbar_init(&bar_e[0], C::EW_WARPS);
        mbar_init(&bar_e[1], C::EW_WARPS);
        mbar_init(&bar_acc, 1);
        mbar_init(&bar_drain, 1);
        mbar_init(&bar_clc, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_tfull[s], 1);
            mbar_init(&bar_tempty[s], C::EW_WARPS + 1);  // elementwise warps and the MMA warp
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(&tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == C::WARP_TMA && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_g);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    const Watchdog wd{&abort_flag, p.status, p.wait_limit_ns};
    // launched as a programmatic dependent: right after the dK/dV grid, whose CTAs let this one
    // launch only once the preprocess is done, it needs no wait and runs in that grid's tail;
    // after anything else (the preprocess itself), it waits before reading
    if (wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");

    // Every role walks the same tile sequence: this CTA's own index (ordinal 0), then the
    // published ones.  Ordinal o >= 1 uses queue slot o & 1 as that slot's use (o - 1) >> 1
    // (slot 1 serves ordinals 1, 3, ...; slot 0 ordinals 2, 4, ...), so it waits for phase
    // parity ((o - 1) >> 1) & 1.  Blocks are counted over the whole
    // sequence (g) for the rings and the per-block barriers, tiles with key blocks (at) for the
    // per-tile barriers.
    auto next_tile = [&](int ti, int& next) {  // consumers: index of tile ordinal ti + 1
        const int s1 = (ti + 1) & 1;
        if (!warp_wait_all(&bar_tfull[s1], (ti >> 1) & 1, wd, kSiteBwdTile)) return false;
        next = tile_ids[s1];
        __syncwarp();
        mbar_arrive_w(&bar_tempty[s1]);
        return true;
    };

    if (warp == C::WARP_TMA) {
        // ------------------------------------------------------------- TMA producer
        int id = static_cast<int>(blockIdx.x), ti = 0, g = 0, at = 0;
        int issued_k = 0, issued_v = 0, issued_res = 0;
        bool clc_pending = false;  // a cancellation request whose response has not landed
        bool ok = true;
        for (;;) {
            const DqTile t = dq_tile<MODE>(p, id);
            if (t.n_it > 0) {
                // Q_i, dO_i of this tile once the previous tile's S and dP products have run
                if (at > 0 && !warp_wait_all(&bar_qfree, (at - 1) & 1, wd, kSiteBwdLoadEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&bar_res, 2 * C::TILE_BYTES);
                for (int pn = 0; pn < C::PANELS; ++pn) {
                    tma_load_rows_w(sQ + pn * C::PANEL_BYTES, &tm_q, &bar_res, 64 * pn,
                                    t.sr.q0 + t.q0, t.qhead, packed);
                    tma_load_rows_w(sG + pn * C::PANEL_BYTES, &tm_g, &bar_res, 64 * pn,
                                    t.sr.q0 + t.q0, t.qhead, packed);
                }
                issued_res = at + 1;
                for (int it = 0; it < t.n_it; ++it) {
                    const int gg = g + it;
                    const int row = t.sr.k0 + it * 128;
                    // V first: dP(it) is issued before S(it), and V's stage frees earlier than K's
                    const int sv = gg % C::VSTAGES;
                    if (!warp_wait_all(&bar_vempty[sv], ((gg / C::VSTAGES) & 1) ^ 1, wd,
                                       kSiteBwdLoadEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bar_vfull[sv], C::TILE_BYTES);
                    if (!(gg == 0 && (p.debug_flags & kDebugDropFirstLoad)))
                        for (int pn = 0; pn < C::PANELS; ++pn)
                            tma_load_rows_w(sV + sv * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_v,
                                            &bar_vfull[sv], 64 * pn, row, t.khead, packed);
                    issued_v = gg + 1;
                    const int sk = gg % C::KSTAGES;
                    if (!warp_wait_all(&bar_kempty[sk], ((gg / C::KSTAGES) & 1) ^ 1, wd,
                                       kSiteBwdLoadEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bar_kfull[sk], C::TILE_BYTES);
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_rows_w(sK + sk * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_k,
                                        &bar_kfull[sk], 64 * pn, row, t.khead, packed);
                    issued_k = gg + 1;
                }
                if (!ok) break;
                g += t.n_it;
                ++at;
            }
            // Take the next tile now, a few blocks before this one ends (the rings keep the
            // producer about three blocks ahead): a tile taken earlier would wait for this CTA
            // while another SM could already run it.  Request ordinal ti + 1 is the request's
            // use ti of the response barrier.
            clc_try_cancel_w(&clc_resp, &bar_clc);
            clc_pending = true;
            if (!warp_wait_all(&bar_clc, ti & 1, wd, kSiteBwdTile)) {
                ok = false;
                break;
            }
            clc_pending = false;
            const int next = clc_cancelled_x(&clc_resp);
            __syncwarp();
            const int s1 = (ti + 1) & 1;
            if (!warp_wait_all(&bar_tempty[s1], ((ti >> 1) & 1) ^ 1, wd, kSiteBwdTile)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                tile_ids[s1] = next;
                mbar_arrive(&bar_tfull[s1]);
            }
            __syncwarp();
            if (next < 0) break;
            id = next;
            ++ti;
        }
        // drain: no copy or cancellation response may still be in flight when the CTA exits
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        if (clc_pending) mbar_wait(&bar_clc, ti & 1, wd_drain, kSiteBwdDrain);
        if (issued_res > 0) mbar_wait(&bar_res, (issued_res - 1) & 1, wd_drain, kSiteBwdDrain);
        for (int it = max(0, issued_k - C::KSTAGES); it < issued_k; ++it)
            mbar_wait(&bar_kfull[it % C::KSTAGES], (it / C::KSTAGES) & 1, wd_drain, kSiteBwdDrain);
        for (int it = max(0, issued_v - C::VSTAGES); it < issued_v; ++it)
            mbar_wait(&bar_vfull[it % C::VSTAGES], (it / C::VSTAGES) & 1, wd_drain, kSiteBwdDrain);
    } else if (warp == C::WARP_MMA) {
        // ------------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdNT = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: both K-major
        constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);   // acc += (TMEM) * (MN-major)
        const uint32_t tS = tbase + C::COL_S, tAcc = tbase + C::COL_ACC;
        const uint64_t dQd = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dGd = sdesc_sw128(smem_u32(sG), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);                // K-major
        const uint64_t mK0 = sdesc_sw128(smem_u32(sK), C::PANEL_BYTES, 1024);    // MN-major
        const uint64_t dV0 = sdesc_sw128(smem_u32(sV), 16, 1024);
        auto issue_s = [=](int gg) {
            dq_issue_nt<D, C::PANEL_BYTES>(tS, dQd,
                                           sdesc_adv(dK0, (gg % C::KSTAGES) * C::TILE_BYTES), kIdNT);
        };
        auto issue_dp = [=](int gg) {
            dq_issue_nt<D, C::PANEL_BYTES>(tbase + C::COL_DP + 128u * (gg & 1), dGd,
                                           sdesc_adv(dV0, (gg % C::VSTAGES) * C::TILE_BYTES), kIdNT);
        };
        auto issue_acc = [=](int gg, bool first) {
            const uint32_t sb = tbase + C::COL_DP + 128u * (gg & 1);
            const uint64_t kb = sdesc_adv(mK0, (gg % C::KSTAGES) * C::TILE_BYTES);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // 16 keys per k-step; dS pairs of keys [16ks, +16)
                mma_ts_w(tAcc, sb + dq_ds_col<C::COLS>(ks), sdesc_adv(kb, ks * 2048), kIdAcc,
                         (!first || ks > 0) ? 1u : 0u);
        };
        auto wait_k = [&](int gg) {
            return warp_wait_all(&bar_kfull[gg % C::KSTAGES], (gg / C::KSTAGES) & 1, wd,
                                 kSiteBwdMmaQ);
        };
        auto wait_v = [&](int gg) {
            return warp_wait_all(&bar_vfull[gg % C::VSTAGES], (gg / C::VSTAGES) & 1, wd,
                                 kSiteBwdMmaQ);
        };
        // dP(gg) -> dP buffer gg % 2, releasing V's stage when it has run
        auto do_dp = [&](int gg) {
            if (!wait_v(gg)) return false;
            tc_fence_after();
            issue_dp(gg);
            mma_commit_w(&bar_dp[gg & 1]);
            mma_commit_w(&bar_vempty[gg % C::VSTAGES]);
            return true;
        };
        // S(gg) once every elementwise warp has loaded S(gg - 1)
        auto do_s = [&](int gg) {
            if (gg > 0 && !warp_wait_all(&bar_sfree, (gg - 1) & 1, wd, kSiteBwdMmaP)) return false;
            if (!wait_k(gg)) return false;
            tc_fence_after();
            issue_s(gg);
            mma_commit_w(&bar_s);
            return true;
        };

        int id = static_cast<int>(blockIdx.x), ti = 0, g = 0, at = 0;
        int committed_k = 0, committed_v = 0;
        bool ok = true;
        for (;;) {
            const int n = dq_tile<MODE>(p, id).n_it;
            if (n > 0) {
                if (!warp_wait_all(&bar_res, at & 1, wd, kSiteBwdMmaKV)) { ok = false; break; }
                // the first products of this tile run while the elementwise warps still read
                // out the previous tile's accumulator
                ok = do_s(g) && do_dp(g);
                committed_v = ok ? g + 1 : committed_v;
                if (ok && n > 1) {
                    ok = do_dp(g + 1);
                    committed_v = ok ? g + 2 : committed_v;
                    ok = ok && do_s(g + 1);
                }
                if (ok && n <= 2) mma_commit_w(&bar_qfree);  // every S, dP of the tile issued
                for (int it = 0; ok && it < n; ++it) {
                    const int gg = g + it;
                    if (!warp_wait_all(&bar_e[gg & 1], (gg >> 1) & 1, wd, kSiteBwdMmaDS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_acc(gg, it == 0);
                    mma_commit_w(&bar_kempty[gg % C::KSTAGES]);
                    committed_k = gg + 1;
                    if (it + 2 < n) {  // dP buffer gg % 2 is free once acc(gg), queued above, ran
                        if (!do_dp(gg + 2)) { ok = false; break; }
                        committed_v = gg + 3;
                        if (!do_s(gg + 2)) { ok = false; break; }
                        if (it + 3 == n) mma_commit_w(&bar_qfree);
                    }
                }
                if (!ok) break;
                mma_commit_w(&bar_acc);
                g += n;
                ++at;
            }
            int next = -1;
            if (!next_tile(ti, next)) { ok = false; break; }
            if (next < 0) break;
            id = next;
            ++ti;
        }
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        mma_commit_w(&bar_drain);
        mbar_wait(&bar_drain, 0, wd_drain, kSiteBwdDrain);
        for (int it = max(0, committed_k - C::KSTAGES); it < committed_k; ++it)
            mbar_wait(&bar_kempty[it % C::KSTAGES], (it / C::KSTAGES) & 1, wd_drain, kSiteBwdDrain);
        for (int it = max(0, committed_v - C::VSTAGES); it < committed_v; ++it)
            mbar_wait(&bar_vempty[it % C::VSTAGES], (it / C::VSTAGES) & 1, wd_drain, kSiteBwdDrain);
        if (ok && at > 0) {
            mbar_wait(&bar_acc, (at - 1) & 1, wd_drain, kSiteBwdDrain);
            mbar_wait(&bar_qfree, (at - 1) & 1, wd_drain, kSiteBwdDrain);
        }
    } else {
        // ------------------------------------------------------------- elementwise (warps 0-15)
        constexpr int CW = C::COLS;       // key columns of this warpgroup in every block
        constexpr int AC = C::ACC_COLS;   // accumulator columns this warpgroup stores
        const int h = warp >> 2;          // key columns [CW h, CW h + CW) of every block
        const int r = threadIdx.x & 127;  // query row within the block = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_base + C::COL_S + static_cast<uint32_t>(CW * h);
        const uint32_t tDP = tbase + lane_base + C::COL_DP + static_cast<uint32_t>(CW * h);
        const uint32_t tAcc = tbase + lane_base + C::COL_ACC;
        const uint64_t c2x2 = f2_make(p.scale_log2, p.scale_log2);
        // -L2 and -Delta of this thread's query row of tile t
        auto row_stats = [&](const DqTile& t, float& nL2, float& nDl) {
            nL2 = 0.0f;
            nDl = 0.0f;
            const size_t row_base = static_cast<size_t>(t.qhead) * L.Rq + t.sr.q0;
            const int qrow = t.q0 + r;
            if (t.n_it > 0 && qrow < t.sr.nq &&
                in_extent(row_base + qrow, 1, L.stat_ext, p.status)) {
                // read at L2 (not through this SM's L1): in fa_bwd this grid starts without
                // waiting, ordered after the preprocess that wrote these only through dK/dV
                nL2 = -__ldcg(p.lse2 + row_base + qrow);
                nDl = -__ldcg(p.delta + row_base + qrow);
            }
        };
        int ti = 0, g = 0, at = 0;
        bool ok = true;
        DqTile t = dq_tile<MODE>(p, static_cast<int>(blockIdx.x));
        float nL2, nDl;
        row_stats(t, nL2, nDl);
        for (;;) {
            const int nq = t.sr.nq, nk = t.sr.nk, n = t.n_it;
            const int qrow = t.q0 + r;  // row within the sequence
            const uint64_t nl2 = f2_make(nL2, nL2), nd2 = f2_make(nDl, nDl);
            for (int it = 0; ok && it < n; ++it) {
                const int gg = g + it;
                const int k0 = it * 128 + CW * h;  // first key of this warpgroup's columns
                const uint32_t tDPb = tDP + 128u * (gg & 1);  // dP(gg), then dS(gg)
                // element-wise mask: blocks straddling the causal diagonal (key > query + shift)
                // and keys beyond the sequence
                const bool diag = p.causal && causal_class_shifted(t.q0, t.q1, it * 128,
                                                                   min(nk, it * 128 + 128),
                                                                   t.shift) == kTileMasked;
                const bool tail = it * 128 + 128 > nk;
                // ---- phase 1: P = exp2(c S - L2) on S, which landed a block ago
                if (!warp_wait_all(&bar_s, gg & 1, wd, kSiteBwdEltS)) { ok = false; break; }
                tc_fence_after();
                uint32_t pv[CW];
#pragma unroll
                for (int c = 0; c < CW; c += 32) tmem_ld32(tS + c, pv + c);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < CW; c += 32) reg_fence32(pv + c);
                tc_fence_before();  // S is in registers: the buffer may take S(gg + 1)
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_sfree);
#pragma unroll
                for (int c = 0; c < CW; c += 2) {
                    const uint64_t x2 = f2_fma(
                        f2_make(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), c2x2, nl2);
                    float pa, pb;
                    f2_split(x2, pa, pb);
                    pa = ex2(pa);
                    pb = ex2(pb);
                    pv[c] = __float_as_uint(pa);
                    pv[c + 1] = __float_as_uint(pb);
                }
                if (diag || tail) {
#pragma unroll
                    for (int c = 0; c < CW; ++c) {
                        const int key = k0 + c;
                        if ((diag && key > qrow + t.shift) || key >= nk) pv[c] = 0u;
                    }
                }
                // ---- phase 2: dS = P o (dP - Delta), bf16 pairs over the first CW / 2 columns
                // one barrier per dP buffer: dP(gg + 2) is issued only after every elementwise
                // warp's arrive for block gg, so a waiter is never a full phase behind
                if (!warp_wait_all(&bar_dp[gg & 1], (gg >> 1) & 1, wd, kSiteBwdEltS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // all CW columns of dP in one round trip to Tensor Memory
                uint32_t dva[CW];
#pragma unroll
                for (int c = 0; c < CW; c += 32) tmem_ld32(tDPb + c, dva + c);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < CW; c += 32) reg_fence32(dva + c);
#pragma unroll
                for (int cb = 0; cb < CW / 32; ++cb) {
                    const uint32_t* dv = dva + 32 * cb;
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const int i = 32 * cb + c;
                        const uint64_t t2 = f2_add(
                            f2_make(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), nd2);
                        float da, db;
                        f2_split(f2_mul(f2_make(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])),
                                        t2),
                                 da, db);
                        pk[c / 2] = pack_bf16x2(da, db);
                    }
                    tmem_st16(tDPb + 16u * cb, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_e[gg & 1]);
            }
            // The next tile's index was published a few blocks ago; its row statistics load
            // while this tile's accumulator is read out.
            int next = -1;
            if (ok && !next_tile(ti, next)) ok = false;
            DqTile tn = t;
            float nL2n = 0.0f, nDln = 0.0f;
            if (next >= 0) {
                tn = dq_tile<MODE>(p, next);
                row_stats(tn, nL2n, nDln);
            }
            // ------------------------------------------------------------- epilogue
            // Warpgroup h stores accumulator columns [h*AC, (h+1)*AC) of its rows.
            if (n > 0) {
                if (ok && warp_wait_all(&bar_acc, at & 1, wd, kSiteBwdEltAcc)) {
                    tc_fence_after();
                    const size_t off = static_cast<size_t>(t.sr.q0 + qrow) * L.dq_rs +
                                       static_cast<size_t>(t.qhead) * L.dq_hs;
                    __nv_bfloat16* dst_row = static_cast<__nv_bfloat16*>(p.dq) + off;
                    const bool in = qrow >= nq || in_extent(off, D, L.dq_ext, p.status);
                    constexpr int CH = AC < 32 ? AC : 32;  // columns per Tensor Memory load
#pragma unroll 1
                    for (int ch = 0; ch < AC / CH; ++ch) {
                        const int c0 = h * AC + CH * ch;
                        uint32_t a[CH];
                        if constexpr (CH == 32) {
                            tmem_ld32(tAcc + c0, a);
                            tmem_wait_ld();
                            reg_fence32(a);
                        } else {
                            tmem_ld16(tAcc + c0, a);
                            tmem_wait_ld();
                            reg_fence16(a);
                        }
                        uint32_t packed_v[CH / 2];
#pragma unroll
                        for (int c = 0; c < CH / 2; ++c)
                            packed_v[c] = pack_bf16x2(__uint_as_float(a[2 * c]) * p.scale,
                                                      __uint_as_float(a[2 * c + 1]) * p.scale);
                        if (qrow < nq && in) st_row<CH / 16>(dst_row + c0, packed_v);
                    }
                    // the accumulator is in registers: the next tile's first product may
                    // overwrite it (the MMA warp issues it only after this warp's next arrive)
                    tc_fence_before();
                } else {
                    ok = false;
                }
                g += n;
                ++at;
            } else if (t.valid && qrow < nq) {
                // a query block that sees no key (more queries than keys, or no keys) has zero
                // gradient
                const size_t off = static_cast<size_t>(t.sr.q0 + qrow) * L.dq_rs +
                                   static_cast<size_t>(t.qhead) * L.dq_hs;
                if (in_extent(off, D, L.dq_ext, p.status))
                    for (int c = h * AC; c < (h + 1) * AC; ++c)
                        static_cast<__nv_bfloat16*>(p.dq)[off + c] = __float2bfloat16_rn(0.0f);
            }
            if (!ok || next < 0) break;
            t = tn;
            nL2 = nL2n;
            nDl = nDln;
            ++ti;
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
    // this grid does not complete before the one it follows
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int D, int MODE>
static cudaError_t launch_dq(const CUtensorMap& q, const CUtensorMap& g, const CUtensorMap& k,
                             const CUtensorMap& v, const BwdParams& p, cudaStream_t st,
                             bool after_dkv)
{
    using C = DqCfg<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fa_bwd_dq_tc_kernel<D, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid(p.L.B * p.L.H * ((p.L.Nq + 127) / 128));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int wait_first = after_dkv ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, fa_bwd_dq_tc_kernel<D, MODE>, q, g, k, v, p, wait_first);
}

// maps: [0] q, [1] k, [2] v, [3] dout (bf16, 128-row boxes)
cudaError_t launch_bwd_dq_tc(int d, const CUtensorMap* maps, const BwdParams& p, cudaStream_t st,
                             bool after_dkv)
{
    const int mode = layout_mode(p.L.cu_q, p.L.H, p.L.Hkv, p.L.Nq, p.L.Nk);
    auto run = [&](auto dc) {
        constexpr int Dc = decltype(dc)::value;
        if (mode == kModePacked) return launch_dq<Dc, kModePacked>(maps[0], maps[3], maps[1], maps[2], p, st, after_dkv);
        if (mode == kModeFixedGroup)
            return launch_dq<Dc, kModeFixedGroup>(maps[0], maps[3], maps[1], maps[2], p, st, after_dkv);
        return launch_dq<Dc, kModeFixed>(maps[0], maps[3], maps[1], maps[2], p, st, after_dkv);
    };
    return d == 64 ? run(std::integral_constant<int, 64>{}) : run(std::integral_constant<int, 128>{});
}

}  // namespace fa
