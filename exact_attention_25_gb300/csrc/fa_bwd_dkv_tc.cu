// dK and dV of backward attention on sm_103a tensor cores: the dK/dV loop of "Backward 구현" in
// "Triton 06: Flash Attention v2" (after the Delta preprocess).  A CTA owns one block of 128
// keys (K_j and V_j resident in shared memory) and sweeps the query blocks i that see it:
//   S^T = K_j Q_i^T,  dP^T = V_j dO_i^T                        (tcgen05, N = 128, smem operands)
//   P^T = exp2(c S^T - L2_i),  dS^T = P^T o (dP^T - Delta_i)   (elementwise warpgroups; the
//                                                               statistics are per column)
//   dV += P^T dO_i,  dK += dS^T Q_i                             (tcgen05, P^T, dS^T from TMEM)
// and dV_j = acc_dV, dK_j = scale * acc_dK.  S and P are recomputed from the stored LSE
// ("Flash Attention IO-awareness principle", recomputation); nothing N x N reaches device memory
// and there are no atomics, so the result is deterministic.
//
// Roles (10 warps): warps 0-7 elementwise, warpgroup h owning query columns [64h, 64h+64) of
// every block (thread = key row = TMEM lane); warp 8 TMA producer; warp 9 TMEM allocator and MMA
// issuer (whole warp, one elected lane issues).
//
// TMEM: S^T [0, 128), dP^T [128, 256), acc dV [256, 256 + d), acc dK [256 + d, 256 + 2d).  The
// elementwise pass of block i runs in two phases.  Phase 1 loads warpgroup h's 64 columns of
// S^T, computes P^T and writes it as bf16 pairs over the first 32 of them; phase 2 loads dP^T,
// computes dS^T and writes it likewise into the dP^T buffer.  Each phase writes its results in
// two halves of 32 query columns per warpgroup and signals each half on its own barrier (all
// eight warps arrive).  Issue order, block i (tcgen05.mma operations of one CTA execute in
// issue order, so a product that overwrites a buffer runs after the one that reads it):
//   wait P^T(i) half 0 | dV += (half 0) | wait half 1 | dV += (half 1) | S^T(i+1) -> S buffer |
//   wait dS^T(i) half 0 | dK += (half 0) | wait half 1 | dK += (half 1) | dP^T(i+1) -> dP buffer
// so the dV product starts while the second half of phase 1 is computed, and phase 1 of
// block i+1 overlaps dK(i) and dP^T(i+1) on the pipe.  Q_i is read by S^T(i) and last by dK(i) (3-stage ring);
// dO_i by dP^T(i) and last by dV(i) (2 stages).
#include <type_traits>

#include "fa_common.cuh"
#include "tc_ptx.cuh"

namespace fa {

template <int D>
struct DkvCfg {
    static constexpr int PANELS = D / 64;
    static constexpr int PANEL_BYTES = 128 * 128;            // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;  // 128 rows x D bf16
    static constexpr int QSTAGES = 3;
    static constexpr int GSTAGES = 2;
    static constexpr int SMEM_BYTES = (2 + QSTAGES + GSTAGES) * TILE_BYTES + 1024;
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D;
};

// D/16 k-steps of a 128 x 128 product of two K-major 128-row tiles, the first overwriting.
template <int D, int PANEL>
__device__ __forceinline__ void dkv_issue_nt(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks / 4) * PANEL + (ks % 4) * 32;
        mma_ss_w(d_tmem, sdesc_adv(adesc, off), sdesc_adv(bdesc, off), idesc, ks > 0 ? 1u : 0u);
    }
}

// acc += (bf16 pairs in TMEM buffer `buf`) * (MN-major 128-row tile), one half of the 8 k-steps
// of 16 streamed rows: warpgroup h's pairs of rows [64h, 64h+64) sit at buf + 64h + [0, 32), and
// HALF selects rows [64h + 32 HALF, 64h + 32 HALF + 32) of both warpgroups (k-steps 2 HALF,
// 2 HALF + 1, 4 + 2 HALF, 5 + 2 HALF), the columns each warpgroup finishes in that half.
template <int HALF>
__device__ __forceinline__ void dkv_issue_acc_half(uint32_t acc, uint32_t buf, uint64_t bdesc,
                                                   uint32_t idesc, bool first)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int ks = (j < 2 ? 0 : 4) + 2 * HALF + (j & 1);
        mma_ts_w(acc, buf + (ks < 4 ? 8u * ks : 64u + 8u * (ks - 4)), sdesc_adv(bdesc, ks * 2048),
                 idesc, (first && ks == 0) ? 0u : 1u);
    }
}

// One work tile: key block kb of (sequence b, key/value head hk), for tile index `id` of the launch
// grid, in the order of tile_order: within a head the first key blocks (most query blocks under
// the causal mask) rank first.  Its streamed blocks are, for each query head g of the group,
// the query blocks s_begin.. that see a key of the block.
struct DkvTile {
    SeqRows sr;
    int b, hk;
    int k0, k1;     // key rows [k0, k1) of the sequence
    int khead;      // head index of the key-side tensors
    int shift;      // bottom-right causal alignment (nk - nq), 0 in the square layout
    int s_begin;    // first query block that sees a key of the block
    int n_per;      // query blocks per query head of the group
    int n_it;       // streamed blocks: G * n_per
    bool valid;     // the block holds at least one key of its sequence
};

template <int MODE>
__device__ __forceinline__ DkvTile dkv_tile(const BwdParams& p, int id)
{
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);
    constexpr bool general = mode_general(MODE);
    const int kblk_max = (L.Nk + 127) / 128;
    int bkv, rank;
    tile_order(id, L.B * L.Hkv, kblk_max, L.order_group, bkv, rank);
    DkvTile t;
    t.b = bkv / L.Hkv;
    t.hk = bkv % L.Hkv;
    t.sr = seq_rows<packed>(L, t.b);
    const int nq = t.sr.nq, nk = t.sr.nk;
    t.k0 = rank * 128;
    t.k1 = min(nk, t.k0 + 128);
    t.valid = t.k0 < nk;
    t.khead = k_head_index<packed>(L, t.b, t.hk);
    t.shift = general ? nk - nq : 0;
    const int nqblk = (nq + 127) / 128;
    int sb = 0;
    if (p.causal && t.valid)
        while (sb < nqblk && causal_class_shifted(sb * 128, min(nq, sb * 128 + 128), t.k0, t.k1,
                                                  t.shift) == kTileSkip)
            ++sb;
    t.s_begin = sb;
    t.n_per = nqblk - sb;
    const int G = general ? L.H / L.Hkv : 1;
    t.n_it = t.valid ? G * t.n_per : 0;
    return t;
}

template <int D, int MODE>
__global__ void __launch_bounds__(DkvCfg<D>::THREADS, 1)
    fa_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_g, const BwdParams p)
{
    using C = DkvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;
    uint8_t* sV = sK + C::TILE_BYTES;
    uint8_t* sQ = sV + C::TILE_BYTES;               // QSTAGES tiles
    uint8_t* sG = sQ + C::QSTAGES * C::TILE_BYTES;  // GSTAGES tiles (dO)

    __shared__ __align__(8) uint64_t bar_res;     // K_j and V_j of a tile landed
    __shared__ __align__(8) uint64_t bar_kvfree;  // every S^T and dP^T product of a tile has run
    __shared__ __align__(8) uint64_t bar_qfull[C::QSTAGES];
    __shared__ __align__(8) uint64_t bar_qempty[C::QSTAGES];
    __shared__ __align__(8) uint64_t bar_gfull[C::GSTAGES];
    __shared__ __align__(8) uint64_t bar_gempty[C::GSTAGES];
    __shared__ __align__(8) uint64_t bar_s;     // S^T of the next block landed
    __shared__ __align__(8) uint64_t bar_dp;    // dP^T of the next block landed
    __shared__ __align__(8) uint64_t bar_p[2];  // both warpgroups wrote half x of their P^T
    __shared__ __align__(8) uint64_t bar_e[2];  // both warpgroups wrote half x of their dS^T
    __shared__ __align__(8) uint64_t bar_acc;   // accumulators of a tile final
    __shared__ __align__(8) uint64_t bar_drain;
    // Tile queue: the producer warp takes further tiles from the launch grid by cluster launch
    // control and publishes their indices (-1: none left) in a two-slot queue.
    __shared__ __align__(16) __int128 clc_resp;
    __shared__ __align__(8) uint64_t bar_clc;        // cancellation response landed
    __shared__ __align__(8) uint64_t bar_tfull[2];   // tile index published
    __shared__ __align__(8) uint64_t bar_tempty[2];  // tile index read by every other warp
    __shared__ int tile_ids[2];
    __shared__ __align__(16) float sL2[2][64];  // -L2 per query column [warpgroup][col]
    __shared__ __align__(16) float sDl[2][64];  // -Delta per query column
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);  // tensors stored token by token
    constexpr bool general = mode_general(MODE);  // grouped heads, Nq != Nk
    const int G = general ? L.H / L.Hkv : 1;  // query heads sharing a key/value head

    if (threadIdx.x == 0) {
        mbar_init(&bar_res, 1);
        mbar_init(&bar_kvfree, 1);
        for (int s = 0; s < C::QSTAGES; ++s) {
            mbar_init(&bar_qfull[s], 1);
            mbar_init(&bar_qempty[s], 1);
        }
        for (int s = 0; s < C::GSTAGES; ++s) {
            mbar_init(&bar_gfull[s], 1);
            mbar_init(&bar_gempty[s], 1);
        }
        mbar_init(&bar_s, 1);
        mbar_init(&bar_dp, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bar_p[x], 8);  // one elected arrive per elementwise warp
            mbar_init(&bar_e[x], 8);
        }
        mbar_init(&bar_acc, 1);
        mbar_init(&bar_drain, 1);
        mbar_init(&bar_clc, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_tfull[s], 1);
            mbar_init(&bar_tempty[s], 9);  // the eight elementwise warps and the MMA warp
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_g);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    const Watchdog wd{&abort_flag, p.status, p.wait_limit_ns};
    // launched as a programmatic dependent of the preprocess: read nothing before it is done;
    // then the dQ grid may launch (it reads only what the preprocess wrote, and the inputs)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Every role walks the same tile sequence: this CTA's own index (ordinal 0), then the
    // published ones.  Ordinal o >= 1 uses queue slot o & 1 as that slot's use (o - 1) >> 1, so
    // it waits for phase parity ((o - 1) >> 1) & 1.  Streamed blocks are counted over the whole
    // sequence (g) for the rings and the per-block barriers, tiles with streamed blocks (at) for
    // the per-tile barriers.
    auto next_tile = [&](int ti, int& next) {  // consumers: index of tile ordinal ti + 1
        const int s1 = (ti + 1) & 1;
        if (!warp_wait_all(&bar_tfull[s1], (ti >> 1) & 1, wd, kSiteBwdTile)) return false;
        next = tile_ids[s1];
        __syncwarp();
        mbar_arrive_w(&bar_tempty[s1]);
        return true;
    };

    if (warp == 8) {
        // ------------------------------------------------------------- TMA producer
        int id = static_cast<int>(blockIdx.x), ti = 0, g = 0, at = 0;
        int issued_q = 0, issued_g = 0, issued_res = 0;
        bool clc_pending = false;  // a cancellation request whose response has not landed
        bool ok = true;
        for (;;) {
            const DkvTile t = dkv_tile<MODE>(p, id);
            if (t.n_it > 0) {
                // K_j, V_j of this tile once the previous tile's S^T and dP^T products have run
                if (at > 0 && !warp_wait_all(&bar_kvfree, (at - 1) & 1, wd, kSiteBwdLoadEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&bar_res, 2 * C::TILE_BYTES);
                for (int pn = 0; pn < C::PANELS; ++pn) {
                    tma_load_rows_w(sK + pn * C::PANEL_BYTES, &tm_k, &bar_res, 64 * pn,
                                    t.sr.k0 + t.k0, t.khead, packed);
                    tma_load_rows_w(sV + pn * C::PANEL_BYTES, &tm_v, &bar_res, 64 * pn,
                                    t.sr.k0 + t.k0, t.khead, packed);
                }
                issued_res = at + 1;
                for (int it = 0; it < t.n_it; ++it) {
                    const int gg = g + it;
                    const int gh = general ? it / t.n_per : 0;
                    const int row = t.sr.q0 + (t.s_begin + it - gh * t.n_per) * 128;
                    const int qhead = q_head_index<packed>(L, t.b, t.hk * G + gh);
                    // Q first: S^T(it) is issued before dP^T(it)
                    const int sq = gg % C::QSTAGES;
                    if (!warp_wait_all(&bar_qempty[sq], ((gg / C::QSTAGES) & 1) ^ 1, wd,
                                       kSiteBwdLoadEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bar_qfull[sq], C::TILE_BYTES);
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_rows_w(sQ + sq * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q,
                                        &bar_qfull[sq], 64 * pn, row, qhead, packed);
                    issued_q = gg + 1;
                    const int sg = gg % C::GSTAGES;
                    if (!warp_wait_all(&bar_gempty[sg], ((gg / C::GSTAGES) & 1) ^ 1, wd,
                                       kSiteBwdLoadEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bar_gfull[sg], C::TILE_BYTES);
                    if (!(gg == 0 && (p.debug_flags & kDebugDropFirstLoad)))
                        for (int pn = 0; pn < C::PANELS; ++pn)
                            tma_load_rows_w(sG + sg * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_g,
                                            &bar_gfull[sg], 64 * pn, row, qhead, packed);
                    issued_g = gg + 1;
                }
                if (!ok) break;
                g += t.n_it;
                ++at;
            }
            // Take the next tile now, a few blocks before this one ends (a tile taken earlier
            // would wait for this CTA while another SM could already run it).  The request for
            // ordinal ti + 1 is use ti of the response barrier.
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
        for (int it = max(0, issued_q - C::QSTAGES); it < issued_q; ++it)
            mbar_wait(&bar_qfull[it % C::QSTAGES], (it / C::QSTAGES) & 1, wd_drain, kSiteBwdDrain);
        for (int it = max(0, issued_g - C::GSTAGES); it < issued_g; ++it)
            mbar_wait(&bar_gfull[it % C::GSTAGES], (it / C::GSTAGES) & 1, wd_drain, kSiteBwdDrain);
    } else if (warp == 9) {
        // ------------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdNT = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T: both K-major
        constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);   // acc += (TMEM) * (MN-major)
        const uint32_t tS = tbase + C::COL_S, tDP = tbase + C::COL_DP;
        const uint32_t tDV = tbase + C::COL_DV, tDK = tbase + C::COL_DK;
        const uint64_t dKd = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dVd = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);               // K-major
        const uint64_t mQ0 = sdesc_sw128(smem_u32(sQ), C::PANEL_BYTES, 1024);   // MN-major
        const uint64_t dG0 = sdesc_sw128(smem_u32(sG), 16, 1024);
        const uint64_t mG0 = sdesc_sw128(smem_u32(sG), C::PANEL_BYTES, 1024);
        auto wait_q = [&](int gg) {
            return warp_wait_all(&bar_qfull[gg % C::QSTAGES], (gg / C::QSTAGES) & 1, wd,
                                 kSiteBwdMmaQ);
        };
        auto wait_g = [&](int gg) {
            return warp_wait_all(&bar_gfull[gg % C::GSTAGES], (gg / C::GSTAGES) & 1, wd,
                                 kSiteBwdMmaQ);
        };
        auto do_s = [&](int gg) {  // S^T(gg) -> S buffer
            if (!wait_q(gg)) return false;
            tc_fence_after();
            dkv_issue_nt<D, C::PANEL_BYTES>(tS, dKd,
                                            sdesc_adv(dQ0, (gg % C::QSTAGES) * C::TILE_BYTES), kIdNT);
            mma_commit_w(&bar_s);
            return true;
        };
        auto do_dp = [&](int gg) {  // dP^T(gg) -> dP buffer
            if (!wait_g(gg)) return false;
            tc_fence_after();
            dkv_issue_nt<D, C::PANEL_BYTES>(tDP, dVd,
                                            sdesc_adv(dG0, (gg % C::GSTAGES) * C::TILE_BYTES), kIdNT);
            mma_commit_w(&bar_dp);
            return true;
        };
        // acc += (TMEM operand) * (MN-major tile), each half issued as soon as both warpgroups
        // have written it
        auto do_acc = [&](uint64_t* bars, int gg, bool first, uint32_t acc, uint32_t buf,
                          uint64_t bdesc) {
            if (!warp_wait_all(&bars[0], gg & 1, wd, kSiteBwdMmaDS)) return false;
            tc_fence_after();
            dkv_issue_acc_half<0>(acc, buf, bdesc, kIdAcc, first);
            if (!warp_wait_all(&bars[1], gg & 1, wd, kSiteBwdMmaDS)) return false;
            tc_fence_after();
            dkv_issue_acc_half<1>(acc, buf, bdesc, kIdAcc, first);
            return true;
        };

        int id = static_cast<int>(blockIdx.x), ti = 0, g = 0, at = 0;
        int committed_q = 0, committed_g = 0;
        bool ok = true;
        for (;;) {
            const int n = dkv_tile<MODE>(p, id).n_it;
            if (n > 0) {
                if (!warp_wait_all(&bar_res, at & 1, wd, kSiteBwdMmaKV)) { ok = false; break; }
                // the first products of this tile run while the elementwise warps still read
                // out the previous tile's accumulators
                ok = do_s(g) && do_dp(g);
                if (ok && n == 1) mma_commit_w(&bar_kvfree);  // every S^T, dP^T of the tile issued
                for (int it = 0; ok && it < n; ++it) {
                    const int gg = g + it;
                    // dV += P^T(gg) dO_gg, then S^T(gg + 1) over the P^T it just read
                    if (!do_acc(bar_p, gg, it == 0, tDV, tS,
                                sdesc_adv(mG0, (gg % C::GSTAGES) * C::TILE_BYTES))) {
                        ok = false;
                        break;
                    }
                    mma_commit_w(&bar_gempty[gg % C::GSTAGES]);
                    committed_g = gg + 1;
                    if (it + 1 < n && !do_s(gg + 1)) { ok = false; break; }
                    // dK += dS^T(gg) Q_gg, then dP^T(gg + 1) over the dS^T it just read
                    if (!do_acc(bar_e, gg, it == 0, tDK, tDP,
                                sdesc_adv(mQ0, (gg % C::QSTAGES) * C::TILE_BYTES))) {
                        ok = false;
                        break;
                    }
                    mma_commit_w(&bar_qempty[gg % C::QSTAGES]);
                    committed_q = gg + 1;
                    if (it + 1 < n) {
                        if (!do_dp(gg + 1)) { ok = false; break; }
                        if (it + 2 == n) mma_commit_w(&bar_kvfree);
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
        for (int it = max(0, committed_q - C::QSTAGES); it < committed_q; ++it)
            mbar_wait(&bar_qempty[it % C::QSTAGES], (it / C::QSTAGES) & 1, wd_drain, kSiteBwdDrain);
        for (int it = max(0, committed_g - C::GSTAGES); it < committed_g; ++it)
            mbar_wait(&bar_gempty[it % C::GSTAGES], (it / C::GSTAGES) & 1, wd_drain, kSiteBwdDrain);
        if (ok && at > 0) {
            mbar_wait(&bar_acc, (at - 1) & 1, wd_drain, kSiteBwdDrain);
            mbar_wait(&bar_kvfree, (at - 1) & 1, wd_drain, kSiteBwdDrain);
        }
    } else {
        // ------------------------------------------------------------- elementwise (warps 0-7)
        const int h = warp >> 2;          // query columns [64h, 64h + 64) of every block
        const int r = threadIdx.x & 127;  // key row within the block = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_base + C::COL_S + 64u * h;
        const uint32_t tDP = tbase + lane_base + C::COL_DP + 64u * h;
        const uint32_t tDV = tbase + lane_base + C::COL_DV, tDK = tbase + lane_base + C::COL_DK;
        const uint64_t c2x2 = f2_make(p.scale_log2, p.scale_log2);
        int id = static_cast<int>(blockIdx.x), ti = 0, g = 0, at = 0;
        bool ok = true;
        for (;;) {
            const DkvTile t = dkv_tile<MODE>(p, id);
            const int nq = t.sr.nq, nk = t.sr.nk, n_it = t.n_it;
            const int krow = t.k0 + r;  // key row within the sequence
            for (int it = 0; ok && it < n_it; ++it) {
                const int gg = g + it;
                const int gh = general ? it / t.n_per : 0;
                const int q0 = (t.s_begin + it - gh * t.n_per) * 128;  // first query of the block
                const size_t row_base =
                    static_cast<size_t>(q_head_index<packed>(L, t.b, t.hk * G + gh)) * L.Rq +
                    t.sr.q0;
                // stage -L2 and -Delta of this warpgroup's 64 query columns (negated, so the
                // passes below are fma / add only; queries beyond N get P = 0).  The first
                // barrier keeps the previous block's values until every thread of the warpgroup
                // is done with them.
                named_bar_sync(1 + h, 128);
                if (r < 64) {
                    const int qi = q0 + 64 * h + r;
                    const bool in = qi < nq && in_extent(row_base + qi, 1, L.stat_ext, p.status);
                    sL2[h][r] = in ? -p.lse2[row_base + qi] : -INFINITY;
                    sDl[h][r] = in ? -p.delta[row_base + qi] : 0.0f;
                }
                named_bar_sync(1 + h, 128);
                const bool diag = p.causal && causal_class_shifted(q0, min(nq, q0 + 128), t.k0,
                                                                   t.k1, t.shift) == kTileMasked;
                // ---- phase 1: P^T = exp2(c S^T - L2), written back as bf16 pairs
                if (!warp_wait_all(&bar_s, gg & 1, wd, kSiteBwdEltS)) { ok = false; break; }
                tc_fence_after();
                uint32_t pv[64];
                tmem_ld32(tS, pv);
                tmem_ld32(tS + 32u, pv + 32);
                tmem_wait_ld();
                reg_fence32(pv);
                reg_fence32(pv + 32);
                // in two halves of 32 columns, each signalled on its own barrier so that the MMA
                // warp can start the dV product on the first while the second is computed
#pragma unroll
                for (int x = 0; x < 2; ++x) {
#pragma unroll
                    for (int c = 32 * x; c < 32 * x + 32; c += 4) {
                        const float4 nl = *reinterpret_cast<const float4*>(&sL2[h][c]);
                        float pa, pb, pc, pd;
                        f2_split(f2_fma(f2_make(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])),
                                        c2x2, f2_make(nl.x, nl.y)),
                                 pa, pb);
                        f2_split(f2_fma(f2_make(__uint_as_float(pv[c + 2]),
                                                __uint_as_float(pv[c + 3])),
                                        c2x2, f2_make(nl.z, nl.w)),
                                 pc, pd);
                        pv[c] = __float_as_uint(ex2(pa));
                        pv[c + 1] = __float_as_uint(ex2(pb));
                        pv[c + 2] = __float_as_uint(ex2(pc));
                        pv[c + 3] = __float_as_uint(ex2(pd));
                    }
                    if (diag) {  // key > query is masked
#pragma unroll
                        for (int c = 32 * x; c < 32 * x + 32; ++c)
                            if (krow > q0 + 64 * h + c + t.shift) pv[c] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        pk[c] = pack_bf16x2(__uint_as_float(pv[32 * x + 2 * c]),
                                            __uint_as_float(pv[32 * x + 2 * c + 1]));
                    tmem_st16(tS + 16u * x, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_p[x]);
                }
                // ---- phase 2: dS^T = P^T o (dP^T - Delta), written back as bf16 pairs
                if (!warp_wait_all(&bar_dp, gg & 1, wd, kSiteBwdEltS)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t dv[32];
                    tmem_ld32(tDP + 32u * cb, dv);
                    tmem_wait_ld();
                    reg_fence32(dv);
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const int i = 32 * cb + c;
                        const float4 nd = *reinterpret_cast<const float4*>(&sDl[h][i]);
                        float da, db, dc, dd;
                        f2_split(f2_mul(f2_make(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])),
                                        f2_add(f2_make(__uint_as_float(dv[c]),
                                                       __uint_as_float(dv[c + 1])),
                                               f2_make(nd.x, nd.y))),
                                 da, db);
                        f2_split(f2_mul(f2_make(__uint_as_float(pv[i + 2]),
                                                __uint_as_float(pv[i + 3])),
                                        f2_add(f2_make(__uint_as_float(dv[c + 2]),
                                                       __uint_as_float(dv[c + 3])),
                                               f2_make(nd.z, nd.w))),
                                 dc, dd);
                        pk[c / 2] = pack_bf16x2(da, db);
                        pk[c / 2 + 1] = pack_bf16x2(dc, dd);
                    }
                    tmem_st16(tDP + 16u * cb, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_e[cb]);
                }
            }
            int next = -1;
            if (ok && !next_tile(ti, next)) ok = false;
            // ------------------------------------------------------------- epilogue
            // Warpgroup h stores accumulator columns [h*D/2, (h+1)*D/2) of its rows.
            if (n_it > 0) {
                if (ok && warp_wait_all(&bar_acc, at & 1, wd, kSiteBwdEltAcc)) {
                    tc_fence_after();
                    const size_t offv = static_cast<size_t>(t.sr.k0 + krow) * L.dv_rs +
                                        static_cast<size_t>(t.khead) * L.dv_hs;
                    const size_t offk = static_cast<size_t>(t.sr.k0 + krow) * L.dk_rs +
                                        static_cast<size_t>(t.khead) * L.dk_hs;
                    const bool inv = krow < nk && in_extent(offv, D, L.dv_ext, p.status);
                    const bool ink = krow < nk && in_extent(offk, D, L.dk_ext, p.status);
                    // dV and dK of the same 32 columns in one Tensor Memory round trip
#pragma unroll 1
                    for (int ch = 0; ch < D / 64; ++ch) {
                        const int c0 = h * (D / 2) + 32 * ch;
                        uint32_t a[32], b[32];
                        tmem_ld32(tDV + c0, a);
                        tmem_ld32(tDK + c0, b);
                        tmem_wait_ld();
                        reg_fence32(a);
                        reg_fence32(b);
                        uint32_t pv[16], pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            pv[c] = pack_bf16x2(__uint_as_float(a[2 * c]), __uint_as_float(a[2 * c + 1]));
                            pk[c] = pack_bf16x2(__uint_as_float(b[2 * c]) * p.scale,
                                                __uint_as_float(b[2 * c + 1]) * p.scale);
                        }
                        if (inv) st_row<2>(static_cast<__nv_bfloat16*>(p.dv) + offv + c0, pv);
                        if (ink) st_row<2>(static_cast<__nv_bfloat16*>(p.dk) + offk + c0, pk);
                    }
                    // the accumulators are in registers: the next tile's first products may
                    // overwrite them (the MMA warp issues those only after this warp's next
                    // arrive)
                    tc_fence_before();
                } else {
                    ok = false;
                }
                g += n_it;
                ++at;
            } else if (t.valid && krow < nk) {
                // a key block that no query sees (a sequence without queries) has zero gradient
                const size_t offk = static_cast<size_t>(t.sr.k0 + krow) * L.dk_rs +
                                    static_cast<size_t>(t.khead) * L.dk_hs;
                const size_t offv = static_cast<size_t>(t.sr.k0 + krow) * L.dv_rs +
                                    static_cast<size_t>(t.khead) * L.dv_hs;
                const bool ink = in_extent(offk, D, L.dk_ext, p.status);
                const bool inv = in_extent(offv, D, L.dv_ext, p.status);
                for (int c = h * (D / 2); c < (h + 1) * (D / 2); ++c) {
                    if (ink) static_cast<__nv_bfloat16*>(p.dk)[offk + c] = __float2bfloat16_rn(0.0f);
                    if (inv) static_cast<__nv_bfloat16*>(p.dv)[offv + c] = __float2bfloat16_rn(0.0f);
                }
            }
            if (!ok || next < 0) break;
            id = next;
            ++ti;
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

template <int D, int MODE>
static cudaError_t launch_dkv(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                              const CUtensorMap& g, const BwdParams& p, cudaStream_t st)
{
    using C = DkvCfg<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fa_bwd_dkv_tc_kernel<D, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid(p.L.B * p.L.Hkv * ((p.L.Nk + 127) / 128));
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
    return cudaLaunchKernelEx(&cfg, fa_bwd_dkv_tc_kernel<D, MODE>, k, v, q, g, p);
}

// maps: [0] q, [1] k, [2] v, [3] dout (bf16, 128-row boxes)
cudaError_t launch_bwd_dkv_tc(int d, const CUtensorMap* maps, const BwdParams& p, cudaStream_t st)
{
    const int mode = layout_mode(p.L.cu_q, p.L.H, p.L.Hkv, p.L.Nq, p.L.Nk);
    auto run = [&](auto dc) {
        constexpr int Dc = decltype(dc)::value;
        if (mode == kModePacked) return launch_dkv<Dc, kModePacked>(maps[1], maps[2], maps[0], maps[3], p, st);
        if (mode == kModeFixedGroup)
            return launch_dkv<Dc, kModeFixedGroup>(maps[1], maps[2], maps[0], maps[3], p, st);
        return launch_dkv<Dc, kModeFixed>(maps[1], maps[2], maps[0], maps[3], p, st);
    };
    return d == 64 ? run(std::integral_constant<int, 64>{}) : run(std::integral_constant<int, 128>{});
}

}  // namespace fa
