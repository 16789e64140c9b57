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

    __shared__ __align__(8) uint64_t bar_res;
    __shared__ __align__(8) uint64_t bar_qfull[C::QSTAGES];
    __shared__ __align__(8) uint64_t bar_qempty[C::QSTAGES];
    __shared__ __align__(8) uint64_t bar_gfull[C::GSTAGES];
    __shared__ __align__(8) uint64_t bar_gempty[C::GSTAGES];
    __shared__ __align__(8) uint64_t bar_s;     // S^T of the next block landed
    __shared__ __align__(8) uint64_t bar_dp;    // dP^T of the next block landed
    __shared__ __align__(8) uint64_t bar_p[2];  // both warpgroups wrote half x of their P^T
    __shared__ __align__(8) uint64_t bar_e[2];  // both warpgroups wrote half x of their dS^T
    __shared__ __align__(8) uint64_t bar_acc;   // accumulators final
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(16) float sL2[2][64];  // -L2 per query column [warpgroup][col]
    __shared__ __align__(16) float sDl[2][64];  // -Delta per query column
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);  // tensors stored token by token
    constexpr bool general = mode_general(MODE);  // grouped heads, Nq != Nk
    const int kblk_max = (L.Nk + 127) / 128;
    // Head-major order; within a head the first key blocks (most query blocks under the causal
    // mask) go first.
    const int bkv = static_cast<int>(blockIdx.x) / kblk_max;
    const int b = bkv / L.Hkv, hk = bkv % L.Hkv;
    const int kb = static_cast<int>(blockIdx.x) % kblk_max;
    const SeqRows sr = seq_rows<packed>(L, b);
    const int nq = sr.nq, nk = sr.nk;
    const int k0 = kb * 128, k1 = min(nk, k0 + 128);
    if (k0 >= nk) return;  // beyond this sequence's keys (whole CTA, before any sync)
    const int khead = k_head_index<packed>(L, b, hk);
    const int G = general ? L.H / L.Hkv : 1;  // query heads sharing this key/value head
    const int shift = general ? nk - nq : 0;  // bottom-right causal alignment
    const int nqblk = (nq + 127) / 128;
    int s_begin = 0;  // query blocks [s_begin, nqblk) see a key of [k0, k1)
    if (p.causal)
        while (s_begin < nqblk &&
               causal_class_shifted(s_begin * 128, min(nq, s_begin * 128 + 128), k0, k1, shift) ==
                   kTileSkip)
            ++s_begin;
    // Streamed blocks: for each query head g of the group, query blocks s_begin.. in order.
    const int n_per = nqblk - s_begin;
    const int n_it = G * n_per;

    if (threadIdx.x == 0) {
        mbar_init(&bar_res, 1);
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

    if (warp == 8) {
        // ------------------------------------------------------------- TMA producer
        mbar_arrive_expect_tx_w(&bar_res, 2 * C::TILE_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn) {
            tma_load_rows_w(sK + pn * C::PANEL_BYTES, &tm_k, &bar_res, 64 * pn, sr.k0 + k0, khead, packed);
            tma_load_rows_w(sV + pn * C::PANEL_BYTES, &tm_v, &bar_res, 64 * pn, sr.k0 + k0, khead, packed);
        }
        int issued_q = 0, issued_g = 0;
        for (int it = 0; it < n_it; ++it) {
            const int g = general ? it / n_per : 0;
            const int row = sr.q0 + (s_begin + it - g * n_per) * 128;
            const int qhead = q_head_index<packed>(L, b, hk * G + g);
            // Q first: S^T(it) is issued before dP^T(it)
            const int sq = it % C::QSTAGES;
            if (!warp_wait_all(&bar_qempty[sq], ((it / C::QSTAGES) & 1) ^ 1, wd, kSiteBwdLoadEmpty))
                break;
            mbar_arrive_expect_tx_w(&bar_qfull[sq], C::TILE_BYTES);
            for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_rows_w(sQ + sq * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q, &bar_qfull[sq],
                              64 * pn, row, qhead, packed);
            issued_q = it + 1;
            const int sg = it % C::GSTAGES;
            if (!warp_wait_all(&bar_gempty[sg], ((it / C::GSTAGES) & 1) ^ 1, wd, kSiteBwdLoadEmpty))
                break;
            mbar_arrive_expect_tx_w(&bar_gfull[sg], C::TILE_BYTES);
            if (!(it == 0 && (p.debug_flags & kDebugDropFirstLoad)))
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_rows_w(sG + sg * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_g,
                                  &bar_gfull[sg], 64 * pn, row, qhead, packed);
            issued_g = it + 1;
        }
        // drain: no copy may still be in flight when the CTA exits
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        mbar_wait(&bar_res, 0, wd_drain, kSiteBwdDrain);
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
        auto wait_q = [&](int it) {
            return warp_wait_all(&bar_qfull[it % C::QSTAGES], (it / C::QSTAGES) & 1, wd,
                                 kSiteBwdMmaQ);
        };
        auto wait_g = [&](int it) {
            return warp_wait_all(&bar_gfull[it % C::GSTAGES], (it / C::GSTAGES) & 1, wd,
                                 kSiteBwdMmaQ);
        };
        auto do_s = [&](int it) {  // S^T(it) -> S buffer
            if (!wait_q(it)) return false;
            tc_fence_after();
            dkv_issue_nt<D, C::PANEL_BYTES>(tS, dKd,
                                            sdesc_adv(dQ0, (it % C::QSTAGES) * C::TILE_BYTES), kIdNT);
            mma_commit_w(&bar_s);
            return true;
        };
        auto do_dp = [&](int it) {  // dP^T(it) -> dP buffer
            if (!wait_g(it)) return false;
            tc_fence_after();
            dkv_issue_nt<D, C::PANEL_BYTES>(tDP, dVd,
                                            sdesc_adv(dG0, (it % C::GSTAGES) * C::TILE_BYTES), kIdNT);
            mma_commit_w(&bar_dp);
            return true;
        };
        // acc += (TMEM operand) * (MN-major tile), each half issued as soon as both warpgroups
        // have written it
        auto do_acc = [&](uint64_t* bars, int it, uint32_t acc, uint32_t buf, uint64_t bdesc) {
            if (!warp_wait_all(&bars[0], it & 1, wd, kSiteBwdMmaDS)) return false;
            tc_fence_after();
            dkv_issue_acc_half<0>(acc, buf, bdesc, kIdAcc, it == 0);
            if (!warp_wait_all(&bars[1], it & 1, wd, kSiteBwdMmaDS)) return false;
            tc_fence_after();
            dkv_issue_acc_half<1>(acc, buf, bdesc, kIdAcc, it == 0);
            return true;
        };

        bool ok = warp_wait_all(&bar_res, 0, wd, kSiteBwdMmaKV);
        int committed_q = 0, committed_g = 0;
        if (ok && n_it > 0) ok = do_s(0) && do_dp(0);
        for (int it = 0; ok && it < n_it; ++it) {
            // dV += P^T(it) dO_it, then S^T(it + 1) over the P^T it just read
            if (!do_acc(bar_p, it, tDV, tS, sdesc_adv(mG0, (it % C::GSTAGES) * C::TILE_BYTES))) {
                ok = false;
                break;
            }
            mma_commit_w(&bar_gempty[it % C::GSTAGES]);
            committed_g = it + 1;
            if (it + 1 < n_it && !do_s(it + 1)) { ok = false; break; }
            // dK += dS^T(it) Q_it, then dP^T(it + 1) over the dS^T it just read
            if (!do_acc(bar_e, it, tDK, tDP, sdesc_adv(mQ0, (it % C::QSTAGES) * C::TILE_BYTES))) {
                ok = false;
                break;
            }
            mma_commit_w(&bar_qempty[it % C::QSTAGES]);
            committed_q = it + 1;
            if (it + 1 < n_it && !do_dp(it + 1)) { ok = false; break; }
        }
        if (ok) mma_commit_w(&bar_acc);
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        mma_commit_w(&bar_drain);
        mbar_wait(&bar_drain, 0, wd_drain, kSiteBwdDrain);
        for (int it = max(0, committed_q - C::QSTAGES); it < committed_q; ++it)
            mbar_wait(&bar_qempty[it % C::QSTAGES], (it / C::QSTAGES) & 1, wd_drain, kSiteBwdDrain);
        for (int it = max(0, committed_g - C::GSTAGES); it < committed_g; ++it)
            mbar_wait(&bar_gempty[it % C::GSTAGES], (it / C::GSTAGES) & 1, wd_drain, kSiteBwdDrain);
        if (ok) mbar_wait(&bar_acc, 0, wd_drain, kSiteBwdDrain);
    } else {
        // ------------------------------------------------------------- elementwise (warps 0-7)
        const int h = warp >> 2;          // query columns [64h, 64h + 64) of every block
        const int r = threadIdx.x & 127;  // key row within the block = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_base + C::COL_S + 64u * h;
        const uint32_t tDP = tbase + lane_base + C::COL_DP + 64u * h;
        const uint32_t tDV = tbase + lane_base + C::COL_DV, tDK = tbase + lane_base + C::COL_DK;
        const int krow = k0 + r;  // key row within the sequence
        const uint64_t c2x2 = f2_make(p.scale_log2, p.scale_log2);
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int g = general ? it / n_per : 0;
            const int q0 = (s_begin + it - g * n_per) * 128;  // first query of the block
            const size_t row_base =
                static_cast<size_t>(q_head_index<packed>(L, b, hk * G + g)) * L.Rq + sr.q0;
            // stage -L2 and -Delta of this warpgroup's 64 query columns (negated, so the passes
            // below are fma / add only; queries beyond N get P = 0).  The first barrier keeps
            // the previous block's values until every thread of the warpgroup is done with them.
            named_bar_sync(1 + h, 128);
            if (r < 64) {
                const int qi = q0 + 64 * h + r;
                const bool in = qi < nq && in_extent(row_base + qi, 1, L.stat_ext, p.status);
                sL2[h][r] = in ? -p.lse2[row_base + qi] : -INFINITY;
                sDl[h][r] = in ? -p.delta[row_base + qi] : 0.0f;
            }
            named_bar_sync(1 + h, 128);
            const bool diag = p.causal && causal_class_shifted(q0, min(nq, q0 + 128), k0, k1,
                                                               shift) == kTileMasked;
            // ---- phase 1: P^T = exp2(c S^T - L2), written back as bf16 pairs
            if (!warp_wait_all(&bar_s, it & 1, wd, kSiteBwdEltS)) { ok = false; break; }
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
                    f2_split(f2_fma(f2_make(__uint_as_float(pv[c + 2]), __uint_as_float(pv[c + 3])),
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
                        if (krow > q0 + 64 * h + c + shift) pv[c] = 0u;
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
            if (!warp_wait_all(&bar_dp, it & 1, wd, kSiteBwdEltS)) { ok = false; break; }
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
                                    f2_add(f2_make(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])),
                                           f2_make(nd.x, nd.y))),
                             da, db);
                    f2_split(f2_mul(f2_make(__uint_as_float(pv[i + 2]), __uint_as_float(pv[i + 3])),
                                    f2_add(f2_make(__uint_as_float(dv[c + 2]), __uint_as_float(dv[c + 3])),
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
        // ------------------------------------------------------------- epilogue
        // Warpgroup h stores accumulator columns [h*D/2, (h+1)*D/2) of its rows.
        if (ok && n_it > 0 && warp_wait_all(&bar_acc, 0, wd, kSiteBwdEltAcc)) {
            tc_fence_after();
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t tAcc = which == 0 ? tDV : tDK;
                const float mul = which == 0 ? 1.0f : p.scale;
                const long long rs = which == 0 ? L.dv_rs : L.dk_rs;
                const long long hs = which == 0 ? L.dv_hs : L.dk_hs;
                const size_t off = static_cast<size_t>(sr.k0 + krow) * rs +
                                   static_cast<size_t>(khead) * hs;
                __nv_bfloat16* dst_row = static_cast<__nv_bfloat16*>(which == 0 ? p.dv : p.dk) + off;
                const bool in = krow >= nk ||
                                in_extent(off, D, which == 0 ? L.dv_ext : L.dk_ext, p.status);
#pragma unroll 1
                for (int ch = 0; ch < D / 64; ++ch) {
                    const int c0 = h * (D / 2) + 32 * ch;
                    uint32_t a[32];
                    tmem_ld32(tAcc + c0, a);
                    tmem_wait_ld();
                    reg_fence32(a);
                    uint32_t packed[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        packed[c] = pack_bf16x2(__uint_as_float(a[2 * c]) * mul,
                                                __uint_as_float(a[2 * c + 1]) * mul);
                    if (krow < nk && in) {
                        uint4* dst = reinterpret_cast<uint4*>(dst_row + c0);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                                packed[4 * c + 3]);
                    }
                }
            }
        } else if (n_it == 0 && krow < nk) {
            // a key block that no query sees (a sequence without queries) has zero gradient
            const size_t offk = static_cast<size_t>(sr.k0 + krow) * L.dk_rs +
                                static_cast<size_t>(khead) * L.dk_hs;
            const size_t offv = static_cast<size_t>(sr.k0 + krow) * L.dv_rs +
                                static_cast<size_t>(khead) * L.dv_hs;
            const bool ink = in_extent(offk, D, L.dk_ext, p.status);
            const bool inv = in_extent(offv, D, L.dv_ext, p.status);
            for (int c = h * (D / 2); c < (h + 1) * (D / 2); ++c) {
                if (ink) static_cast<__nv_bfloat16*>(p.dk)[offk + c] = __float2bfloat16_rn(0.0f);
                if (inv) static_cast<__nv_bfloat16*>(p.dv)[offv + c] = __float2bfloat16_rn(0.0f);
            }
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
    fa_bwd_dkv_tc_kernel<D, MODE><<<grid, C::THREADS, C::SMEM_BYTES, st>>>(k, v, q, g, p);
    return cudaGetLastError();
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
