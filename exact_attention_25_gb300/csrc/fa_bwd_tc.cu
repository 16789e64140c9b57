// Backward attention on sm_103a tensor cores, in the two-loop structure of "Backward 구현" /
// "Forward/Backward 전체 흐름 요약" of "Triton 06: Flash Attention v2" (after the Delta
// preprocess): a dK/dV kernel whose CTA owns one block of 128 keys and sweeps the query
// blocks, and a dQ kernel whose CTA owns one block of 128 queries and sweeps the key blocks.
// S and P are recomputed from Q, K and the stored base-2 LSE (recomputation section of
// "Flash Attention IO-awareness principle"); nothing N x N touches device memory and no
// atomics are used, so the result is deterministic.
//
// One template serves both kernels.  With X, Y the resident tiles and A, B the streamed ones:
//   dK/dV (KV = true):  X = K_j, Y = V_j, A = Q_i, B = dO_i
//       T1 = X A^T = S^T, T2 = Y B^T = dP^T               (tcgen05, operands in smem)
//       P^T = exp2(c S^T - L2), dS^T = P^T o (dP^T - Delta)  (elementwise warpgroups)
//       acc1 += P^T B = dV,  acc2 += dS^T A = dK / scale   (tcgen05, first operand in TMEM)
//   dQ (KV = false):    X = Q_i, Y = dO_i, A = K_j, B = V_j
//       T1 = S, T2 = dP, dS = P o (dP - Delta), acc2 += dS A = dQ / scale
// Roles (10 warps): two elementwise warpgroups (warps 0-3 and 4-7; thread = row of X = TMEM
// lane), warpgroup h owning half h (streamed rows [64h, 64h+64)) of every block; warp 8 TMA
// producer; warp 9 TMEM allocator + MMA issuer (whole warp, one elected lane issues).
// Pipeline: the T1/T2 products are issued per half (N = 64), and half h of block i+1 is issued
// right after the accumulating products of half h of block i, so the tensor pipe always has
// the other half's products queued while a warpgroup runs its elementwise pass:
//   TC:  acc(i,0) | T(i+1,0) | acc(i,1) | T(i+1,1) | acc(i+1,0) | ...
//   WG0:             elementwise(i+1, 0) .........|
//   WG1:                        elementwise(i+1, 1) ..........|
// TMEM columns: half h: T1 [128h, 128h+64), T2 [128h+64, 128h+128); acc1 [256, 256+d),
// acc2 [256+d, 256+2d).  The bf16 P^T / dS^T of half h (32 columns of packed pairs) overwrite
// the first 32 columns of that half's T1 / T2, chunk by chunk, after they were loaded.
#include <type_traits>

#include "fa_common.cuh"
#include "tc_ptx.cuh"

namespace fa {

template <int D>
struct BwdCfg {
    static constexpr int PANELS = D / 64;
    static constexpr int PANEL_BYTES = 128 * 128;
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;      // 128 rows x D bf16
    static constexpr int STAGES = 2;
    static constexpr int SMEM_RES = 2 * TILE_BYTES;              // X, Y
    static constexpr int SMEM_STREAM = STAGES * 2 * TILE_BYTES;  // (A, B) per stage
    static constexpr int SMEM_BYTES = SMEM_RES + SMEM_STREAM + 1024;
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
};

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// T = X A^T for one 128-row streamed tile: D/16 k-steps of 16 (N = 128), first overwrites.
template <int D, int PANEL>
__device__ __forceinline__ void bwd_issue_t(uint32_t d_tmem, uint64_t xdesc, uint64_t adesc,
                                            uint32_t idesc)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks / 4) * PANEL + (ks % 4) * 32;
        mma_ss_w(d_tmem, sdesc_adv(xdesc, off), sdesc_adv(adesc, off), idesc, ks > 0 ? 1u : 0u);
    }
}

// Accumulating products of one 64-row half: 4 k-steps of 16 streamed rows.
// acc1 += T1(bf16) * B (dK/dV kernel only), acc2 += T2(bf16) * A; MN-major B / A descriptors
// already point at the half's first row.
template <bool KV>
__device__ __forceinline__ void bwd_issue_acc(uint32_t acc1, uint32_t acc2, uint32_t t1,
                                              uint32_t t2, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t acc_first)
{
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        const uint32_t acc = ks > 0 ? 1u : acc_first;
        if (KV) mma_ts_w(acc1, t1 + 8u * ks, sdesc_adv(bdesc, ks * 2048), idesc, acc);
        mma_ts_w(acc2, t2 + 8u * ks, sdesc_adv(adesc, ks * 2048), idesc, acc);
    }
}

template <int D, bool KV>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    fa_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_y,
                     const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b, const BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sX = smem;
    uint8_t* sY = sX + C::TILE_BYTES;
    uint8_t* sAB = sY + C::TILE_BYTES;  // stage s: A at sAB + s*2*TILE, B right after

    __shared__ __align__(8) uint64_t bar_res;
    __shared__ __align__(8) uint64_t bar_full[C::STAGES];
    __shared__ __align__(8) uint64_t bar_empty[C::STAGES];
    __shared__ __align__(8) uint64_t bar_t[2];  // half h of T1, T2 ready
    __shared__ __align__(8) uint64_t bar_e[2];  // half h of the bf16 operands written
    __shared__ __align__(8) uint64_t bar_acc;   // accumulators final
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(16) float sL2[2][2][64];  // -L2 per streamed row [half][parity][row]
    __shared__ __align__(16) float sDl[2][2][64];  // -Delta per streamed row
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = p.N;
    const int nblk = (N + 127) / 128;
    // Head-major order, so the CTAs resident at one time share one or two heads' tiles in L2.
    // Within a head the heaviest blocks go first: for dK/dV the first key blocks see the most
    // query blocks under the causal mask; for dQ the last query blocks see the most key blocks.
    const int bh = static_cast<int>(blockIdx.x) / nblk;
    const int yb = static_cast<int>(blockIdx.x) % nblk;
    const int xb = KV ? yb : nblk - 1 - yb;
    const int x0 = xb * 128, x1 = min(N, x0 + 128);
    // Streamed blocks visited: a contiguous range [s_begin, s_end).
    int s_begin = 0, s_end = nblk;
    if (p.causal) {
        if (KV) {  // query blocks that see any key of [x0, x1)
            while (s_begin < nblk &&
                   causal_tile_class(s_begin * 128, min(N, s_begin * 128 + 128), x0, x1) == kTileSkip)
                ++s_begin;
        } else {   // key blocks seen by any query of [x0, x1)
            s_end = 0;
            while (s_end < nblk &&
                   causal_tile_class(x0, x1, s_end * 128, min(N, s_end * 128 + 128)) != kTileSkip)
                ++s_end;
        }
    }
    const int n_it = s_end - s_begin;

    if (threadIdx.x == 0) {
        mbar_init(&bar_res, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bar_t[h], 1);
            mbar_init(&bar_e[h], 4);  // one elected arrive per warp of the warpgroup
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
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_y);
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    const Watchdog wd{&abort_flag, p.status, p.wait_limit_ns};

    if (warp == 8) {
        // ------------------------------------------------------------- TMA producer
        {  // the whole warp runs the loop; elect.sync picks the issuing lane
            mbar_arrive_expect_tx_w(&bar_res, 2 * C::TILE_BYTES);
            for (int pn = 0; pn < C::PANELS; ++pn) {
                tma_load_3d_w(sX + pn * C::PANEL_BYTES, &tm_x, &bar_res, 64 * pn, x0, bh);
                tma_load_3d_w(sY + pn * C::PANEL_BYTES, &tm_y, &bar_res, 64 * pn, x0, bh);
            }
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (it / C::STAGES) & 1;
                if (!warp_wait_all(&bar_empty[s], ph ^ 1, wd, kSiteBwdLoadEmpty)) break;
                uint8_t* sA = sAB + s * 2 * C::TILE_BYTES;
                uint8_t* sB = sA + C::TILE_BYTES;
                const int row = (s_begin + it) * 128;
                mbar_arrive_expect_tx_w(&bar_full[s], 2 * C::TILE_BYTES);
                for (int pn = 0; pn < C::PANELS; ++pn) {
                    tma_load_3d_w(sA + pn * C::PANEL_BYTES, &tm_a, &bar_full[s], 64 * pn, row, bh);
                    if (!(it == 0 && (p.debug_flags & kDebugDropFirstLoad)))
                        tma_load_3d_w(sB + pn * C::PANEL_BYTES, &tm_b, &bar_full[s], 64 * pn, row, bh);
                }
                issued = it + 1;
            }
            volatile int no_abort = 0;
            const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
            mbar_wait(&bar_res, 0, wd_drain, kSiteBwdDrain);
            for (int it = max(0, issued - C::STAGES); it < issued; ++it)
                mbar_wait(&bar_full[it % C::STAGES], (it / C::STAGES) & 1, wd_drain, kSiteBwdDrain);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------- MMA issuer
        {  // the whole warp runs the loop (warp-uniform values); elect.sync picks the issuer
            constexpr uint32_t kIdT = idesc_bf16_f32(128, 64, 0, 0);   // T_h = X A_h^T
            constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);  // acc += (TMEM) * (MN-major)
            const uint32_t tAcc1 = tbase + 256u, tAcc2 = tbase + 256u + D;
            // Everything the issue loop needs lives in scalar registers: base descriptors are
            // built once and advanced by byte offsets (stage, half, k-step), so the single
            // issuing thread keeps pace with the tensor core.
            const uint64_t dX = sdesc_sw128(smem_u32(sX), 16, 1024);
            const uint64_t dY = sdesc_sw128(smem_u32(sY), 16, 1024);
            const uint64_t dA0 = sdesc_sw128(smem_u32(sAB), 16, 1024);           // K-major
            const uint64_t mA0 = sdesc_sw128(smem_u32(sAB), C::PANEL_BYTES, 1024);  // MN-major
            // T1, T2 of half h of streamed block `it` (streamed rows [64h, 64h+64)).
            auto issue_t = [=](int it, int h) {
                const uint32_t so = (it % C::STAGES) * 2 * C::TILE_BYTES + 8192u * h;
                const uint32_t t1 = tbase + 128u * h;
                bwd_issue_t<D, C::PANEL_BYTES>(t1, dX, sdesc_adv(dA0, so), kIdT);
                bwd_issue_t<D, C::PANEL_BYTES>(t1 + 64u, dY, sdesc_adv(dA0, so + C::TILE_BYTES), kIdT);
            };
            // Accumulating products of half h of streamed block `it`.
            auto issue_acc = [=](int it, int h) {
                const uint32_t so = (it % C::STAGES) * 2 * C::TILE_BYTES + 8192u * h;
                const uint32_t t1 = tbase + 128u * h;
                bwd_issue_acc<KV>(tAcc1, tAcc2, t1, t1 + 64u, sdesc_adv(mA0, so),
                                  sdesc_adv(mA0, so + C::TILE_BYTES), kIdAcc,
                                  (it > 0 || h > 0) ? 1u : 0u);
            };

            bool ok = warp_wait_all(&bar_res, 0, wd, kSiteBwdMmaKV);
            int committed = 0;
            if (ok && n_it > 0) {
                ok = warp_wait_all(&bar_full[0], 0, wd, kSiteBwdMmaQ);
                if (ok) {
                    tc_fence_after();
                    issue_t(0, 0);
                    mma_commit_w(&bar_t[0]);
                    issue_t(0, 1);
                    mma_commit_w(&bar_t[1]);
                }
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const bool more = it + 1 < n_it;
                for (int h = 0; h < 2; ++h) {
                    if (!warp_wait_all(&bar_e[h], it & 1, wd, kSiteBwdMmaDS)) { ok = false; break; }
                    tc_fence_after();
                    issue_acc(it, h);
                    if (h == 1) {
                        mma_commit_w(&bar_empty[it % C::STAGES]);
                        committed = it + 1;
                    }
                    if (more) {
                        if (h == 0) {
                            const int s1 = (it + 1) % C::STAGES;
                            if (!warp_wait_all(&bar_full[s1], ((it + 1) / C::STAGES) & 1, wd,
                                               kSiteBwdMmaQ)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        // half h of T is free: its readers (issue_acc above) precede in issue order
                        issue_t(it + 1, h);
                        mma_commit_w(&bar_t[h]);
                    }
                }
            }
            if (ok) mma_commit_w(&bar_acc);
            volatile int no_abort = 0;
            const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
            mma_commit_w(&bar_drain);
            mbar_wait(&bar_drain, 0, wd_drain, kSiteBwdDrain);
            for (int it = max(0, committed - C::STAGES); it < committed; ++it)
                mbar_wait(&bar_empty[it % C::STAGES], (it / C::STAGES) & 1, wd_drain, kSiteBwdDrain);
            if (ok) mbar_wait(&bar_acc, 0, wd_drain, kSiteBwdDrain);
        }
    } else {
        // ------------------------------------------------------------- elementwise (warps 0-7)
        const int h = warp >> 2;           // half of the streamed block this warpgroup owns
        const int r = threadIdx.x & 127;   // row of the resident block = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tT1 = tbase + lane_base + 128u * h, tT2 = tT1 + 64u;
        const uint32_t tAcc1 = tbase + lane_base + 256u, tAcc2 = tbase + lane_base + 256u + D;
        const float c2 = p.scale_log2;
        const size_t row_base = static_cast<size_t>(bh) * N;
        const int xrow = x0 + r;
        // dQ kernel: the row statistics of this thread's query row are fixed.
        float L2_self = 0.0f, D_self = 0.0f;
        if (!KV && xrow < N) {
            L2_self = p.lse2[row_base + xrow];
            D_self = p.delta[row_base + xrow];
        }
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int s0 = (s_begin + it) * 128;  // first row of the streamed block
            if (KV) {  // stage L2 / Delta of this half's 64 query rows
                if (r < 64) {  // stored negated, so the pass below is fma / add only
                    const int qi = s0 + 64 * h + r;
                    sL2[h][it & 1][r] = (qi < N) ? -p.lse2[row_base + qi] : -INFINITY;
                    sDl[h][it & 1][r] = (qi < N) ? -p.delta[row_base + qi] : 0.0f;
                }
                named_bar_sync(1 + h, 128);
            }
            if (!warp_wait_all(&bar_t[h], it & 1, wd, kSiteBwdEltS)) { ok = false; break; }
            tc_fence_after();
            // element-wise mask: causal diagonal block, and (dQ kernel) keys beyond N
            const bool diag = p.causal &&
                              causal_tile_class(KV ? s0 : x0, KV ? min(N, s0 + 128) : x1,
                                                KV ? x0 : s0, KV ? x1 : min(N, s0 + 128)) == kTileMasked;
            const bool tail = !KV && (s0 + 128 > N);
            // 64 columns in 4 chunks of 16, software-pipelined: the TMEM load of chunk c+1 is
            // in flight while chunk c is computed and stored.  bf16 results of chunk c go to
            // columns [8c, 8c+8), which chunks 0..c have already loaded.
            const uint64_t c2x2 = f2_make(c2, c2);
            auto chunk = [&](auto mask_tag, int c, const uint32_t* sv, const uint32_t* dpv) {
                constexpr bool MASK = decltype(mask_tag)::value;
                uint32_t pkP[8], pkS[8];
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    float4 nl, nd;
                    if (KV) {  // per-column statistics (negated) for 4 columns
                        nl = *reinterpret_cast<const float4*>(&sL2[h][it & 1][16 * c + e]);
                        nd = *reinterpret_cast<const float4*>(&sDl[h][it & 1][16 * c + e]);
                    } else {   // per-row statistics of this thread's query row
                        nl = make_float4(-L2_self, -L2_self, -L2_self, -L2_self);
                        nd = make_float4(-D_self, -D_self, -D_self, -D_self);
                    }
#pragma unroll
                    for (int u = 0; u < 4; u += 2) {
                        const float nla = u ? nl.z : nl.x, nlb = u ? nl.w : nl.y;
                        const float nda = u ? nd.z : nd.x, ndb = u ? nd.w : nd.y;
                        const uint64_t x2 =
                            f2_fma(f2_make(__uint_as_float(sv[e + u]), __uint_as_float(sv[e + u + 1])),
                                   c2x2, f2_make(nla, nlb));
                        float xa, xb;
                        f2_split(x2, xa, xb);
                        float pa = ex2(xa), pb = ex2(xb);
                        if (MASK) {
                            const int col = 64 * h + 16 * c + e + u;  // streamed row offset
                            const int keya = KV ? xrow : s0 + col, qrya = KV ? s0 + col : xrow;
                            const int keyb = KV ? xrow : s0 + col + 1, qryb = KV ? s0 + col + 1 : xrow;
                            if ((diag && keya > qrya) || (tail && keya >= N)) pa = 0.0f;
                            if ((diag && keyb > qryb) || (tail && keyb >= N)) pb = 0.0f;
                        }
                        const uint64_t t2 = f2_add(
                            f2_make(__uint_as_float(dpv[e + u]), __uint_as_float(dpv[e + u + 1])),
                            f2_make(nda, ndb));
                        float da, db;
                        f2_split(f2_mul(f2_make(pa, pb), t2), da, db);
                        pkP[(e + u) / 2] = pack_bf16x2(pa, pb);
                        pkS[(e + u) / 2] = pack_bf16x2(da, db);
                    }
                }
                if (KV) tmem_st8(tT1 + 8u * c, pkP);
                tmem_st8(tT2 + 8u * c, pkS);
            };
            auto half_pass = [&](auto mask_tag) {
                uint32_t s0v[16], d0v[16], s1v[16], d1v[16];
                tmem_ld16(tT1, s0v);
                tmem_ld16(tT2, d0v);
                tmem_wait_ld();
                reg_fence16(s0v);
                reg_fence16(d0v);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t* cs = (c & 1) ? s1v : s0v;
                    uint32_t* cd = (c & 1) ? d1v : d0v;
                    uint32_t* ns = (c & 1) ? s0v : s1v;
                    uint32_t* nd = (c & 1) ? d0v : d1v;
                    if (c + 1 < 4) {
                        tmem_ld16(tT1 + 16u * (c + 1), ns);
                        tmem_ld16(tT2 + 16u * (c + 1), nd);
                    }
                    chunk(mask_tag, c, cs, cd);
                    if (c + 1 < 4) {
                        tmem_wait_ld();
                        reg_fence16(ns);
                        reg_fence16(nd);
                    }
                }
            };
            if (diag || tail)
                half_pass(std::true_type{});
            else
                half_pass(std::false_type{});
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_e[h]);
        }
        // ------------------------------------------------------------- epilogue
        // Warpgroup h stores accumulator columns [h*D/2, (h+1)*D/2) of its rows.
        if (ok && n_it > 0 && warp_wait_all(&bar_acc, 0, wd, kSiteBwdEltAcc)) {
            tc_fence_after();
            __nv_bfloat16* out2 = static_cast<__nv_bfloat16*>(KV ? p.dk : p.dq);
            __nv_bfloat16* out1 = static_cast<__nv_bfloat16*>(p.dv);
#pragma unroll 1
            for (int which = KV ? 0 : 1; which < 2; ++which) {
                const uint32_t tAcc = which == 0 ? tAcc1 : tAcc2;
                const float mul = which == 0 ? 1.0f : p.scale;
                __nv_bfloat16* dst_row = (which == 0 ? out1 : out2) + (row_base + xrow) * D;
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
                    if (xrow < N) {
                        uint4* dst = reinterpret_cast<uint4*>(dst_row + c0);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                                packed[4 * c + 3]);
                    }
                }
            }
        } else if (n_it == 0 && xrow < N) {
            // a block that no streamed block touches has zero gradient (cannot occur for
            // square causal attention, kept for completeness)
            __nv_bfloat16* out2 = static_cast<__nv_bfloat16*>(KV ? p.dk : p.dq);
            for (int c = h * (D / 2); c < (h + 1) * (D / 2); ++c) {
                out2[(row_base + xrow) * D + c] = __float2bfloat16_rn(0.0f);
                if (KV) static_cast<__nv_bfloat16*>(p.dv)[(row_base + xrow) * D + c] = __float2bfloat16_rn(0.0f);
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

template <int D, bool KV>
static cudaError_t launch_one(const CUtensorMap& x, const CUtensorMap& y, const CUtensorMap& a,
                              const CUtensorMap& b, const BwdParams& p, cudaStream_t st)
{
    using C = BwdCfg<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fa_bwd_tc_kernel<D, KV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid(p.BH * ((p.N + 127) / 128));
    fa_bwd_tc_kernel<D, KV><<<grid, C::THREADS, C::SMEM_BYTES, st>>>(x, y, a, b, p);
    return cudaGetLastError();
}

// maps: [0] q, [1] k, [2] v, [3] dout (bf16, 128-row boxes)
cudaError_t launch_bwd_tc_stage(int d, int stage, const CUtensorMap* maps, const BwdParams& p,
                                cudaStream_t st)
{
    const CUtensorMap &q = maps[0], &k = maps[1], &v = maps[2], &g = maps[3];
    if (stage == 1)
        return d == 64 ? launch_one<64, true>(k, v, q, g, p, st) : launch_one<128, true>(k, v, q, g, p, st);
    return d == 64 ? launch_one<64, false>(q, g, k, v, p, st) : launch_one<128, false>(q, g, k, v, p, st);
}

cudaError_t launch_bwd_tc(int d, const CUtensorMap* maps, const BwdParams& p, cudaStream_t st)
{
    cudaError_t e = launch_bwd_tc_stage(d, 1, maps, p, st);
    if (e != cudaSuccess) return e;
    return launch_bwd_tc_stage(d, 2, maps, p, st);
}

}  // namespace fa
