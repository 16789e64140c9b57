// Split-KV decode attention on sm_103a tensor cores, for few queries per sequence over a long
// key/value history with grouped key/value heads.  "서빙에서 Flash Attention 이득이 예상보다 작은
// 경우" of "Flash Attention IO-awareness principle" notes that decoding with GQA leaves the
// per-head tiles of the prefill kernel too few to fill the GPU and points to decoding kernels
// (FlashDecoding) instead; this is that layout of the same exact computation:
//   - the query rows of one (sequence, key/value head) pair, G = H / Hkv heads x nq queries
//     (row r = i * G + g), share one 128-row tile, so the group reads its K and V once;
//   - the sequence's key blocks are split into `splits` contiguous ranges, one CTA each, so
//     B * Hkv * splits CTAs stream the key/value history in parallel;
//   - each range keeps the online softmax of the "Tiling" section (running max, rescaled sum)
//     and, with splits > 1, writes its O normalised by its own weights and its log-sum-exp;
//     fa_decode_combine_kernel merges the ranges with the same rescaling rule
//     (O = sum_s e^{lse_s} O_s / sum_s e^{lse_s}, lse = log sum_s e^{lse_s}).
// Roles (6 warps): warps 0-3 softmax (thread = tile row = TMEM lane), warp 4 TMA producer,
// warp 5 TMEM allocator and MMA issuer.  TMEM: two S buffers [0,128), [128,256) so S of block
// j+1 is computed while the softmax works on block j (P of a block, bf16 pairs, overwrites the
// upper half of its S buffer), O at [256, 256+d).
#include "fa_decode.cuh"
#include "tc_ptx.cuh"

namespace fa {

template <int D>
struct DecCfg {
    static constexpr int BN = 128;                 // keys per block
    static constexpr int PANELS = D / 64;          // 128-byte swizzle panels per row
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
    static constexpr int STAGES = (D == 128) ? 3 : 6;
    static constexpr int SMEM_BYTES = TILE_BYTES + 2 * STAGES * TILE_BYTES + 1024;
    static constexpr int THREADS = 192;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units, as in the forward kernel
};

// S = Q K^T over D/16 k-steps (both operands K-major in 128B-swizzled panels).
template <int D, int PANEL>
__device__ __forceinline__ void dec_issue_qk(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc,
                                             uint32_t idesc)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks / 4) * PANEL + (ks % 4) * 32;
        mma_ss_w(d_tmem, sdesc_adv(qdesc, off), sdesc_adv(kdesc, off), idesc, ks > 0 ? 1u : 0u);
    }
}

// O += P V: P (bf16 pairs) from TMEM, V (MN-major) from shared memory; 8 k-steps of 16 keys.
__device__ __forceinline__ void dec_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc,
                                             uint32_t idesc, uint32_t acc_first)
{
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        mma_ts_w(d_tmem, p_tmem + 8u * ks, sdesc_adv(vdesc, ks * 2048), idesc,
                 ks > 0 ? 1u : acc_first);
}

template <int D>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const DecodeParams p)
{
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + C::TILE_BYTES;
    uint8_t* sV = sK + C::STAGES * C::TILE_BYTES;

    __shared__ __align__(8) uint64_t bar_q;
    __shared__ __align__(8) uint64_t bar_kfull[C::STAGES];
    __shared__ __align__(8) uint64_t bar_vfull[C::STAGES];
    __shared__ __align__(8) uint64_t bar_kempty[C::STAGES];
    __shared__ __align__(8) uint64_t bar_vempty[C::STAGES];
    __shared__ __align__(8) uint64_t bar_sfull[2];  // S of a block landed in buffer b
    __shared__ __align__(8) uint64_t bar_pfull;     // softmax wrote P (and rescaled O)
    __shared__ __align__(8) uint64_t bar_pv;        // the P V product of a block has run
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout& L = p.L;
    const int split = static_cast<int>(blockIdx.x) % p.splits;
    const int rest = static_cast<int>(blockIdx.x) / p.splits;
    const int chunk = rest % p.head_chunks, bkv = rest / p.head_chunks;
    const int b = bkv / L.Hkv, hk = bkv % L.Hkv;
    const int h0 = hk * (L.H / L.Hkv) + chunk * p.G;  // first query head of this CTA
    const int G = p.G;

    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&bar_kfull[s], 1);
            mbar_init(&bar_vfull[s], 1);
            mbar_init(&bar_kempty[s], 1);
            mbar_init(&bar_vempty[s], 1);
        }
        mbar_init(&bar_sfull[0], 1);
        mbar_init(&bar_sfull[1], 1);
        mbar_init(&bar_pfull, 4);  // one elected arrive per softmax warp
        mbar_init(&bar_pv, 1);
        mbar_init(&bar_drain, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(&tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    const Watchdog wd{&abort_flag, p.status, p.wait_limit_ns};
    // This grid is launched as a programmatic dependent of the work before it on the stream, so
    // its set-up above (which touches no global memory) overlaps that work's end; every input,
    // the sequence starts included, is read only after that work has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const SeqRows sr = seq_rows<true>(L, b);
    const int nq = min(sr.nq, p.q_box), nk = sr.nk;
    const int shift = nk - nq;  // bottom-right causal alignment
    // This CTA's key blocks [jb, jb + J): a balanced share of all blocks of the sequence (the
    // last query sees every key, so under the causal mask too every block is needed).  A
    // sequence without queries streams nothing and stores nothing.
    const int nkb = (nk + C::BN - 1) / C::BN;
    const int jb = static_cast<int>((static_cast<long long>(nkb) * split) / p.splits);
    const int J = nq == 0 ? 0
                          : static_cast<int>((static_cast<long long>(nkb) * (split + 1)) / p.splits) - jb;
    // The combine kernel may be scheduled now (programmatic dependent launch); it waits for
    // this whole grid to finish before it reads the partial results.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 4) {
        // ------------------------------------------------------------- TMA producer
        // Q: one 3-D box of (64 columns, G heads, q_box tokens) per panel, rows in (token, head)
        // order; the rows of the tile past G * q_box are never written and never stored.
        const uint32_t q_bytes = static_cast<uint32_t>(C::PANELS * 128 * G * p.q_box);
        mbar_arrive_expect_tx_w(&bar_q, q_bytes);
        for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_3d_w(sQ + pn * C::PANEL_BYTES, &tm_q, &bar_q, 64 * pn, h0, sr.q0);
        int issued = 0;
        for (int jj = 0; jj < J; ++jj) {
            const int s = jj % C::STAGES;
            const uint32_t ph = (jj / C::STAGES) & 1;
            const int row = sr.k0 + (jb + jj) * C::BN;
            if (!warp_wait_all(&bar_kempty[s], ph ^ 1, wd, kSiteFwdLoadEmpty)) break;
            mbar_arrive_expect_tx_w(&bar_kfull[s], C::TILE_BYTES);
            for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_3d_w(sK + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_k, &bar_kfull[s],
                              64 * pn, hk, row);
            if (!warp_wait_all(&bar_vempty[s], ph ^ 1, wd, kSiteFwdLoadEmpty)) break;
            mbar_arrive_expect_tx_w(&bar_vfull[s], C::TILE_BYTES);
            if (!(jj == 0 && (p.debug_flags & kDebugDropFirstLoad)))
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_3d_w(sV + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_v,
                                  &bar_vfull[s], 64 * pn, hk, row);
            issued = jj + 1;
        }
        // no copy may land after the CTA exits (bounded waits that ignore the abort flag)
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        mbar_wait(&bar_q, 0, wd_drain, kSiteFwdDrain);
        for (int jj = max(0, issued - C::STAGES); jj < issued; ++jj) {
            const int s = jj % C::STAGES;
            const uint32_t ph = (jj / C::STAGES) & 1;
            mbar_wait(&bar_kfull[s], ph, wd_drain, kSiteFwdDrain);
            mbar_wait(&bar_vfull[s], ph, wd_drain, kSiteFwdDrain);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------- MMA issuer
        // Per block jj: S(jj+1) into the other buffer as soon as K(jj+1) is in (the buffer held
        // P(jj-1), whose P V product was issued before, and MMAs run in issue order), then
        // P V of block jj once the softmax has written P(jj).
        constexpr uint32_t kIdS = idesc_bf16_f32(128, C::BN, 0, 0);  // S = Q K^T
        constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);     // O += P V
        const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv0 = sdesc_sw128(smem_u32(sV), C::PANEL_BYTES, 1024);
        const uint32_t tO = tbase + 256u;
        bool ok = J > 0 && warp_wait_all(&bar_q, 0, wd, kSiteFwdMmaQ);
        ok = ok && warp_wait_all(&bar_kfull[0], 0, wd, kSiteFwdMmaK);
        int committed_k = 0, committed_v = 0;
        if (ok) {
            tc_fence_after();
            dec_issue_qk<D, C::PANEL_BYTES>(tbase, dq0, dk0, kIdS);
            mma_commit_w(&bar_sfull[0]);
            mma_commit_w(&bar_kempty[0]);
            committed_k = 1;
        }
        for (int jj = 0; ok && jj < J; ++jj) {
            const int s = jj % C::STAGES;
            if (jj + 1 < J) {
                const int s1 = (jj + 1) % C::STAGES;
                if (!warp_wait_all(&bar_kfull[s1], ((jj + 1) / C::STAGES) & 1, wd, kSiteFwdMmaK)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                dec_issue_qk<D, C::PANEL_BYTES>(tbase + 128u * ((jj + 1) & 1), dq0,
                                                sdesc_adv(dk0, s1 * C::TILE_BYTES), kIdS);
                mma_commit_w(&bar_sfull[(jj + 1) & 1]);
                mma_commit_w(&bar_kempty[s1]);
                committed_k = jj + 2;
            }
            if (!warp_wait_all(&bar_pfull, jj & 1, wd, kSiteFwdMmaP)) { ok = false; break; }
            if (!warp_wait_all(&bar_vfull[s], (jj / C::STAGES) & 1, wd, kSiteFwdMmaV)) {
                ok = false;
                break;
            }
            tc_fence_after();
            dec_issue_pv(tO, tbase + 128u * (jj & 1) + 64u, sdesc_adv(dv0, s * C::TILE_BYTES),
                         kIdPV, jj > 0 ? 1u : 0u);
            mma_commit_w(&bar_pv);
            mma_commit_w(&bar_vempty[s]);
            committed_v = jj + 1;
        }
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        mma_commit_w(&bar_drain);
        mbar_wait(&bar_drain, 0, wd_drain, kSiteFwdDrain);
        for (int jj = max(0, committed_k - C::STAGES); jj < committed_k; ++jj)
            mbar_wait(&bar_kempty[jj % C::STAGES], (jj / C::STAGES) & 1, wd_drain, kSiteFwdDrain);
        for (int jj = max(0, committed_v - C::STAGES); jj < committed_v; ++jj)
            mbar_wait(&bar_vempty[jj % C::STAGES], (jj / C::STAGES) & 1, wd_drain, kSiteFwdDrain);
    } else {
        // ------------------------------------------------------------- softmax (warps 0-3)
        const int r = threadIdx.x;  // tile row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tbase + lane_base + 256u;
        const int i = r / G;  // query of this row within the sequence (head h0 + r % G)
        // x = S * c with c = scale * log2(e); for c <= 0 the scores are scaled first so that
        // masked entries stay -inf (as in the forward kernel).
        const float c2 = p.scale_log2;
        const bool prescale = !(c2 > 0.0f);
        const float cf = prescale ? 1.0f : c2;
        // Key blocks from jmask on need the element-wise mask (the causal edge, the ragged last
        // block); this row sees the keys [0, klim] of the sequence.
        int jmask = nk / C::BN;
        int klim = nk - 1;
        if (p.causal) {
            const int e = shift + 1;
            jmask = min(jmask, e > 0 ? e / C::BN : 0);
            klim = min(klim, i + shift);
        }
        float m = -INFINITY, l = 0.0f, lr = 0.0f;
        bool ok = true;
        for (int jj = 0; ok && jj < J; ++jj) {
            const int j = jb + jj;
            const uint32_t tS = tbase + lane_base + 128u * (jj & 1);
            if (!warp_wait_all(&bar_sfull[jj & 1], (jj >> 1) & 1, wd, kSiteFwdSoftmaxS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr32[128];
            tmem_ld32(tS + 0, sr32);
            tmem_ld32(tS + 32, sr32 + 32);
            tmem_ld32(tS + 64, sr32 + 64);
            tmem_ld32(tS + 96, sr32 + 96);
            tmem_wait_ld();
            reg_fence32(sr32);
            reg_fence32(sr32 + 32);
            reg_fence32(sr32 + 64);
            reg_fence32(sr32 + 96);
            float x[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr32[c]);
            if (prescale) {
#pragma unroll
                for (int c = 0; c < 128; ++c) x[c] *= c2;
            }
            if (j >= jmask) {
                const int lim = klim - j * C::BN;  // last visible key column in this block
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > lim) x[c] = -INFINITY;
            }
            float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
            for (int c = 4; c < 124; c += 8) {
                mx0 = fmax3(mx0, x[c], x[c + 1]);
                mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
                mx2 = fmax3(mx2, x[c + 4], x[c + 5]);
                mx3 = fmax3(mx3, x[c + 6], x[c + 7]);
            }
            mx0 = fmax3(mx0, x[124], x[125]);
            mx1 = fmax3(mx1, x[126], x[127]);
            const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cf;
            // rescale only when the max grew by more than the threshold (exact either way)
            float alpha = 1.0f;
            const bool need = mt > m + C::RESCALE_THRESHOLD;
            if (need) {
                alpha = ex2(m - mt);
                m = mt;
                l *= alpha;
                lr *= alpha;
            }
            const float neg_m = (m == -INFINITY) ? 0.0f : -m;
            const uint64_t cf2 = f2_make(cf, cf), nm2 = f2_make(neg_m, neg_m);
            uint64_t lsa = f2_make(0.f, 0.f), lsb = lsa, lra = lsa, lrb = lsa;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const int e = cb * 32 + c;
                    float p0, p1, p2, p3;
                    f2_split(f2_fma(f2_make(x[e], x[e + 1]), cf2, nm2), p0, p1);
                    f2_split(f2_fma(f2_make(x[e + 2], x[e + 3]), cf2, nm2), p2, p3);
                    p0 = ex2(p0);
                    p1 = ex2(p1);
                    p2 = ex2(p2);
                    p3 = ex2(p3);
                    const uint32_t w01 = pack_bf16x2(p0, p1);
                    const uint32_t w23 = pack_bf16x2(p2, p3);
                    lsa = f2_add(lsa, f2_make(p0, p1));
                    lsb = f2_add(lsb, f2_make(p2, p3));
                    // lr sums the bf16-rounded weights the P V product uses
                    lra = f2_add(lra, f2_make(__uint_as_float(w01 << 16),
                                              __uint_as_float(w01 & 0xFFFF0000u)));
                    lrb = f2_add(lrb, f2_make(__uint_as_float(w23 << 16),
                                              __uint_as_float(w23 & 0xFFFF0000u)));
                    pk[c / 2] = w01;
                    pk[c / 2 + 1] = w23;
                }
                tmem_st16(tS + 64u + 16u * cb, pk);
            }
            {
                float a0, a1, b0, b1;
                f2_split(f2_add(lsa, lsb), a0, a1);
                f2_split(f2_add(lra, lrb), b0, b1);
                l += a0 + a1;
                lr += b0 + b1;
            }
            // O holds blocks < jj once the P V product of block jj - 1 has run
            if (jj > 0) {
                if (!warp_wait_all(&bar_pv, (jj - 1) & 1, wd, kSiteFwdSoftmaxO)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32u * ch, o);
                        tmem_wait_ld();
                        reg_fence32(o);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(tO + 32u * ch, o);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_pfull);
        }
        // ------------------------------------------------------------- epilogue
        // Row r holds query i of head h0 + g.  With one split this is the final result;
        // with several, the range's O normalised by its own weights and its natural-log LSE.
        // A row that sees no key of the range (or a range without blocks) gives O = 0 and
        // lse = -inf, which the combine step weighs with e^{-inf} = 0.
        bool have = ok && J > 0;
        if (have) have = warp_wait_all(&bar_pv, (J - 1) & 1, wd, kSiteFwdSoftmaxO);
        if (have) tc_fence_after();
        const bool valid = r < G * nq;
        const int g = r - i * G;
        const size_t t = static_cast<size_t>(sr.q0) + i;  // token row of the packed tensors
        const int h = h0 + g;
        const float inv_l = lr > 0.0f ? 1.0f / lr : 0.0f;
        const float lse_row = (have && l > 0.0f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
        const size_t o_off = t * L.o_rs + static_cast<size_t>(h) * L.o_hs;
        const size_t part_off = ((static_cast<size_t>(split) * L.Rq + t) * L.H + h) * D;
        const size_t lse_off = static_cast<size_t>(h) * L.Rq + t;
        const size_t lsep_off = (static_cast<size_t>(split) * L.H + h) * L.Rq + t;
        const bool o_in = !valid || (p.splits == 1 ? in_extent(o_off, D, L.o_ext, p.status)
                                                   : in_extent(part_off, D, p.part_ext, p.status));
        const bool lse_in = !valid || (p.splits == 1
                                           ? p.lse == nullptr || in_extent(lse_off, 1, L.stat_ext, p.status)
                                           : in_extent(lsep_off, 1, p.part_ext / D, p.status));
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tO + 32u * ch, o);
                tmem_wait_ld();
                reg_fence32(o);
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = 0u;
            }
            if (!valid || !o_in) continue;
            if (p.splits == 1) {
                uint32_t packed[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    packed[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                            __uint_as_float(o[2 * c + 1]) * inv_l);
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + o_off + 32 * ch);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                        packed[4 * c + 3]);
            } else {
                float4* dst = reinterpret_cast<float4*>(p.o_part + part_off + 32 * ch);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_float4(__uint_as_float(o[4 * c]) * inv_l,
                                         __uint_as_float(o[4 * c + 1]) * inv_l,
                                         __uint_as_float(o[4 * c + 2]) * inv_l,
                                         __uint_as_float(o[4 * c + 3]) * inv_l);
            }
        }
        if (valid && lse_in) {
            if (p.splits == 1) {
                if (p.lse != nullptr) p.lse[lse_off] = lse_row;
            } else {
                p.lse_part[lsep_off] = lse_row;
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

// Merge of the split ranges of every (token, head) row: one warp per row, each lane owning
// d / 32 columns.  With M = max_s lse_s and w_s = e^{lse_s - M}:
//   O = sum_s w_s O_s / sum_s w_s,   lse = M + log sum_s w_s;
// a row whose ranges all saw no key (M = -inf) gets O = 0 and lse = -inf.  The ranges go in
// batches of SB (2, 4 or 8, the smallest that holds all ranges, else 8) whose LSE and
// partial-O loads are all issued before any is used (one memory round trip per batch);
// batches merge by the same rule, the running sums rescaled to the running max.
template <int D, int SB>
__global__ void __launch_bounds__(256) fa_decode_combine_kernel(const DecodeParams p)
{
    constexpr int EPL = D / 32;  // columns per lane
    // launched as a programmatic dependent of the split kernel: wait until that grid has
    // completed and its partial results are visible; the next decode step's split grid may then
    // be scheduled (it waits for this grid before reading anything)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const Layout& L = p.L;
    const size_t rows = static_cast<size_t>(L.Rq) * L.H;
    const int lane = threadIdx.x & 31;
    const size_t warps_total = static_cast<size_t>(gridDim.x) * (blockDim.x / 32);
    for (size_t row = static_cast<size_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
         row < rows; row += warps_total) {
        const size_t t = row / L.H;
        const int h = static_cast<int>(row - t * L.H);
        float mx = -INFINITY, wsum = 0.0f;
        float acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.0f;
        for (int s0 = 0; s0 < p.splits; s0 += SB) {
            float ls[SB];
            float v[SB][EPL];
#pragma unroll
            for (int k = 0; k < SB; ++k) {
                const int s = s0 + k;
                ls[k] = -INFINITY;
#pragma unroll
                for (int e = 0; e < EPL; ++e) v[k][e] = 0.0f;
                if (s < p.splits) {
                    ls[k] = p.lse_part[(static_cast<size_t>(s) * L.H + h) * L.Rq + t];
                    const float* src =
                        p.o_part + ((static_cast<size_t>(s) * L.Rq + t) * L.H + h) * D + lane * EPL;
                    if constexpr (EPL == 4) {
                        const float4 x = *reinterpret_cast<const float4*>(src);
                        v[k][0] = x.x; v[k][1] = x.y; v[k][2] = x.z; v[k][3] = x.w;
                    } else {
                        const float2 x = *reinterpret_cast<const float2*>(src);
                        v[k][0] = x.x; v[k][1] = x.y;
                    }
                }
            }
            float bm = mx;
#pragma unroll
            for (int k = 0; k < SB; ++k) bm = fmaxf(bm, ls[k]);
            if (bm == -INFINITY) continue;  // no range so far saw a key (the same for the warp)
            const float rs = (mx == -INFINITY) ? 0.0f : expf(mx - bm);  // rescale the running sums
            wsum *= rs;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] *= rs;
#pragma unroll
            for (int k = 0; k < SB; ++k) {
                const float w = (ls[k] == -INFINITY) ? 0.0f : expf(ls[k] - bm);
                wsum += w;
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, v[k][e], acc[e]);
            }
            mx = bm;
        }
        const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
        const size_t o_off = t * L.o_rs + static_cast<size_t>(h) * L.o_hs;
        if (!in_extent(o_off, D, L.o_ext, p.status)) continue;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + o_off + lane * EPL;
        if constexpr (EPL == 4) {
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
        if (lane == 0 && p.lse != nullptr)
            p.lse[static_cast<size_t>(h) * L.Rq + t] = (mx == -INFINITY) ? -INFINITY : mx + logf(wsum);
    }
}

template <int D>
static cudaError_t launch_decode_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const DecodeParams& p,
                                      cudaStream_t st, int num_sms)
{
    using C = DecCfg<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fa_decode_split_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid(p.L.B * p.L.Hkv * p.head_chunks * p.splits);
    {
        // programmatic dependent launch: the split grid's set-up overlaps the end of the work
        // before it on the stream
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, fa_decode_split_kernel<D>, tq, tk, tv, p);
        if (e != cudaSuccess || p.splits == 1) return e;
    }
    const long rows = static_cast<long>(p.L.Rq) * p.L.H;
    long blocks = (rows + 7) / 8;  // 8 warps (rows) per CTA
    const long cap = static_cast<long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    // programmatic dependent launch: the combine grid's launch overlaps the split grid's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.splits <= 2) return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, 2>, p);
    if (p.splits <= 4) return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, 4>, p);
    return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, 8>, p);
}

cudaError_t launch_decode(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const DecodeParams& p, cudaStream_t st,
                          int num_sms)
{
    if (d == 64) return launch_decode_impl<64>(tq, tk, tv, p, st, num_sms);
    return launch_decode_impl<128>(tq, tk, tv, p, st, num_sms);
}

}  // namespace fa
