// Forward attention on sm_103a tensor cores: TMA-staged Q/K/V tiles, tcgen05.mma into
// Tensor Memory, warp-specialised producer / MMA / softmax roles, online softmax in fp32
// with exp2, un-scaled accumulation and one final 1/l, causal two-stage split, ragged tails.
//
// One CTA owns NT = 2 query tiles of 128 rows of one head (the FlashAttention-2 Q-outer
// loop order, "FA2·FA3" section of "Flash Attention IO-awareness principle") and streams
// the key/value blocks of 128 keys through shared-memory rings (K and V stages are released
// separately: K(j) after the S products of block j, V(j) after its P V products, so the copy
// of K(j+2) starts a block and a half before its first use).  Roles (10 warps):
//   warps 0-3   softmax of query tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax of query tile 1
//   warp  8     TMA producer (whole warp, one elected lane issues)
//   warp  9     TMEM allocator + MMA issuer (whole warp, one elected lane issues)
// TMEM columns: S_t at [128t, 128t+128) (fp32), P_t (bf16 pairs) aliased on the upper half
// of S_t, O_t at [256 + t*d, 256 + (t+1)*d) (fp32, un-normalised); at d = 64, O_t at
// [256 + 128t, 384 + 128t), whose column 64 accumulates the row sum of the bf16 P (the P V
// product runs at N = 80 against V and a constant ones-column panel).  At d = 64 and for
// e4m3 the softmax warps signal P in two halves of 64 keys and the MMA warp issues each half
// of the P V product as soon as it has landed (FwdCfg::SPLIT_P).
//
// The e4m3 variant (F8, d = 128; fixed-length square heads or packed batches) runs the same
// schedule on 8-bit operands with kind::f8f6f4 MMAs (K = 32 per MMA): Q and K tiles of 128
// rows x 128 bytes, P rounded to e4m3 (four per TMEM column, at columns [64, 96) of S_t),
// and V read from a transposed copy V^T [d, keys] per (sequence, key/value head) so that
// both operands of O += P V are K-major.  The
// descale factors of Q and K are folded into the softmax scale on the host; V's is applied
// with 1/l in the epilogue.  O is normalised by the fp32 row sum l.
#include <type_traits>

#include "fa_common.cuh"
#include "tc_ptx.cuh"

namespace fa {

template <int D, bool F8 = false>
struct FwdCfg {
    static constexpr int BM = 128;                 // query rows per tile
    static constexpr int NT = 2;                   // query tiles per CTA
    static constexpr int BN = 128;                 // keys per block
    static constexpr int ELEM = F8 ? 1 : 2;        // bytes per operand element
    static constexpr int PANEL_ELEMS = 128 / ELEM; // elements in one 128-byte panel row
    static constexpr int PANELS = D / PANEL_ELEMS; // 128-byte swizzle panels per row
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
    static constexpr int KSTEPS_QK = D * ELEM / 32;   // MMAs per S product (32 bytes of K each)
    static constexpr int KSTEPS_PV = BN * ELEM / 32;  // MMAs per P V product
    static constexpr int STAGES = (D == 128 && !F8) ? 2 : 4;
    static constexpr int SMEM_Q = NT * TILE_BYTES;
    static constexpr int SMEM_K = STAGES * TILE_BYTES;
    static constexpr int SMEM_V = STAGES * TILE_BYTES;
    // d = 64: the P V product runs at N = 80 against V and the first 16 columns of a constant
    // panel whose first column is 1.0, so O's column 64 accumulates the sum of the bf16 P
    // weights on the tensor core (the row sum that normalises O), instead of ~190 softmax
    // instructions per row and block.
    static constexpr bool SUM_ON_MMA = (D == 64 && !F8);
    static constexpr int O_COLS = SUM_ON_MMA ? 128 : D;  // TMEM columns of one O accumulator
    static constexpr int SMEM_ONES = SUM_ON_MMA ? PANEL_BYTES : 0;
    static constexpr int SMEM_BYTES = SMEM_Q + SMEM_K + SMEM_V + SMEM_ONES + 1024;  // + slack
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units: P stays below 2^8
    // P is signalled to the MMA warp in two halves of 64 keys, so that the P V product starts
    // on the first half while the second is computed.  Measured on GB300: 5 % faster at d = 64
    // and 2.4 % for e4m3, but 11 % slower for the bf16 forward at d = 128, which therefore
    // signals the whole of P at once.
    static constexpr bool SPLIT_P = (D == 64) || F8;
};

// S = Q K^T for one 128-row query tile: KSTEPS k-steps of 32 bytes of d (16 bf16 or 32 e4m3
// elements), the first overwriting D.  Executed by the whole MMA warp; one elected lane
// issues each MMA.
template <int KSTEPS, int PANEL, bool F8>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc,
                                         uint32_t idesc)
{
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        const uint32_t off = (ks / 4) * PANEL + (ks % 4) * 32;
        if constexpr (F8)
            mma_ss_w_f8(d_tmem, sdesc_adv(qdesc, off), sdesc_adv(kdesc, off), idesc, ks > 0 ? 1u : 0u);
        else
            mma_ss_w(d_tmem, sdesc_adv(qdesc, off), sdesc_adv(kdesc, off), idesc, ks > 0 ? 1u : 0u);
    }
}

// O += P V over k-steps [KS0, KS1): P from TMEM (8 columns = 32 bytes of keys per k-step), V
// from shared memory: bf16 V is MN-major (a k-step of 16 keys is 16 rows = 2048 bytes
// further), e4m3 V^T is K-major (a k-step of 32 keys is 32 bytes further along its rows).
template <int KS0, int KS1, bool F8>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc,
                                         uint32_t idesc, uint32_t acc_first)
{
#pragma unroll
    for (int ks = KS0; ks < KS1; ++ks) {
        if constexpr (F8)
            mma_ts_w_f8(d_tmem, p_tmem + 8u * ks, sdesc_adv(vdesc, ks * 32), idesc,
                        ks > 0 ? 1u : acc_first);
        else
            mma_ts_w(d_tmem, p_tmem + 8u * ks, sdesc_adv(vdesc, ks * 2048), idesc,
                     ks > 0 ? 1u : acc_first);
    }
}

// One work tile: the NT = 2 query tiles qt0, qt0 + 1 of (sequence b, query head h), for tile
// index `id` of the launch grid, in the order of tile_order: within a head the last pairs (most
// key blocks under the causal mask) rank first.
struct FwdTile {
    SeqRows sr;
    int b;
    int qt0, nt;       // first query tile and query tiles in the pair (1 or 2)
    int qhead, khead;  // head indices of the query-side and key-side tensors
    int vthead;        // e4m3: the V^T matrix of this (sequence, key/value head)
    int shift;         // bottom-right causal alignment (nk - nq), 0 in the square layout
    int J[2];          // key blocks visited by each query tile: a prefix 0 .. J[t] - 1
    int Jmax;
    bool valid;        // the pair holds at least one query of its sequence
};

template <int MODE, int BM, int BN, int NT>
__device__ __forceinline__ FwdTile fwd_tile(const FwdParams& p, int id)
{
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);
    constexpr bool general = mode_general(MODE);
    const int n_pairs = ((L.Nq + BM - 1) / BM + NT - 1) / NT;
    int bhead, rank;
    tile_order(id, L.B * L.H, n_pairs, L.order_group, bhead, rank);
    const int h = bhead % L.H;
    FwdTile t;
    t.b = bhead / L.H;
    t.sr = seq_rows<packed>(L, t.b);
    const int nq = t.sr.nq, nk = t.sr.nk;
    const int n_qtiles = (nq + BM - 1) / BM;
    const int n_kblocks = (nk + BN - 1) / BN;
    t.qt0 = (n_pairs - 1 - rank) * NT;
    t.valid = t.qt0 < n_qtiles;
    t.nt = t.valid ? min(NT, n_qtiles - t.qt0) : 0;
    t.qhead = q_head_index<packed>(L, t.b, h);
    const int hk = general ? h / (L.H / L.Hkv) : h;
    t.khead = k_head_index<packed>(L, t.b, hk);
    t.vthead = t.b * L.Hkv + hk;
    t.shift = general ? nk - nq : 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        t.J[q] = 0;
        if (q < t.nt) {
            if (!p.causal) {
                t.J[q] = n_kblocks;
            } else {
                const int q1 = min(nq, (t.qt0 + q + 1) * BM);
                const int kend = min(nk, q1 + t.shift);  // keys [0, kend) are seen by some row
                t.J[q] = kend > 0 ? (kend + BN - 1) / BN : 0;
            }
        }
    }
    t.Jmax = max(t.J[0], t.J[1]);
    return t;
}

template <int D, int MODE, bool F8>
__global__ void __launch_bounds__(FwdCfg<D, F8>::THREADS, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p)
{
    using C = FwdCfg<D, F8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + C::SMEM_Q;
    uint8_t* sV = sK + C::SMEM_K;
    uint8_t* sOnes = sV + C::SMEM_V;  // d = 64 only: the constant column panel

    __shared__ __align__(8) uint64_t bar_q;      // the Q tiles of a pair landed
    __shared__ __align__(8) uint64_t bar_qfree;  // every S product of a pair has run
    __shared__ __align__(8) uint64_t bar_kfull[C::STAGES];
    __shared__ __align__(8) uint64_t bar_vfull[C::STAGES];
    __shared__ __align__(8) uint64_t bar_kempty[C::STAGES];  // K of a block no longer read
    __shared__ __align__(8) uint64_t bar_vempty[C::STAGES];  // V of a block no longer read
    __shared__ __align__(8) uint64_t bar_sfull[C::NT];
    // half x of P_t written ([t][1] alone, for the whole of P, when P is not split)
    __shared__ __align__(8) uint64_t bar_pfull[C::NT][2];
    __shared__ __align__(8) uint64_t bar_ofinal[C::NT];
    __shared__ __align__(8) uint64_t bar_drain;
    // Tile queue: the producer warp takes further tiles from the launch grid by cluster launch
    // control and publishes their indices (-1: none left) in a two-slot queue.
    __shared__ __align__(16) __int128 clc_resp;
    __shared__ __align__(8) uint64_t bar_clc;        // cancellation response landed
    __shared__ __align__(8) uint64_t bar_tfull[2];   // tile index published
    __shared__ __align__(8) uint64_t bar_tempty[2];  // tile index read by every other warp
    __shared__ int tile_ids[2];
    // Per softmax warp, the state that only tile boundaries use (tile index, ordinal, S products
    // of its slot so far, finished pairs of its slot), kept out of the registers that the
    // softmax loop needs.
    __shared__ int sm_state[8][4];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout& L = p.L;
    constexpr bool packed = mode_packed(MODE);  // tensors stored token by token
    auto tile_of = [&](int id) { return fwd_tile<MODE, C::BM, C::BN, C::NT>(p, id); };

    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 1);
        mbar_init(&bar_qfree, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&bar_kfull[s], 1);
            mbar_init(&bar_vfull[s], 1);
            mbar_init(&bar_kempty[s], 1);
            mbar_init(&bar_vempty[s], 1);
        }
        for (int t = 0; t < C::NT; ++t) {
            mbar_init(&bar_sfull[t], 1);
            mbar_init(&bar_pfull[t][0], 4);  // one elected arrive per softmax warp
            mbar_init(&bar_pfull[t][1], 4);
            mbar_init(&bar_ofinal[t], 1);
        }
        mbar_init(&bar_drain, 1);
        mbar_init(&bar_clc, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_tfull[s], 1);
            mbar_init(&bar_tempty[s], 9);  // the eight softmax warps and the MMA warp
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (C::SUM_ON_MMA) {
        // 128 key rows x 64 bf16 columns, 128-byte swizzled like a TMA-written MN-major tile:
        // column 0 of key row r sits in 16-byte chunk (0 ^ r % 8) of the row.  Written by the
        // 256 softmax threads, then made visible to the tensor core (async proxy).
        if (warp < 8) {
            uint4* dst = reinterpret_cast<uint4*>(sOnes);
            for (int i = threadIdx.x; i < C::PANEL_BYTES / 16; i += 256) {
                const int row = i >> 3, chunk = i & 7;
                dst[i] = make_uint4(chunk == (row & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    const Watchdog wd{&abort_flag, p.status, p.wait_limit_ns};

    // Every role walks the same tile sequence: this CTA's own index (ordinal 0), then the
    // published ones.  Ordinal o >= 1 uses queue slot o & 1 as that slot's use (o - 1) >> 1, so
    // it waits for phase parity ((o - 1) >> 1) & 1.  Key blocks are counted over the whole
    // sequence for the rings, the S products of each query-tile slot for that slot's S and P
    // barriers, pairs with key blocks for the Q barriers.
    auto next_tile = [&](int ti, int& next) {  // consumers: index of tile ordinal ti + 1
        const int s1 = (ti + 1) & 1;
        if (!warp_wait_all(&bar_tfull[s1], (ti >> 1) & 1, wd, kSiteFwdTile)) return false;
        next = tile_ids[s1];
        __syncwarp();
        mbar_arrive_w(&bar_tempty[s1]);
        return true;
    };

    if (warp == 8) {
        // ------------------------------------------------------------- TMA producer
        // the whole warp runs the loop; elect.sync picks the issuing lane
        int id = static_cast<int>(blockIdx.x), ti = 0, gk = 0, at = 0;
        int issued = 0, issued_q = 0;
        bool clc_pending = false;  // a cancellation request whose response has not landed
        bool ok = true;
        for (;;) {
            const FwdTile t = tile_of(id);
            if (t.Jmax > 0) {
                // this pair's Q tiles once the previous pair's S products have run
                if (at > 0 && !warp_wait_all(&bar_qfree, (at - 1) & 1, wd, kSiteFwdLoadEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&bar_q, t.nt * C::TILE_BYTES);
                for (int q = 0; q < t.nt; ++q)
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_rows_w(sQ + q * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_q, &bar_q,
                                        C::PANEL_ELEMS * pn, t.sr.q0 + (t.qt0 + q) * C::BM, t.qhead,
                                        packed);
                issued_q = at + 1;
                for (int j = 0; j < t.Jmax; ++j) {
                    const int gj = gk + j;
                    const int s = gj % C::STAGES;
                    const uint32_t ph = (gj / C::STAGES) & 1;
                    // K and V stages are released separately (K after the last S product that
                    // reads it, V after the last P V product), so K runs two blocks ahead.
                    if (!warp_wait_all(&bar_kempty[s], ph ^ 1, wd, kSiteFwdLoadEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bar_kfull[s], C::TILE_BYTES);
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_rows_w(sK + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_k,
                                        &bar_kfull[s], C::PANEL_ELEMS * pn, t.sr.k0 + j * C::BN,
                                        t.khead, packed);
                    if (!warp_wait_all(&bar_vempty[s], ph ^ 1, wd, kSiteFwdLoadEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bar_vfull[s], C::TILE_BYTES);
                    if (gj == 0 && (p.debug_flags & kDebugDropFirstLoad)) {
                        // (watchdog test: the announced V tile never arrives)
                    } else if constexpr (F8) {
                        // V^T tile: the d rows of this head, keys [j BN, j BN + BN) (x in bytes)
                        tma_load_3d_w(sV + s * C::TILE_BYTES, &tm_v, &bar_vfull[s], j * C::BN, 0,
                                      t.vthead);
                    } else {
                        for (int pn = 0; pn < C::PANELS; ++pn)
                            tma_load_rows_w(sV + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &tm_v,
                                            &bar_vfull[s], C::PANEL_ELEMS * pn,
                                            t.sr.k0 + j * C::BN, t.khead, packed);
                    }
                    issued = gj + 1;
                }
                if (!ok) break;
                gk += t.Jmax;
                ++at;
            }
            // Take the next tile now, a few blocks before this one ends (a tile taken earlier
            // would wait for this CTA while another SM could already run it).  The request for
            // ordinal ti + 1 is use ti of the response barrier.
            clc_try_cancel_w(&clc_resp, &bar_clc);
            clc_pending = true;
            if (!warp_wait_all(&bar_clc, ti & 1, wd, kSiteFwdTile)) {
                ok = false;
                break;
            }
            clc_pending = false;
            const int next = clc_cancelled_x(&clc_resp);
            __syncwarp();
            const int s1 = (ti + 1) & 1;
            if (!warp_wait_all(&bar_tempty[s1], ((ti >> 1) & 1) ^ 1, wd, kSiteFwdTile)) {
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
        // Let no copy or cancellation response land after the CTA exits: wait (bounded,
        // ignoring the abort flag) for the last ones this warp issued.
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        if (clc_pending) mbar_wait(&bar_clc, ti & 1, wd_drain, kSiteFwdDrain);
        if (issued_q > 0) mbar_wait(&bar_q, (issued_q - 1) & 1, wd_drain, kSiteFwdDrain);
        for (int j = max(0, issued - C::STAGES); j < issued; ++j) {
            const int s = j % C::STAGES;
            const uint32_t ph = (j / C::STAGES) & 1;
            mbar_wait(&bar_kfull[s], ph, wd_drain, kSiteFwdDrain);
            mbar_wait(&bar_vfull[s], ph, wd_drain, kSiteFwdDrain);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------- MMA issuer
        // the whole warp runs the loop (warp-uniform values); elect.sync picks the issuer
        constexpr uint32_t kIdS = F8 ? idesc_e4m3_f32(128, C::BN)  // S = Q K^T
                                     : idesc_bf16_f32(128, C::BN, 0, 0);
        // (d = 64: N = 80 covers V's 64 columns and the first 16 of the constant panel, whose
        // column 0 gives the row sum; the rest of the panel is zero and needs no product)
        constexpr uint32_t kIdPV = F8 ? idesc_e4m3_f32(128, D)  // O += P V
                                      : idesc_bf16_f32(128, C::SUM_ON_MMA ? D + 16 : D, 0, 1);
        // Everything the issue loop needs lives in scalar registers: base descriptors are
        // built once and advanced by byte offsets (stage, tile, k-step), so the single
        // issuing thread keeps pace with the tensor core.
        const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
        // V is MN-major; its second 64-column panel is the next panel of the stage (d = 128)
        // or the constant column panel (d = 64), at a stage-dependent distance.  (e4m3: V^T
        // is K-major, 128 d rows of 128 key bytes.)
        const uint64_t dv0 = F8 ? sdesc_sw128(smem_u32(sV), 16, 1024)
                                : sdesc_sw128(smem_u32(sV), C::PANEL_BYTES, 1024);
        const uint64_t dvo = sdesc_sw128(smem_u32(sV), smem_u32(sOnes) - smem_u32(sV), 1024);
        auto vdesc = [&](int s) {
            if constexpr (C::SUM_ON_MMA) {
                // stage s: start address up, distance to the constant panel down, by the
                // same number of 16-byte units (both fields sit in the low word and stay
                // in range, so neither borrows nor carries)
                const uint32_t u = static_cast<uint32_t>(s * C::TILE_BYTES) >> 4;
                return (dvo & 0xFFFFFFFF00000000ull) |
                       static_cast<uint32_t>(static_cast<uint32_t>(dvo) + u - (u << 16));
            } else {
                return sdesc_adv(dv0, s * C::TILE_BYTES);
            }
        };
        // O_t += P_t V, each half of the keys as soon as the softmax warps have written it
        // (SPLIT_P), else all of it once P is complete; `ph` is the parity of this block's P.
        auto issue_pv_halves = [&](int t, uint32_t ph, uint32_t tO, uint32_t tP, uint64_t vd,
                                   uint32_t acc_first) {
            constexpr int KH = C::SPLIT_P ? C::KSTEPS_PV / 2 : 0;
            if constexpr (C::SPLIT_P) {
                if (!warp_wait_all(&bar_pfull[t][0], ph, wd, kSiteFwdMmaP)) return false;
                tc_fence_after();
                issue_pv<0, KH, F8>(tO, tP, vd, kIdPV, acc_first);
            }
            if (!warp_wait_all(&bar_pfull[t][1], ph, wd, kSiteFwdMmaP)) return false;
            tc_fence_after();
            issue_pv<KH, C::KSTEPS_PV, F8>(tO, tP, vd, kIdPV, acc_first);
            return true;
        };
        const uint32_t tS0 = tbase, tS1 = tbase + 128u;
        const uint32_t tO0 = tbase + 256u, tO1 = tbase + 256u + C::O_COLS;

        int id = static_cast<int>(blockIdx.x), ti = 0, gk = 0, at = 0;
        int cs0 = 0, cs1 = 0;  // S products issued so far into slot 0 / slot 1
        int committed_k = 0, committed_v = 0;  // key blocks whose K / V release was committed
        bool ok = true;
        for (;;) {
            const FwdTile t = tile_of(id);
            const int J0 = t.J[0], J1 = t.J[1], Jmax = t.Jmax;
            // (no key block at all: nothing to issue, the softmax warps write empty rows)
            if (Jmax > 0) {
                if (!warp_wait_all(&bar_q, at & 1, wd, kSiteFwdMmaQ) ||
                    !warp_wait_all(&bar_kfull[gk % C::STAGES], (gk / C::STAGES) & 1, wd,
                                   kSiteFwdMmaK)) {
                    ok = false;
                    break;
                }
                // S of this pair's first block; the previous pair's last P V products, issued
                // before, have read the P these products overwrite
                tc_fence_after();
                const uint64_t kd0 = sdesc_adv(dk0, (gk % C::STAGES) * C::TILE_BYTES);
                if (J0 > 0) {
                    issue_qk<C::KSTEPS_QK, C::PANEL_BYTES, F8>(tS0, dq0, kd0, kIdS);
                    mma_commit_w(&bar_sfull[0]);
                }
                if (J1 > 0) {
                    issue_qk<C::KSTEPS_QK, C::PANEL_BYTES, F8>(tS1, sdesc_adv(dq0, C::TILE_BYTES), kd0,
                                                               kIdS);
                    mma_commit_w(&bar_sfull[1]);
                }
                mma_commit_w(&bar_kempty[gk % C::STAGES]);  // K(0) is read by these S products only
                committed_k = gk + 1;
                if (Jmax == 1) mma_commit_w(&bar_qfree);
                for (int j = 0; ok && j < Jmax; ++j) {
                    const int gj = gk + j;
                    const int s = gj % C::STAGES;
                    const uint32_t ph = (gj / C::STAGES) & 1;
                    const int s1 = (gj + 1) % C::STAGES;
                    const uint32_t ph1 = ((gj + 1) / C::STAGES) & 1;
                    const uint64_t vd = vdesc(s);
                    const uint64_t kd1 = sdesc_adv(dk0, s1 * C::TILE_BYTES);
                    const uint32_t acc_first = j > 0 ? 1u : 0u;
                    if (!warp_wait_all(&bar_vfull[s], ph, wd, kSiteFwdMmaV)) { ok = false; break; }
                    bool k_next = false;
                    // query tile 0
                    if (j < J0) {
                        if (!issue_pv_halves(0, (cs0 + j) & 1, tO0, tS0 + 64u, vd, acc_first)) {
                            ok = false;
                            break;
                        }
                        if (j + 1 == J0) {
                            mma_commit_w(&bar_ofinal[0]);
                        } else {
                            if (!warp_wait_all(&bar_kfull[s1], ph1, wd, kSiteFwdMmaK)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            k_next = true;
                            issue_qk<C::KSTEPS_QK, C::PANEL_BYTES, F8>(tS0, dq0, kd1, kIdS);
                            mma_commit_w(&bar_sfull[0]);
                        }
                    }
                    // query tile 1
                    if (j < J1) {
                        if (!issue_pv_halves(1, (cs1 + j) & 1, tO1, tS1 + 64u, vd, acc_first)) {
                            ok = false;
                            break;
                        }
                        if (j + 1 == J1) {
                            mma_commit_w(&bar_ofinal[1]);
                        } else {
                            if (!k_next) {
                                if (!warp_wait_all(&bar_kfull[s1], ph1, wd, kSiteFwdMmaK)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                            }
                            issue_qk<C::KSTEPS_QK, C::PANEL_BYTES, F8>(
                                tS1, sdesc_adv(dq0, C::TILE_BYTES), kd1, kIdS);
                            mma_commit_w(&bar_sfull[1]);
                            k_next = true;
                        }
                    }
                    if (k_next) {  // K(j + 1) has been read by every S product that needs it
                        mma_commit_w(&bar_kempty[s1]);
                        committed_k = gj + 2;
                    }
                    if (j + 2 == Jmax) mma_commit_w(&bar_qfree);  // every S of the pair issued
                    mma_commit_w(&bar_vempty[s]);  // V(j) has been read by the P V products
                    committed_v = gj + 1;
                }
                if (!ok) break;
                cs0 += J0;
                cs1 += J1;
                gk += Jmax;
                ++at;
            }
            int next = -1;
            if (!next_tile(ti, next)) { ok = false; break; }
            if (next < 0) break;
            id = next;
            ++ti;
        }
        // Wait until every commit this thread issued has arrived, so no arrive lands on
        // shared memory after the CTA exits (bounded; ignores the abort flag).
        volatile int no_abort = 0;
        const Watchdog wd_drain{&no_abort, p.status, p.wait_limit_ns};
        mma_commit_w(&bar_drain);
        mbar_wait(&bar_drain, 0, wd_drain, kSiteFwdDrain);
        for (int j = max(0, committed_k - C::STAGES); j < committed_k; ++j)
            mbar_wait(&bar_kempty[j % C::STAGES], (j / C::STAGES) & 1, wd_drain, kSiteFwdDrain);
        for (int j = max(0, committed_v - C::STAGES); j < committed_v; ++j)
            mbar_wait(&bar_vempty[j % C::STAGES], (j / C::STAGES) & 1, wd_drain, kSiteFwdDrain);
        if (ok && at > 0) mbar_wait(&bar_qfree, (at - 1) & 1, wd_drain, kSiteFwdDrain);
    } else if (warp < 8) {
        // ------------------------------------------------------------- softmax
        const int t = warp >> 2;  // query-tile slot of the pair
        const int r = threadIdx.x & 127;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_base + 128u * t;
        const uint32_t tP = tS + 64u;
        const uint32_t tO = tbase + lane_base + 256u + static_cast<uint32_t>(t * C::O_COLS);
        // Softmax runs on x = S * c with c = scale*log2(e) (exp2 form).  For c <= 0 the
        // scores are pre-multiplied so that masked entries remain -inf after scaling.
        const float c2 = p.scale_log2;
        const bool prescale = !(c2 > 0.0f);
        const float cf = prescale ? 1.0f : c2;
        volatile int* st = sm_state[warp];  // tile index, ordinal, S products, finished pairs
        if (lane == 0) {
            st[0] = static_cast<int>(blockIdx.x);
            st[1] = 0;
            st[2] = 0;
            st[3] = 0;
        }
        __syncwarp();
        bool ok = true;
        for (;;) {
            const int id = st[0];
            // Element-wise masking is needed from key block jmask on: the blocks that straddle
            // the causal diagonal of this tile and the ragged last block.  This row sees the
            // keys [0, klim] of the sequence.  (Only these live through the loop; the epilogue
            // derives the row's place again.)
            int jmask, klim, Jt;
            {
                const FwdTile tl = tile_of(id);
                const int nk = tl.sr.nk;
                const int qt = tl.qt0 + t;
                const int qrow = qt * C::BM + r;  // row within the sequence
                jmask = nk / C::BN;
                klim = nk - 1;
                if (p.causal) {
                    const int e = qt * C::BM + tl.shift + 1;  // blocks below e / BN: all visible
                    jmask = min(jmask, e > 0 ? e / C::BN : 0);
                    klim = min(klim, qrow + tl.shift);
                }
                Jt = t ? tl.J[1] : tl.J[0];
            }
            float m = -INFINITY;  // running max of x (possibly stale by < threshold)
            float l = 0.0f;       // running sum of exp2(x - m) (fp32, before rounding): the LSE
            float lr = 0.0f;      // running sum of the bf16-rounded exp2(x - m): normalises O
            for (int j = 0; ok && j < Jt; ++j) {
                const uint32_t pph = static_cast<uint32_t>(st[2] + j) & 1u;
                if (!warp_wait_all(&bar_sfull[t], pph, wd, kSiteFwdSoftmaxS)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[128];
                tmem_ld32(tS + 0, sr);
                tmem_ld32(tS + 32, sr + 32);
                tmem_ld32(tS + 64, sr + 64);
                tmem_ld32(tS + 96, sr + 96);
                tmem_wait_ld();
                reg_fence32(sr);
                reg_fence32(sr + 32);
                reg_fence32(sr + 64);
                reg_fence32(sr + 96);
                float x[128];
#pragma unroll
                for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
                if (prescale) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) x[c] *= c2;
                }
                // Element-wise mask only on blocks that straddle the causal diagonal and on the
                // ragged last block.
                if (j >= jmask) {
                    const int lim = klim - j * C::BN;  // last visible key column in this block
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > lim) x[c] = -INFINITY;
                }
                // Row max: four independent chains of three-input maxima.
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
                // Rescale only when the max grew by more than the threshold: l and O then keep
                // sharing the same (stale) reference m, so the result stays exact.
                float alpha = 1.0f;
                const bool need = mt > m + C::RESCALE_THRESHOLD;
                if (need) {
                    alpha = ex2(m - mt);  // m = -inf on the first block gives 0
                    m = mt;
                    l *= alpha;
                    lr *= alpha;
                }
                // O still holds the sum up to block j-1 (the commit that signalled S for block j
                // also covers the P V product of block j-1); it is rescaled before the P V
                // product that accumulates into it is signalled: with the first half of P when P
                // is split (then only half of x is still live), else after all of P.
                auto rescale_o = [&]() {
                    if (j > 0 && __any_sync(0xffffffffu, need)) {
                        // (d = 64: columns 64..95 hold the rounded row sum, rescaled with O)
#pragma unroll 1
                        for (int ch = 0; ch < (C::SUM_ON_MMA ? D / 32 + 1 : D / 32); ++ch) {
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
                };
                const float neg_m = (m == -INFINITY) ? 0.0f : -m;
                // exp2(x c - m) on pairs (f32x2 fma), both row sums as f32x2 adds: the exact one
                // over the fp32 values and the one over their bf16 roundings.
                const uint64_t cf2 = f2_make(cf, cf), nm2 = f2_make(neg_m, neg_m);
                uint64_t lsa = f2_make(0.f, 0.f), lsb = lsa, lra = lsa, lrb = lsa;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const int i = cb * 32 + c;
                        float p0, p1, p2, p3;
                        f2_split(f2_fma(f2_make(x[i], x[i + 1]), cf2, nm2), p0, p1);
                        f2_split(f2_fma(f2_make(x[i + 2], x[i + 3]), cf2, nm2), p2, p3);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        p2 = ex2(p2);
                        p3 = ex2(p3);
                        if constexpr (F8) {  // e4m3 P, four keys per column; O is normalised by l
                            lsa = f2_add(lsa, f2_make(p0, p1));
                            lsb = f2_add(lsb, f2_make(p2, p3));
                            pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
                            continue;
                        }
                        const uint32_t w01 = pack_bf16x2(p0, p1);
                        const uint32_t w23 = pack_bf16x2(p2, p3);
                        lsa = f2_add(lsa, f2_make(p0, p1));
                        lsb = f2_add(lsb, f2_make(p2, p3));
                        // lr sums the bf16-rounded weights that the P V product uses, so that
                        // O = sum(P V) / lr is an exact convex combination of those weights
                        // (at d = 64 the tensor core forms this sum in O's column 64).
                        if constexpr (!C::SUM_ON_MMA) {
                            lra = f2_add(lra, f2_make(__uint_as_float(w01 << 16),
                                                      __uint_as_float(w01 & 0xFFFF0000u)));
                            lrb = f2_add(lrb, f2_make(__uint_as_float(w23 << 16),
                                                      __uint_as_float(w23 & 0xFFFF0000u)));
                        }
                        pk[c / 2] = w01;
                        pk[c / 2 + 1] = w23;
                    }
                    if constexpr (F8)
                        tmem_st8(tP + 8u * cb, pk);
                    else
                        tmem_st16(tP + 16u * cb, pk);
                    if (C::SPLIT_P && cb == 1) {  // keys [0, 64) of P are in place: first half
                        rescale_o();
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar_pfull[t][0]);
                    }
                }
                {
                    float a0, a1, b0, b1;
                    f2_split(f2_add(lsa, lsb), a0, a1);
                    f2_split(f2_add(lra, lrb), b0, b1);
                    l += a0 + a1;
                    lr += b0 + b1;
                }
                if constexpr (!C::SPLIT_P) rescale_o();
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_pfull[t][1]);
            }
            int next = -1;
            if (ok && !next_tile(st[1], next)) ok = false;
            // ------------------------------------------------------------- epilogue
            // Where this row goes, derived again rather than held in registers across the loop.
            const FwdTile tl = tile_of(st[0]);
            const int nq = tl.sr.nq;
            const int qrow = (tl.qt0 + t) * C::BM + r;
            const size_t orow_off = static_cast<size_t>(tl.sr.q0 + qrow) * L.o_rs +
                                    static_cast<size_t>(tl.qhead) * L.o_hs;
            const size_t lse_off = static_cast<size_t>(tl.qhead) * L.Rq + tl.sr.q0 + qrow;
            const bool live = t < tl.nt && qrow < nq;
            const bool o_in = !live || in_extent(orow_off, D, L.o_ext, p.status);
            const bool lse_in =
                !live || p.lse == nullptr || in_extent(lse_off, 1, L.stat_ext, p.status);
            if (Jt > 0) {
                if (ok && warp_wait_all(&bar_ofinal[t], st[3] & 1, wd, kSiteFwdSoftmaxO)) {
                    tc_fence_after();
                    // a row that sees no key (possible when queries outnumber keys) stays 0
                    if constexpr (C::SUM_ON_MMA) {  // the rounded row sum from O's column 64
                        uint32_t sc[32];
                        tmem_ld32(tO + 64u, sc);
                        tmem_wait_ld();
                        reg_fence32(sc);
                        lr = __uint_as_float(sc[0]);
                    }
                    float inv_l;
                    if constexpr (F8)
                        inv_l = l > 0.0f ? p.v_descale / l : 0.0f;
                    else
                        inv_l = lr > 0.0f ? 1.0f / lr : 0.0f;
                    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + orow_off;
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32u * ch, o);
                        tmem_wait_ld();
                        reg_fence32(o);
                        uint32_t packed_v[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            packed_v[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                                      __uint_as_float(o[2 * c + 1]) * inv_l);
                        if (qrow < nq && o_in) {
                            uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                dst[c] = make_uint4(packed_v[4 * c], packed_v[4 * c + 1],
                                                    packed_v[4 * c + 2], packed_v[4 * c + 3]);
                        }
                    }
                    if (qrow < nq && p.lse != nullptr && lse_in)
                        p.lse[lse_off] = (m + __log2f(l)) * kLn2;
                    // O is in registers: the next pair's first P V product may overwrite it
                    // (the MMA warp issues it only after this warp's next arrive)
                    tc_fence_before();
                } else {
                    ok = false;
                }
                __syncwarp();
                if (lane == 0) {
                    st[2] += Jt;
                    st[3] += 1;
                }
            } else if (t < tl.nt && qrow < nq) {
                // the whole tile sees no key: O = 0 and lse = log(0) = -inf
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow_off);
                if (o_in)
                    for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
                if (p.lse != nullptr && lse_in) p.lse[lse_off] = -INFINITY;
            }
            if (!ok || next < 0) break;
            __syncwarp();
            if (lane == 0) {
                st[0] = next;
                st[1] += 1;
            }
            __syncwarp();
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

template <int D, int MODE, bool F8 = false>
static cudaError_t launch_fwd_tc_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const FwdParams& p, cudaStream_t st)
{
    using C = FwdCfg<D, F8>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fa_fwd_tc_kernel<D, MODE, F8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int n_qtiles = (p.L.Nq + C::BM - 1) / C::BM;
    const int n_pairs = (n_qtiles + C::NT - 1) / C::NT;
    dim3 grid(p.L.B * p.L.H * n_pairs);
    fa_fwd_tc_kernel<D, MODE, F8><<<grid, C::THREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd_tc(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const FwdParams& p, cudaStream_t st)
{
    const int mode = layout_mode(p.L.cu_q, p.L.H, p.L.Hkv, p.L.Nq, p.L.Nk);
    auto run = [&](auto dc) {
        constexpr int Dc = decltype(dc)::value;
        if (mode == kModePacked) return launch_fwd_tc_impl<Dc, kModePacked>(tq, tk, tv, p, st);
        if (mode == kModeFixedGroup) return launch_fwd_tc_impl<Dc, kModeFixedGroup>(tq, tk, tv, p, st);
        return launch_fwd_tc_impl<Dc, kModeFixed>(tq, tk, tv, p, st);
    };
    return d == 64 ? run(std::integral_constant<int, 64>{}) : run(std::integral_constant<int, 128>{});
}

// e4m3 forward, d = 128: fixed-length square heads or packed batches (grouped heads, Nq !=
// Nk); tvt maps the transposed V^T copy.
cudaError_t launch_fwd_fp8_tc(const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tvt, const FwdParams& p, cudaStream_t st)
{
    if (p.L.cu_q != nullptr) return launch_fwd_tc_impl<128, kModePacked, true>(tq, tk, tvt, p, st);
    return launch_fwd_tc_impl<128, kModeFixed, true>(tq, tk, tvt, p, st);
}

}  // namespace fa
