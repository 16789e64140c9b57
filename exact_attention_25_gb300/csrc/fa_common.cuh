// Shared definitions of the attention library: parameter blocks, watchdog sites, and the
// causal block classification used by every kernel and by the host-side scheduler.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Watchdog sites written into the device status word when a bounded wait expires.
enum WaitSite : int {
    kSiteFwdLoadEmpty = 1,
    kSiteFwdMmaQ,
    kSiteFwdMmaK,
    kSiteFwdMmaV,
    kSiteFwdMmaP,
    kSiteFwdSoftmaxS,
    kSiteFwdSoftmaxO,
    kSiteFwdDrain,
    kSiteFwdTile,  // the next tile's index (persistent kernels)
    kSiteBwdLoadEmpty = 16,
    kSiteBwdMmaKV,
    kSiteBwdMmaQ,
    kSiteBwdMmaP,
    kSiteBwdMmaDS,
    kSiteBwdEltS,
    kSiteBwdEltAcc,
    kSiteBwdDrain,
    kSiteBwdTile,
};

// Test hook: the producer announces the bytes of its first streamed tile but never issues
// the copy, so the barrier guarding that tile never completes and every bounded wait on it
// must expire (watchdog test).  Never set in normal operation.
constexpr int kDebugDropFirstLoad = 1;
// Test hook of checked builds: the host passes every buffer extent one row short, so the
// bounds checks must catch (and skip) the last row's accesses.
constexpr int kDebugShrinkExtents = 2;

// Status word value of a failed bounds check (checked builds); wait sites are below 64.
constexpr int kStatusOutOfBounds = 0x0B0B;

// Checked builds (-DFA_CHECKED) verify every direct global access of n elements at element
// offset off against the extent of its buffer; a violation is recorded in the status word
// and the access is skipped.  Regular builds compile the check away.
#ifdef FA_CHECKED
__device__ __forceinline__ bool in_extent(long long off, long long n, long long extent, int* status)
{
    if (off >= 0 && off + n <= extent) return true;
    atomicCAS(status, 0, kStatusOutOfBounds);
    return false;
}
#else
__device__ __forceinline__ constexpr bool in_extent(long long, long long, long long, int*)
{
    return true;
}
#endif

// Causal mask (key index <= query index, top-left aligned): classification of the key
// block [k0, k1) against the query block [q0, q1), following the two-stage split of the
// FlashAttention-2 Triton write-up ("개선 3: Causal Mask 2-Stage"):
//   FULL   - every key <= every query: no mask needed ("stage 1"),
//   MASKED - the block straddles the diagonal: mask element-wise ("stage 2"),
//   SKIP   - every key is in the future of every query: never visited.
enum TileClass : int { kTileFull = 0, kTileMasked = 1, kTileSkip = 2 };

__host__ __device__ inline int causal_tile_class(int q0, int q1, int k0, int k1)
{
    if (k0 > q1 - 1) return kTileSkip;
    if (k1 - 1 <= q0) return kTileFull;
    return kTileMasked;
}

// Order of the work tiles of a launch over `heads` heads of `nblk` tiles each, tile rank 0
// being the heaviest of a head under the causal mask.  Heads go in groups of `gsize` consecutive
// heads; within a group the tiles go by rank, the group's heads interleaved, and groups follow
// one another.  So the heaviest tiles of a group start first and its light ones fill the end,
// instead of the last head's heaviest tile starting when everything else is nearly done, while
// the tiles resident at one time still share the key/value (or query) rows of a few heads in
// L2.  gsize = 1 is plain head-major order.  Tile `id` in [0, heads * nblk) maps to one (head,
// rank) pair, and every pair is reached once.
__host__ __device__ inline void tile_order(int id, int heads, int nblk, int gsize, int& head,
                                           int& rank)
{
    const int g0 = id / (gsize * nblk) * gsize;   // first head of the tile's group
    const int gh = min(gsize, heads - g0);        // heads in that group (the last may be short)
    const int p = id - g0 * nblk;                 // position within the group
    rank = p / gh;
    head = g0 + p % gh;
}

// Where the rows of one (sequence, head) problem live.  Two layouts:
//   fixed length  q/o/dO/dQ [B, H, Nq, d], k/v/dK/dV [B, Hkv, Nk, d]: head index b*H + h (or
//                 b*Hkv + hk), row offset 0;
//   packed        q/o/dO/dQ [total_q, H, d], k/v/dK/dV [total_k, Hkv, d] with the sequences
//                 back to back ("variable length", cu_q / cu_k = B+1 sequence starts): head
//                 index h (or hk), row offset cu[b].
// Per-row statistics (lse, Delta, base-2 LSE) are [head index][Rq].  Query head h reads key /
// value head h / (H / Hkv) (grouped-query attention; Hkv = H is ordinary multi-head).
//
// Every tensor-core kernel is compiled for three modes: the fixed-length layout with Nq == Nk
// and Hkv == H (kModeFixed, which skips the group loop and the causal shift), the fixed-length
// layout with grouped heads and Nq != Nk allowed (kModeFixedGroup), and the packed layout
// (kModePacked).
enum LayoutMode : int { kModeFixed = 0, kModeFixedGroup = 1, kModePacked = 2 };

__host__ __device__ constexpr bool mode_packed(int mode) { return mode == kModePacked; }
__host__ __device__ constexpr bool mode_general(int mode) { return mode != kModeFixed; }
inline int layout_mode(const void* cu_q, int H, int Hkv, int Nq, int Nk)
{
    if (cu_q != nullptr) return kModePacked;
    return (H != Hkv || Nq != Nk) ? kModeFixedGroup : kModeFixed;
}
struct Layout {
    const int* cu_q;       // packed layout: B+1 query-row starts (device), else null
    const int* cu_k;       // packed layout: B+1 key-row starts (device), else null
    int B, H, Hkv;         // sequences, query heads, key/value heads (H % Hkv == 0)
    int Nq, Nk;            // fixed: rows per sequence; packed: largest sequence (grid, clamps)
    int Rq, Rk;            // rows per head index: fixed Nq, Nk; packed total_q, total_k
    // Element strides of one row and one head index of the tensors the kernels address
    // directly (q, k, v and dO are read through tensor maps that carry their own strides).
    long long o_rs, o_hs;
    long long do_rs, do_hs;
    long long dq_rs, dq_hs;
    long long dk_rs, dk_hs;
    long long dv_rs, dv_hs;
    // Element extents of those buffers and of the per-row statistics (lse, Delta, base-2
    // LSE), checked in checked builds only.
    long long o_ext, do_ext, dq_ext, dk_ext, dv_ext, stat_ext;
    int order_group;  // heads per group of the tensor-core kernels' tile order (tile_order)
};

// Rows of sequence b: global row offsets q0 / k0 and lengths nq / nk.  Packed offsets and
// lengths are clamped to the tensors (Rq, Rk) and to Nq / Nk, so that inconsistent sequence
// starts can never address memory outside the caller's buffers.
struct SeqRows {
    int q0, nq, k0, nk;
};

template <bool PACKED>
__device__ __forceinline__ SeqRows seq_rows(const Layout& L, int b)
{
    SeqRows s;
    if constexpr (!PACKED) {
        s.q0 = 0; s.nq = L.Nq; s.k0 = 0; s.nk = L.Nk;
        return s;
    }
    const int qa = min(max(L.cu_q[b], 0), L.Rq), qb = min(max(L.cu_q[b + 1], qa), L.Rq);
    const int ka = min(max(L.cu_k[b], 0), L.Rk), kb = min(max(L.cu_k[b + 1], ka), L.Rk);
    s.q0 = qa; s.nq = min(qb - qa, L.Nq);
    s.k0 = ka; s.nk = min(kb - ka, L.Nk);
    return s;
}

template <bool PACKED>
__device__ __forceinline__ int q_head_index(const Layout& L, int b, int h)
{
    return PACKED ? h : b * L.H + h;
}
template <bool PACKED>
__device__ __forceinline__ int k_head_index(const Layout& L, int b, int hk)
{
    return PACKED ? hk : b * L.Hkv + hk;
}

// Bottom-right causal alignment for a problem of nq queries and nk keys: query i sees key j
// iff j <= i + (nk - nq).  For nq == nk this is the square mask above; a chunk of the last nq
// queries of a longer sequence (chunked prefill) sees every earlier key.  The shifted query
// bounds go through causal_tile_class unchanged.
__device__ __forceinline__ int causal_class_shifted(int q0, int q1, int k0, int k1, int shift)
{
    return causal_tile_class(q0 + shift, q1 + shift, k0, k1);
}

// Parameters of the forward kernels.  The SIMT kernels use N and BH (fixed layout, square);
// the tensor-core kernels use the layout L.
struct FwdParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int N;
    int BH;
    float scale;       // softmax scale applied to Q K^T
    float scale_log2;  // scale * log2(e), folded once on the host
    int causal;
    int* status;       // device status word (watchdog)
    unsigned long long wait_limit_ns;
    int debug_flags;   // test hook: kDebugDropFirstLoad
    float v_descale;   // e4m3 forward: the factor that turns stored V codes into values
    Layout L;
};

// Parameters of the backward kernels.
struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const void* dout;
    const float* lse;  // natural-log LSE from the forward
    void* dq;
    void* dk;
    void* dv;
    float* delta;      // workspace: Delta_i = rowsum(dO o O), [B*H, N]
    float* lse2;       // workspace: base-2 LSE (lse * log2 e), [B*H, N]
    int N;
    int BH;
    float scale;
    float scale_log2;
    int causal;
    int* status;
    unsigned long long wait_limit_ns;
    int debug_flags;
    Layout L;
};

}  // namespace fa
