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
    kSiteBwdLoadEmpty = 16,
    kSiteBwdMmaKV,
    kSiteBwdMmaQ,
    kSiteBwdMmaP,
    kSiteBwdMmaDS,
    kSiteBwdEltS,
    kSiteBwdEltAcc,
    kSiteBwdDrain,
};

// Test hook: the producer announces the bytes of its first streamed tile but never issues
// the copy, so the barrier guarding that tile never completes and every bounded wait on it
// must expire (watchdog test).  Never set in normal operation.
constexpr int kDebugDropFirstLoad = 1;

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

// Parameters of the forward kernels.  All tensors are contiguous [B*H, N, d] (LSE [B*H, N]).
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
};

}  // namespace fa
