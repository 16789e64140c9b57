// Portable SIMT kernels (CUDA cores, fp32 math):
//   - forward with the tiled online softmax (the fp32 path; also a cross-check for bf16),
//   - backward preprocess Delta_i = rowsum(dO_i o O_i) and the base-2 LSE (used by every
//     backward path),
//   - backward as the two loops of "Backward 구현" in "Triton 06: Flash Attention v2":
//     a dK/dV kernel (outer loop over key rows, inner over query blocks) and a dQ kernel
//     (outer loop over query rows, inner over key blocks).  No atomics: deterministic.
// One warp owns 4 rows; a CTA of 4 warps owns 16 rows and stages 32-row tiles of the other
// operands in shared memory.
#include "fa_common.cuh"
#include "tc_ptx.cuh"

namespace fa {

constexpr int kSimtWarps = 4;
constexpr int kSimtRowsPerWarp = 4;
constexpr int kSimtRows = kSimtWarps * kSimtRowsPerWarp;  // rows owned by one CTA
constexpr int kSimtTile = 32;                              // rows of a staged tile

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p)
{
    return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_elem(T* p, float v);
template <>
__device__ __forceinline__ void st_elem<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_elem<__nv_bfloat16>(__nv_bfloat16* p, float v)
{
    *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Four consecutive elements as fp32 (one 16-byte load for fp32, one 8-byte load for bf16).
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p)
{
    return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p)
{
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

// Stage rows [row0, row0+ROWS) of one head into shared memory as fp32 with row stride ld;
// rows at or beyond N are zero.  Every thread of the NT-thread CTA first loads all of its
// 4-element vectors into registers and only then stores them, so the loads of a whole tile
// are in flight together.
template <typename T, int D, int ROWS, int NT = 128>
__device__ __forceinline__ void stage_rows(float* dst, int ld, const T* head, int row0, int N)
{
    constexpr int NV = ROWS * D / 4;          // 4-element vectors in the tile
    constexpr int PER = (NV + NT - 1) / NT;   // per thread
    float4 vals[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = (static_cast<int>(threadIdx.x) + i * NT) * 4;
        const int r = e / D, c = e % D;
        const int g = row0 + r;
        vals[i] = (e < ROWS * D && g < N) ? load4(head + static_cast<size_t>(g) * D + c)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = (static_cast<int>(threadIdx.x) + i * NT) * 4;
        if (e < ROWS * D) {
            float* d = dst + (e / D) * ld + (e % D);
            d[0] = vals[i].x;
            d[1] = vals[i].y;
            d[2] = vals[i].z;
            d[3] = vals[i].w;
        }
    }
}

// The two halves of stage_rows, for a tile whose loads fly while the previous one is used:
// rows [row0, row0+ROWS) of one head into this thread's registers (zero beyond N) ...
template <typename T, int D, int ROWS, int NT>
__device__ __forceinline__ void load_rows(float4 (&vals)[(ROWS * D / 4 + NT - 1) / NT],
                                          const T* head, int row0, int N)
{
    constexpr int PER = (ROWS * D / 4 + NT - 1) / NT;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = (static_cast<int>(threadIdx.x) + i * NT) * 4;
        const int r = e / D, c = e % D;
        const int g = row0 + r;
        vals[i] = (e < ROWS * D && g < N) ? load4(head + static_cast<size_t>(g) * D + c)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// ... and from the registers into shared memory with row stride ld.
template <int D, int ROWS, int NT>
__device__ __forceinline__ void store_rows(float* dst, int ld,
                                           const float4 (&vals)[(ROWS * D / 4 + NT - 1) / NT])
{
    constexpr int PER = (ROWS * D / 4 + NT - 1) / NT;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = (static_cast<int>(threadIdx.x) + i * NT) * 4;
        if (e < ROWS * D) {
            float* d = dst + (e / D) * ld + (e % D);
            d[0] = vals[i].x;
            d[1] = vals[i].y;
            d[2] = vals[i].z;
            d[3] = vals[i].w;
        }
    }
}

// Dot product of two D-vectors in shared memory with four independent partial sums.
template <int D>
__device__ __forceinline__ float dot_smem(const float* a, const float* b)
{
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int c = 0; c < D; c += 4) {
        s0 = fmaf(a[c], b[c], s0);
        s1 = fmaf(a[c + 1], b[c + 1], s1);
        s2 = fmaf(a[c + 2], b[c + 2], s2);
        s3 = fmaf(a[c + 3], b[c + 3], s3);
    }
    return (s0 + s1) + (s2 + s3);
}

// ----------------------------------------------------------------------------------------
// Forward: O and LSE for 16 query rows per CTA, RPW rows per warp (4: 128 threads, each V
// element read from shared memory serves four rows; 1: 512 threads, for grids too small to
// fill the GPU, where each warp's chain of dependent steps per key tile is the time).  Every
// row is computed the same way either way.
// ----------------------------------------------------------------------------------------
template <typename T, int D, int RPW>
__global__ void __launch_bounds__(kSimtRows / RPW * 32) fa_fwd_simt_kernel(const FwdParams p)
{
    constexpr int NT = kSimtRows / RPW * 32;  // threads
    constexpr int DL = D / 32;  // output columns per lane
    extern __shared__ float sm[];
    float* Qs = sm;                          // [16][D]
    float* Ks = Qs + kSimtRows * D;          // [32][D+1]
    float* Vs = Ks + kSimtTile * (D + 1);    // [32][D]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, bh = blockIdx.y;
    const int row_base = blockIdx.x * kSimtRows;
    const size_t hoff = static_cast<size_t>(bh) * N * D;
    const T* q = static_cast<const T*>(p.q) + hoff;
    const T* k = static_cast<const T*>(p.k) + hoff;
    const T* v = static_cast<const T*>(p.v) + hoff;
    stage_rows<T, D, kSimtRows, NT>(Qs, D, q, row_base, N);

    const float c2 = p.scale_log2;
    float m[RPW], l[RPW], o[RPW][DL];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.0f;
#pragma unroll
        for (int t = 0; t < DL; ++t) o[rr][t] = 0.0f;
    }
    const int last_row = min(N - 1, row_base + kSimtRows - 1);
    const int n_tiles = p.causal ? (last_row / kSimtTile + 1) : (N + kSimtTile - 1) / kSimtTile;
    // With one row per warp the K and V tiles go through registers one tile ahead (one or two
    // vectors a thread), so the loads of tile kt + 1 are in flight while tile kt is computed;
    // with four rows per warp those registers would cost occupancy.
    constexpr bool kAhead = RPW == 1;
    constexpr int PER = (kSimtTile * D / 4 + NT - 1) / NT;
    float4 kreg[PER], vreg[PER];
    if constexpr (kAhead) {
        load_rows<T, D, kSimtTile, NT>(kreg, k, 0, N);
        load_rows<T, D, kSimtTile, NT>(vreg, v, 0, N);
    }
    for (int kt = 0; kt < n_tiles; ++kt) {
        __syncthreads();
        if constexpr (kAhead) {
            store_rows<D, kSimtTile, NT>(Ks, D + 1, kreg);
            store_rows<D, kSimtTile, NT>(Vs, D, vreg);
        } else {
            stage_rows<T, D, kSimtTile, NT>(Ks, D + 1, k, kt * kSimtTile, N);
            stage_rows<T, D, kSimtTile, NT>(Vs, D, v, kt * kSimtTile, N);
        }
        __syncthreads();
        if (kAhead && kt + 1 < n_tiles) {
            load_rows<T, D, kSimtTile, NT>(kreg, k, (kt + 1) * kSimtTile, N);
            load_rows<T, D, kSimtTile, NT>(vreg, v, (kt + 1) * kSimtTile, N);
        }
        const int key = kt * kSimtTile + lane;
        // scores of this warp's rows against the tile's keys (lane = key) ...
        float pr[RPW], alpha[RPW];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int lr = warp * RPW + rr;
            const int row = row_base + lr;
            const float s = dot_smem<D>(Qs + lr * D, Ks + lane * (D + 1));
            const bool valid = key < N && (!p.causal || key <= row);
            pr[rr] = valid ? s * c2 : -INFINITY;
        }
        // ... the online-softmax update of each row (rows with nothing visible yet keep their
        // state: alpha = 1, weights 0) ...
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const float mnew = fmaxf(m[rr], warp_max(pr[rr]));
            if (mnew == -INFINITY) {
                alpha[rr] = 1.0f;
                pr[rr] = 0.0f;
                continue;
            }
            alpha[rr] = ex2(m[rr] - mnew);
            pr[rr] = ex2(pr[rr] - mnew);
            l[rr] = l[rr] * alpha[rr] + warp_sum(pr[rr]);
            m[rr] = mnew;
        }
        // ... and O += P V for all rows at once (one V read per key serves every row)
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
            for (int t = 0; t < DL; ++t) o[rr][t] *= alpha[rr];
#pragma unroll 4
        for (int c = 0; c < kSimtTile; ++c) {
            float vc[DL];
#pragma unroll
            for (int t = 0; t < DL; ++t) vc[t] = Vs[c * D + lane + 32 * t];
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                const float pc = __shfl_sync(0xffffffffu, pr[rr], c);
#pragma unroll
                for (int t = 0; t < DL; ++t) o[rr][t] = fmaf(pc, vc[t], o[rr][t]);
            }
        }
    }
    T* out = static_cast<T*>(p.o) + hoff;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int row = row_base + warp * RPW + rr;
        if (row >= N) continue;
        const float inv = 1.0f / l[rr];
#pragma unroll
        for (int t = 0; t < DL; ++t)
            st_elem(out + static_cast<size_t>(row) * D + lane + 32 * t, o[rr][t] * inv);
        if (lane == 0 && p.lse) p.lse[static_cast<size_t>(bh) * N + row] = (m[rr] + __log2f(l[rr])) * kLn2;
    }
}

// ----------------------------------------------------------------------------------------
// Backward preprocess: Delta_i = sum_c dO_ic O_ic (fp32 accumulation) and lse2_i = lse_i *
// log2(e).  D/8 threads per row, 16-byte loads for bf16 (D/4 threads, 16 B, for fp32).
// ----------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const BwdParams p)
{
    // the dK/dV grid after this one (a programmatic dependent) may set up now; it waits for this
    // grid before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int EPV = 16 / sizeof(T);  // elements per 16-byte vector
    constexpr int TPR = D / EPV;         // threads per row (8, 16 or 32)
    constexpr int RPW = 32 / TPR;        // rows per warp and iteration
    // Rows t = hh * Rq + i of the statistics arrays: row i of head index hh, whose elements sit
    // at i * rs + hh * hs with the strides of O and of dO.
    const Layout& L = p.L;
    const size_t n_heads = static_cast<size_t>(L.cu_q == nullptr ? L.B * L.H : L.H);
    const size_t rows = n_heads * static_cast<size_t>(L.Rq);
    const int lane = threadIdx.x & 31;
    const int sub = lane % TPR;
    const size_t warps_total = static_cast<size_t>(gridDim.x) * (blockDim.x / 32);
    const size_t gw = static_cast<size_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    // The loop bound is uniform across the warp, so the shuffles below see all 32 lanes.
    for (size_t base = gw * RPW; base < rows; base += warps_total * RPW) {
        const size_t row = base + lane / TPR;
        const size_t hh = row / static_cast<size_t>(L.Rq), i = row - hh * static_cast<size_t>(L.Rq);
        const size_t off_o = i * static_cast<size_t>(L.o_rs) + hh * static_cast<size_t>(L.o_hs);
        const size_t off_g = i * static_cast<size_t>(L.do_rs) + hh * static_cast<size_t>(L.do_hs);
        const bool valid = row < rows && in_extent(off_o, D, L.o_ext, p.status) &&
                           in_extent(off_g, D, L.do_ext, p.status) &&
                           in_extent(row, 1, L.stat_ext, p.status);
        float acc = 0.0f;
        if (valid) {
            const uint4 a = reinterpret_cast<const uint4*>(static_cast<const T*>(p.o) + off_o)[sub];
            const uint4 b = reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) + off_g)[sub];
            const T* ea = reinterpret_cast<const T*>(&a);
            const T* eb = reinterpret_cast<const T*>(&b);
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc = fmaf(ld_elem(ea + e), ld_elem(eb + e), acc);
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
        if (valid && sub == 0) {
            p.delta[row] = acc;
            p.lse2[row] = p.lse[row] * kLog2e;
        }
    }
}

// ----------------------------------------------------------------------------------------
// Backward dQ (outer loop over query rows, inner over key tiles).
// ----------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) fa_bwd_dq_simt_kernel(const BwdParams p)
{
    constexpr int DL = D / 32;
    extern __shared__ float sm[];
    float* Qs = sm;                          // [16][D]
    float* Gs = Qs + kSimtRows * D;          // dO rows [16][D]
    float* Ks = Gs + kSimtRows * D;          // [32][D+1]
    float* Vs = Ks + kSimtTile * (D + 1);    // [32][D+1]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, bh = blockIdx.y;
    const int row_base = blockIdx.x * kSimtRows;
    const size_t hoff = static_cast<size_t>(bh) * N * D;
    const T* q = static_cast<const T*>(p.q) + hoff;
    const T* k = static_cast<const T*>(p.k) + hoff;
    const T* v = static_cast<const T*>(p.v) + hoff;
    const T* g = static_cast<const T*>(p.dout) + hoff;
    stage_rows<T, D, kSimtRows>(Qs, D, q, row_base, N);
    stage_rows<T, D, kSimtRows>(Gs, D, g, row_base, N);
    float L2[kSimtRowsPerWarp], Dl[kSimtRowsPerWarp], acc[kSimtRowsPerWarp][DL];
#pragma unroll
    for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
        const int row = row_base + warp * kSimtRowsPerWarp + rr;
        const size_t ri = static_cast<size_t>(bh) * N + min(row, N - 1);
        L2[rr] = p.lse2[ri];
        Dl[rr] = p.delta[ri];
#pragma unroll
        for (int t = 0; t < DL; ++t) acc[rr][t] = 0.0f;
    }
    const float c2 = p.scale_log2;
    const int last_row = min(N - 1, row_base + kSimtRows - 1);
    const int n_tiles = p.causal ? (last_row / kSimtTile + 1) : (N + kSimtTile - 1) / kSimtTile;
    for (int kt = 0; kt < n_tiles; ++kt) {
        __syncthreads();
        stage_rows<T, D, kSimtTile>(Ks, D + 1, k, kt * kSimtTile, N);
        stage_rows<T, D, kSimtTile>(Vs, D + 1, v, kt * kSimtTile, N);
        __syncthreads();
        const int key = kt * kSimtTile + lane;
#pragma unroll
        for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
            const int lr = warp * kSimtRowsPerWarp + rr;
            const int row = row_base + lr;
            float s = 0.0f, dp = 0.0f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                s = fmaf(Qs[lr * D + c], Ks[lane * (D + 1) + c], s);
                dp = fmaf(Gs[lr * D + c], Vs[lane * (D + 1) + c], dp);
            }
            const bool valid = key < N && row < N && (!p.causal || key <= row);
            const float pr = valid ? ex2(s * c2 - L2[rr]) : 0.0f;
            const float ds = pr * (dp - Dl[rr]);
#pragma unroll 4
            for (int c = 0; c < kSimtTile; ++c) {
                const float dc = __shfl_sync(0xffffffffu, ds, c);
#pragma unroll
                for (int t = 0; t < DL; ++t) acc[rr][t] = fmaf(dc, Ks[c * (D + 1) + lane + 32 * t], acc[rr][t]);
            }
        }
    }
    T* dq = static_cast<T*>(p.dq) + hoff;
#pragma unroll
    for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
        const int row = row_base + warp * kSimtRowsPerWarp + rr;
        if (row >= N) continue;
#pragma unroll
        for (int t = 0; t < DL; ++t)
            st_elem(dq + static_cast<size_t>(row) * D + lane + 32 * t, acc[rr][t] * p.scale);
    }
}

// ----------------------------------------------------------------------------------------
// Backward dK, dV (outer loop over key rows, inner over query tiles).
// ----------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) fa_bwd_dkv_simt_kernel(const BwdParams p)
{
    constexpr int DL = D / 32;
    extern __shared__ float sm[];
    float* Kw = sm;                          // own key rows [16][D]
    float* Vw = Kw + kSimtRows * D;          // own value rows [16][D]
    float* Qs = Vw + kSimtRows * D;          // [32][D+1]
    float* Gs = Qs + kSimtTile * (D + 1);    // dO tile [32][D+1]
    float* Ls = Gs + kSimtTile * (D + 1);    // lse2 of the tile [32]
    float* Ds = Ls + kSimtTile;              // Delta of the tile [32]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, bh = blockIdx.y;
    const int key_base = blockIdx.x * kSimtRows;
    const size_t hoff = static_cast<size_t>(bh) * N * D;
    const T* q = static_cast<const T*>(p.q) + hoff;
    const T* k = static_cast<const T*>(p.k) + hoff;
    const T* v = static_cast<const T*>(p.v) + hoff;
    const T* g = static_cast<const T*>(p.dout) + hoff;
    stage_rows<T, D, kSimtRows>(Kw, D, k, key_base, N);
    stage_rows<T, D, kSimtRows>(Vw, D, v, key_base, N);
    float dk[kSimtRowsPerWarp][DL], dv[kSimtRowsPerWarp][DL];
#pragma unroll
    for (int rr = 0; rr < kSimtRowsPerWarp; ++rr)
#pragma unroll
        for (int t = 0; t < DL; ++t) dk[rr][t] = dv[rr][t] = 0.0f;
    const float c2 = p.scale_log2;
    const int first_tile = p.causal ? key_base / kSimtTile : 0;
    const int n_tiles = (N + kSimtTile - 1) / kSimtTile;
    for (int it = first_tile; it < n_tiles; ++it) {
        __syncthreads();
        stage_rows<T, D, kSimtTile>(Qs, D + 1, q, it * kSimtTile, N);
        stage_rows<T, D, kSimtTile>(Gs, D + 1, g, it * kSimtTile, N);
        if (threadIdx.x < kSimtTile) {
            const int i = it * kSimtTile + threadIdx.x;
            Ls[threadIdx.x] = (i < N) ? p.lse2[static_cast<size_t>(bh) * N + i] : INFINITY;
            Ds[threadIdx.x] = (i < N) ? p.delta[static_cast<size_t>(bh) * N + i] : 0.0f;
        }
        __syncthreads();
        const int qi = it * kSimtTile + lane;
#pragma unroll
        for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
            const int lk = warp * kSimtRowsPerWarp + rr;
            const int key = key_base + lk;
            float s = 0.0f, dp = 0.0f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                s = fmaf(Qs[lane * (D + 1) + c], Kw[lk * D + c], s);
                dp = fmaf(Gs[lane * (D + 1) + c], Vw[lk * D + c], dp);
            }
            const bool valid = qi < N && key < N && (!p.causal || key <= qi);
            const float pr = valid ? ex2(s * c2 - Ls[lane]) : 0.0f;
            const float ds = pr * (dp - Ds[lane]);
#pragma unroll 4
            for (int c = 0; c < kSimtTile; ++c) {
                const float pc = __shfl_sync(0xffffffffu, pr, c);
                const float dc = __shfl_sync(0xffffffffu, ds, c);
#pragma unroll
                for (int t = 0; t < DL; ++t) {
                    dv[rr][t] = fmaf(pc, Gs[c * (D + 1) + lane + 32 * t], dv[rr][t]);
                    dk[rr][t] = fmaf(dc, Qs[c * (D + 1) + lane + 32 * t], dk[rr][t]);
                }
            }
        }
    }
    T* dK = static_cast<T*>(p.dk) + hoff;
    T* dV = static_cast<T*>(p.dv) + hoff;
#pragma unroll
    for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
        const int key = key_base + warp * kSimtRowsPerWarp + rr;
        if (key >= N) continue;
#pragma unroll
        for (int t = 0; t < DL; ++t) {
            st_elem(dK + static_cast<size_t>(key) * D + lane + 32 * t, dk[rr][t] * p.scale);
            st_elem(dV + static_cast<size_t>(key) * D + lane + 32 * t, dv[rr][t]);
        }
    }
}

// ----------------------------------------------------------------------------------------
// Launchers.
// ----------------------------------------------------------------------------------------
template <typename K>
static cudaError_t set_smem(K kernel, int bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T, int D, int RPW>
static cudaError_t fwd_simt_rpw(const FwdParams& p, cudaStream_t st, dim3 grid)
{
    const int smem = (kSimtRows * D + kSimtTile * (D + 1) + kSimtTile * D) * 4;
    cudaError_t e = set_smem(fa_fwd_simt_kernel<T, D, RPW>, smem);
    if (e != cudaSuccess) return e;
    fa_fwd_simt_kernel<T, D, RPW><<<grid, kSimtRows / RPW * 32, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t fwd_simt(const FwdParams& p, cudaStream_t st, int num_sms)
{
    dim3 grid((p.N + kSimtRows - 1) / kSimtRows, p.BH);
    // fewer CTAs than SMs: one row per warp shortens each CTA's dependent chain four times
    if (static_cast<long long>(grid.x) * grid.y < num_sms) return fwd_simt_rpw<T, D, 1>(p, st, grid);
    return fwd_simt_rpw<T, D, 4>(p, st, grid);
}

cudaError_t launch_fwd_simt(int d, int is_f32, const FwdParams& p, cudaStream_t st, int num_sms)
{
    if (is_f32)
        return d == 64 ? fwd_simt<float, 64>(p, st, num_sms) : fwd_simt<float, 128>(p, st, num_sms);
    return d == 64 ? fwd_simt<__nv_bfloat16, 64>(p, st, num_sms)
                   : fwd_simt<__nv_bfloat16, 128>(p, st, num_sms);
}

template <typename T, int D>
static cudaError_t bwd_pre(const BwdParams& p, cudaStream_t st, int num_sms)
{
    constexpr int TPR = D / (16 / sizeof(T));
    const long rows = static_cast<long>(p.L.cu_q == nullptr ? p.L.B * p.L.H : p.L.H) * p.L.Rq;
    const int rows_per_block = 256 / TPR;
    long blocks = (rows + rows_per_block - 1) / rows_per_block;
    const long cap = static_cast<long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    fa_bwd_preprocess_kernel<T, D><<<static_cast<int>(blocks), 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(int d, int is_f32, const BwdParams& p, cudaStream_t st, int num_sms)
{
    if (is_f32) return d == 64 ? bwd_pre<float, 64>(p, st, num_sms) : bwd_pre<float, 128>(p, st, num_sms);
    return d == 64 ? bwd_pre<__nv_bfloat16, 64>(p, st, num_sms)
                   : bwd_pre<__nv_bfloat16, 128>(p, st, num_sms);
}

template <typename T, int D>
static cudaError_t bwd_simt(const BwdParams& p, cudaStream_t st)
{
    const int smem_dq = (2 * kSimtRows * D + 2 * kSimtTile * (D + 1)) * 4;
    const int smem_dkv = (2 * kSimtRows * D + 2 * kSimtTile * (D + 1) + 2 * kSimtTile) * 4;
    cudaError_t e = set_smem(fa_bwd_dq_simt_kernel<T, D>, smem_dq);
    if (e != cudaSuccess) return e;
    e = set_smem(fa_bwd_dkv_simt_kernel<T, D>, smem_dkv);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kSimtRows - 1) / kSimtRows, p.BH);
    fa_bwd_dkv_simt_kernel<T, D><<<grid, 128, smem_dkv, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    fa_bwd_dq_simt_kernel<T, D><<<grid, 128, smem_dq, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_simt(int d, int is_f32, const BwdParams& p, cudaStream_t st)
{
    if (is_f32) return d == 64 ? bwd_simt<float, 64>(p, st) : bwd_simt<float, 128>(p, st);
    return d == 64 ? bwd_simt<__nv_bfloat16, 64>(p, st) : bwd_simt<__nv_bfloat16, 128>(p, st);
}

}  // namespace fa
