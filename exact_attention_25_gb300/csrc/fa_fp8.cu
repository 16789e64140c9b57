// Preparation for the e4m3 forward: V [B*H, N, d] -> V^T [B*H, d, Npad] (Npad = N rounded up
// to 16 keys, the pad keys zero), so that V enters O += P V as a K-major operand like P.
// HBM-bound: one read and one write of V.  Each CTA moves 64 keys x 128 bytes of one head
// through shared memory: 16-byte row loads in, 16-byte stores of 16 consecutive keys of one
// d column out.
#include "fa_common.cuh"

namespace fa {

constexpr int kVtKeys = 64;      // keys per CTA
constexpr int kVtThreads = 256;

__global__ void __launch_bounds__(kVtThreads) fa_vt_transpose_kernel(const uint8_t* __restrict__ v,
                                                                     uint8_t* __restrict__ vt,
                                                                     int N, int Npad, int nkb)
{
    constexpr int D = 128;
    __shared__ __align__(16) uint8_t tile[kVtKeys][D];
    const long long bh = blockIdx.x / nkb;
    const int k0 = (blockIdx.x % nkb) * kVtKeys;
    const uint8_t* src = v + (bh * N) * D;
    // in: 64 rows of 8 uint4; rows beyond N are zero
    for (int i = threadIdx.x; i < kVtKeys * D / 16; i += kVtThreads) {
        const int r = i / (D / 16), c = i % (D / 16);
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (k0 + r < N) val = reinterpret_cast<const uint4*>(src + static_cast<long long>(k0 + r) * D)[c];
        reinterpret_cast<uint4*>(tile[r])[c] = val;
    }
    __syncthreads();
    // out: d row `col`, keys [k0 + 16 g, k0 + 16 g + 16); a warp covers 32 consecutive
    // columns of one key group, so its shared-memory reads fall in 8 consecutive words
    uint8_t* dst = vt + bh * D * static_cast<long long>(Npad);
    for (int i = threadIdx.x; i < D * (kVtKeys / 16); i += kVtThreads) {
        const int col = i % D, g = i / D;
        const int kk = k0 + 16 * g;
        if (kk >= Npad) continue;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = 16 * g + 4 * q;
            w[q] = static_cast<uint32_t>(tile[r][col]) | (static_cast<uint32_t>(tile[r + 1][col]) << 8) |
                   (static_cast<uint32_t>(tile[r + 2][col]) << 16) |
                   (static_cast<uint32_t>(tile[r + 3][col]) << 24);
        }
        *reinterpret_cast<uint4*>(dst + static_cast<long long>(col) * Npad + kk) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_vt_transpose(const void* v, void* vt, int BH, int N, int Npad, cudaStream_t st)
{
    const int nkb = (Npad + kVtKeys - 1) / kVtKeys;
    fa_vt_transpose_kernel<<<static_cast<unsigned>(BH) * nkb, kVtThreads, 0, st>>>(
        static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), N, Npad, nkb);
    return cudaGetLastError();
}

}  // namespace fa
