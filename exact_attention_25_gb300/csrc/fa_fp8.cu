// Preparation for the e4m3 forward: V -> V^T [B*Hkv, d, Kpad], one d x Kpad matrix of key
// bytes per (sequence, key/value head), Kpad = the longest sequence's key count rounded up to
// 16, keys past a sequence's end zero.  V enters O += P V as a K-major operand like P, and a
// block of keys always starts at a 16-byte multiple of its row (the tensor-copy rule), also
// for packed sequences that start anywhere.  HBM-bound: one read and one write of V.  Each
// CTA moves 64 keys x 128 bytes of one (sequence, head) through shared memory: 16-byte row
// loads in, 16-byte stores of 16 consecutive keys of one d column out.
#include "fa_common.cuh"

namespace fa {

constexpr int kVtKeys = 64;      // keys per CTA
constexpr int kVtThreads = 256;

// Fixed layout: V is [B, H, N, d] (head index b*H + h); packed: V is [total_k, Hkv, d] and
// sequence b owns the key rows seq_rows(L, b) (offsets clamped to the tensor, as in the
// attention kernels).  v_ext / vt_ext: element extents, tested in checked builds.
template <bool PACKED>
__global__ void __launch_bounds__(kVtThreads)
    fa_vt_transpose_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt, const Layout L,
                           int Kpad, int nkb, long long v_ext, long long vt_ext, int* status)
{
    constexpr int D = 128;
    __shared__ __align__(16) uint8_t tile[kVtKeys][D];
    const int z = static_cast<int>(blockIdx.x) / nkb;  // b * Hkv + hk
    const int b = z / L.Hkv, hk = z % L.Hkv;
    const SeqRows sr = seq_rows<PACKED>(L, b);
    const int k0 = (static_cast<int>(blockIdx.x) % nkb) * kVtKeys;
    // in: 64 key rows of 8 uint4; keys past the sequence's end are zero
    for (int i = threadIdx.x; i < kVtKeys * D / 16; i += kVtThreads) {
        const int r = i / (D / 16), c = i % (D / 16);
        const int key = k0 + r;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (key < sr.nk) {
            const long long off = PACKED
                ? (static_cast<long long>(sr.k0 + key) * L.Hkv + hk) * D
                : (static_cast<long long>(z) * L.Rk + key) * D;
            if (in_extent(off, D, v_ext, status)) val = reinterpret_cast<const uint4*>(v + off)[c];
        }
        reinterpret_cast<uint4*>(tile[r])[c] = val;
    }
    __syncthreads();
    // out: d row `col`, keys [k0 + 16 g, k0 + 16 g + 16); a warp covers 32 consecutive
    // columns of one key group, so its shared-memory reads fall in 8 consecutive words
    const long long base = static_cast<long long>(z) * D * Kpad;
    for (int i = threadIdx.x; i < D * (kVtKeys / 16); i += kVtThreads) {
        const int col = i % D, g = i / D;
        const int kk = k0 + 16 * g;
        if (kk >= Kpad) continue;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = 16 * g + 4 * q;
            w[q] = static_cast<uint32_t>(tile[r][col]) | (static_cast<uint32_t>(tile[r + 1][col]) << 8) |
                   (static_cast<uint32_t>(tile[r + 2][col]) << 16) |
                   (static_cast<uint32_t>(tile[r + 3][col]) << 24);
        }
        const long long off = base + static_cast<long long>(col) * Kpad + kk;
        if (in_extent(off, 16, vt_ext, status))
            *reinterpret_cast<uint4*>(vt + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One CTA per (sequence, key/value head, 64 keys).  L: the call's layout (B, Hkv, Rk, cu_k).
cudaError_t launch_vt_transpose(const void* v, void* vt, const Layout& L, int Kpad, int* status,
                                cudaStream_t st)
{
    const int nkb = (Kpad + kVtKeys - 1) / kVtKeys;
    const long long pairs = static_cast<long long>(L.B) * L.Hkv;
    const bool packed = L.cu_k != nullptr;
    const long long v_ext = static_cast<long long>(L.Rk) * 128 * (packed ? L.Hkv : pairs);
    const long long vt_ext = pairs * 128 * Kpad;
    const unsigned grid = static_cast<unsigned>(pairs * nkb);
    if (packed)
        fa_vt_transpose_kernel<true><<<grid, kVtThreads, 0, st>>>(
            static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), L, Kpad, nkb, v_ext, vt_ext, status);
    else
        fa_vt_transpose_kernel<false><<<grid, kVtThreads, 0, st>>>(
            static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), L, Kpad, nkb, v_ext, vt_ext, status);
    return cudaGetLastError();
}

}  // namespace fa
