// Preparation for the e4m3 forward: V -> V^T [B*Hkv, d, Kpad], one d x Kpad matrix of key
// bytes per (sequence, key/value head), Kpad = the longest sequence's key count rounded up to
// 16, keys past a sequence's end zero.  V enters O += P V as a K-major operand like P, and a
// block of keys always starts at a 16-byte multiple of its row (the tensor-copy rule), also
// for packed sequences that start anywhere.  HBM-bound: one read and one write of V.  Each
// CTA moves 128 keys x 128 bytes of one (sequence, head) through shared memory: 16-byte row
// loads in, 4 x 4 byte-block transposes, 16-byte stores of 16 consecutive keys of one d row
// out.
#include "fa_common.cuh"

namespace fa {

constexpr int kVtKeys = 128;     // keys per CTA
constexpr int kVtThreads = 256;

// Byte transpose of a 4 x 4 block: w[i] holds bytes (i, 0..3) (key row i, four d columns);
// o[j] receives bytes (0..3, j) (d row j, four keys), key i in byte i.
__device__ __forceinline__ void transpose4x4(const uint32_t w[4], uint32_t o[4])
{
    const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140);  // w0.b0 w1.b0 w0.b1 w1.b1
    const uint32_t t1 = __byte_perm(w[0], w[1], 0x7362);  // w0.b2 w1.b2 w0.b3 w1.b3
    const uint32_t t2 = __byte_perm(w[2], w[3], 0x5140);
    const uint32_t t3 = __byte_perm(w[2], w[3], 0x7362);
    o[0] = __byte_perm(t0, t2, 0x5410);
    o[1] = __byte_perm(t0, t2, 0x7632);
    o[2] = __byte_perm(t1, t3, 0x5410);
    o[3] = __byte_perm(t1, t3, 0x7632);
}

// Fixed layout: V is [B, H, N, d] (head index b*H + h); packed: V is [total_k, Hkv, d] and
// sequence b owns the key rows seq_rows(L, b) (offsets clamped to the tensor, as in the
// attention kernels).  v_ext / vt_ext: element extents, tested in checked builds.
// Each thread writes four d rows x 16 keys: 16 32-bit shared loads (four 4 x 4 blocks), 32
// byte permutes, four 16-byte stores.
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
    // in: 128 key rows of 8 uint4; keys past the sequence's end are zero
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
        // 16-byte chunk c of row r sits at chunk c ^ (r / 16 mod 8): the reads below then
        // fall in 32 distinct banks
        reinterpret_cast<uint4*>(tile[r])[c ^ ((r >> 4) & 7)] = val;
    }
    __syncthreads();
    // out: d rows [4 dg, 4 dg + 4), keys [k0 + 16 kg, k0 + 16 kg + 16).  Lane = kg + 8 (dg mod
    // 4), so each 16-byte store of a warp writes four whole 128-byte rows of V^T.
    const int lane = threadIdx.x & 31;
    const int kg = lane & 7, dg = (threadIdx.x >> 5) * 4 + (lane >> 3);
    const int kk = k0 + 16 * kg;
    if (kk >= Kpad) return;
    uint32_t out[4][4];  // [d row j][4-key group q]
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4], o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)  // word dg mod 4 of chunk dg / 4, swizzled by kg
            w[i] = *reinterpret_cast<const uint32_t*>(
                &tile[16 * kg + 4 * q + i][16 * ((dg >> 2) ^ kg) + 4 * (dg & 3)]);
        transpose4x4(w, o);
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j][q] = o[j];
    }
    const long long base = static_cast<long long>(z) * D * Kpad;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const long long off = base + static_cast<long long>(4 * dg + j) * Kpad + kk;
        if (in_extent(off, 16, vt_ext, status))
            *reinterpret_cast<uint4*>(vt + off) = make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
    }
}

// One CTA per (sequence, key/value head, 128 keys).  L: the call's layout (B, Hkv, Rk, cu_k).
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
