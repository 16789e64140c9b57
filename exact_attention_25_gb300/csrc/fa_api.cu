// Host side of the C ABI declared in include/fa.h: argument validation (before any CUDA
// call), TMA tensor-map construction, kernel dispatch and the device status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "fa_common.cuh"
#include "fa_decode.cuh"

namespace fa {
cudaError_t launch_fwd_tc(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const FwdParams& p, cudaStream_t st);
cudaError_t launch_fwd_simt(int d, int is_f32, const FwdParams& p, cudaStream_t st,
                            int num_sms);
cudaError_t launch_bwd_preprocess(int d, int is_f32, const BwdParams& p, cudaStream_t st,
                                  int num_sms);
cudaError_t launch_bwd_simt(int d, int is_f32, const BwdParams& p, cudaStream_t st);
// maps: [0] q, [1] k, [2] v, [3] dout (bf16, 128-row boxes)
cudaError_t launch_bwd_dkv_tc(int d, const CUtensorMap* maps, const BwdParams& p, cudaStream_t st);
cudaError_t launch_bwd_dq_tc(int d, const CUtensorMap* maps, const BwdParams& p, cudaStream_t st,
                             bool after_dkv);
cudaError_t launch_decode(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const DecodeParams& p, cudaStream_t st,
                          int num_sms);
cudaError_t launch_fwd_fp8_tc(const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tvt, const FwdParams& p, cudaStream_t st);
cudaError_t launch_vt_transpose(const void* v, void* vt, const Layout& L, int Kpad, int* status,
                                cudaStream_t st);

// Device status word written by bounded waits that give up (0 = fine).
__device__ int g_status_word;
}  // namespace fa

namespace {

thread_local std::string t_last_error;
unsigned long long g_wait_limit_ns = 2000000000ull;
int g_debug_flags = 0;

int fail(int code, const std::string& what)
{
    t_last_error = what;
    return code;
}

int cuda_fail(cudaError_t e, const char* where)
{
    return fail(FA_ERR_LAUNCH, std::string(where) + ": " + cudaGetErrorString(e));
}

struct DeviceInfo {
    bool ready = false;
    int major = 0, minor = 0, sms = 0;
    int* status = nullptr;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

int device_info(DeviceInfo** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(FA_ERR_LAUNCH, "device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        if ((e = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            (e = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
            (e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)))
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (di.major != 10 || di.minor != 3)
            return fail(FA_ERR_UNSUPPORTED_DEVICE,
                        "this build targets sm_103a (compute capability 10.3) only");
        void* ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, fa::g_status_word)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(status)");
        di.status = static_cast<int*>(ptr);
        di.ready = true;
    }
    *out = &di;
    return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return FA_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled entry point not available");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FA_OK;
}

// 3-D view of a bf16 tensor for 128-row tiles of one head; box = 64 columns (one 128-byte
// swizzle panel) x `rows` rows x 1 head.  Fixed layout [heads, R, d]: dimensions (d, R, heads);
// packed layout [R, heads, d] (token by token): dimensions (d, heads, R).  Rows beyond R read
// as zero.
// rs, hs: element strides of a row and of a head index.
int make_map(CUtensorMap* m, const void* base, long long heads, long long R, int d, int rows,
             bool packed, long long rs, long long hs)
{
    const cuuint64_t dd = static_cast<cuuint64_t>(d);
    const cuuint64_t nh = static_cast<cuuint64_t>(heads), nr = static_cast<cuuint64_t>(R);
    cuuint64_t dims[3] = {dd, packed ? nh : nr, packed ? nr : nh};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(packed ? hs : rs) * 2,
                             static_cast<cuuint64_t>(packed ? rs : hs) * 2};
    cuuint32_t box[3] = {64, packed ? 1u : static_cast<cuuint32_t>(rows),
                         packed ? static_cast<cuuint32_t>(rows) : 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed with code " + std::to_string(r));
    return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int N, int d, float scale, int causal, int dtype)
{
    if (dtype != FA_BF16 && dtype != FA_F32) return fail(FA_ERR_INVALID_ARG, "dtype must be FA_BF16 or FA_F32");
    if (B < 1 || H < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, H and N must be >= 1");
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED_D, "d must be 64 or 128");
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    const long long elems = static_cast<long long>(B) * H * N * d;
    if (elems >= (1LL << 31)) return fail(FA_ERR_TOO_LARGE, "B*H*N*d must be < 2^31");
    return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The bytes [p, p + n) of one tensor of a call.
struct Span {
    const void* p;
    size_t n;
};

bool spans_meet(const Span& a, const Span& b)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Whether an output shares a byte with another output, an input or the workspace.  The
// backward's kernels overlap in time (dQ runs in the tail of dK/dV), so such a call would race.
bool outputs_overlap(const Span* out, int nout, const Span* in, int nin)
{
    for (int i = 0; i < nout; ++i) {
        for (int j = i + 1; j < nout; ++j)
            if (spans_meet(out[i], out[j])) return true;
        for (int j = 0; j < nin; ++j)
            if (spans_meet(out[i], in[j])) return true;
    }
    return false;
}

const char* const kOverlapMsg =
    "dq, dk and dv must not overlap one another, an input or the workspace";

// Element strides (row, head index) of the eight tensors of a call, in the order
// q, k, v, o, dout, dq, dk, dv.
struct Strides {
    long long rs[8], hs[8];
};
enum { kQ = 0, kK, kV, kO, kDO, kDQ, kDK, kDV };

// The strides the kernels address directly go into the layout; q, k, v, dout go into maps.
// Also sets the element extents that checked builds test accesses against: the smallest
// buffer holding every row of every head index at those strides (R rows of each head index;
// the fixed-length layout's head index runs over B*H, the packed one's over H).  The layout's
// sizes (cu_q, B, H, Hkv, Rq, Rk) must be set first.
void put_strides(fa::Layout& L, const Strides& st, int d)
{
    L.o_rs = st.rs[kO]; L.o_hs = st.hs[kO];
    L.do_rs = st.rs[kDO]; L.do_hs = st.hs[kDO];
    L.dq_rs = st.rs[kDQ]; L.dq_hs = st.hs[kDQ];
    L.dk_rs = st.rs[kDK]; L.dk_hs = st.hs[kDK];
    L.dv_rs = st.rs[kDV]; L.dv_hs = st.hs[kDV];
    const long long bq = L.cu_q ? 1 : L.B;
    const long long hq = bq * L.H, hk = bq * L.Hkv;
    // the watchdog test hook's companion: every extent one row short
    const long long cut = (g_debug_flags & fa::kDebugShrinkExtents) ? 1 : 0;
    auto ext = [&](int t, long long heads, long long rows) {
        return rows < 1 ? 0 : (rows - 1) * st.rs[t] + (heads - 1) * st.hs[t] + d - cut * st.rs[t];
    };
    L.o_ext = ext(kO, hq, L.Rq);
    L.do_ext = ext(kDO, hq, L.Rq);
    L.dq_ext = ext(kDQ, hq, L.Rq);
    L.dk_ext = ext(kDK, hk, L.Rk);
    L.dv_ext = ext(kDV, hk, L.Rk);
    L.stat_ext = hq * L.Rq - cut;
}

// Fixed-length entry points: [B, H, N, d] for every tensor, [B, H, N] statistics.
Strides fixed_strides(int N, int d)
{
    Strides st;
    for (int t = 0; t < 8; ++t) {
        st.rs[t] = d;
        st.hs[t] = static_cast<long long>(N) * d;
    }
    return st;
}

fa::Layout fixed_layout(int B, int H, int N, int d)
{
    fa::Layout L{};
    L.cu_q = L.cu_k = nullptr;
    L.B = B; L.H = H; L.Hkv = H;
    L.Nq = L.Nk = N;
    L.Rq = L.Rk = N;
    L.order_group = 1;
    put_strides(L, fixed_strides(N, d), d);
    return L;
}

// Heads per group of the tensor-core kernels' tile order (tile_order): under the causal mask,
// as many heads as keep the rows that one head's tiles stream (K and V, or Q and dO: 4 N d bytes
// in bf16) within 32 MB of L2, at most 16; without the mask every tile costs the same and the
// plain head-major order (1) keeps the fewest heads resident.
int order_group(int N, int d, int causal)
{
    if (!causal) return 1;
    const long long per_head = 4LL * N * d;
    const long long g = (32LL << 20) / (per_head > 0 ? per_head : 1);
    return static_cast<int>(g < 1 ? 1 : (g > 16 ? 16 : g));
}

// The four bf16 maps of the tensor-core kernels: q, k, v, and (backward) dout.
int make_maps(CUtensorMap* maps, const void* q, const void* k, const void* v, const void* dout,
              const fa::Layout& L, int d, const Strides& st)
{
    int rc = get_encoder();
    if (rc) return rc;
    const bool packed = L.cu_q != nullptr;
    const long long nhq = packed ? L.H : static_cast<long long>(L.B) * L.H;
    const long long nhk = packed ? L.Hkv : static_cast<long long>(L.B) * L.Hkv;
    if ((rc = make_map(&maps[0], q, nhq, L.Rq, d, 128, packed, st.rs[kQ], st.hs[kQ])) ||
        (rc = make_map(&maps[1], k, nhk, L.Rk, d, 128, packed, st.rs[kK], st.hs[kK])) ||
        (rc = make_map(&maps[2], v, nhk, L.Rk, d, 128, packed, st.rs[kV], st.hs[kV])))
        return rc;
    if (dout && (rc = make_map(&maps[3], dout, nhq, L.Rq, d, 128, packed, st.rs[kDO],
                               st.hs[kDO])))
        return rc;
    return FA_OK;
}

int fwd_entry(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int d, float scale, int causal, int dtype, int impl, void* stream)
{
    int rc = check_common(B, H, N, d, scale, causal, dtype);
    if (rc) return rc;
    if (impl != 0 && impl != 1) return fail(FA_ERR_INVALID_ARG, "impl must be 0 or 1");
    if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA_ERR_MISALIGNED, "q, k, v, o must be 16-byte aligned (lse 4-byte)");
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    fa::FwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    p.N = N; p.BH = B * H; p.scale = scale; p.scale_log2 = scale * fa::kLog2e;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    p.L = fixed_layout(B, H, N, d);
    p.L.order_group = order_group(N, d, causal);
    cudaError_t e;
    if (dtype == FA_F32 || impl == 1) {
        e = fa::launch_fwd_simt(d, dtype == FA_F32, p, st, di->sms);
    } else {
        CUtensorMap maps[4];
        if ((rc = make_maps(maps, q, k, v, nullptr, p.L, d, fixed_strides(N, d)))) return rc;
        e = fa::launch_fwd_tc(d, maps[0], maps[1], maps[2], p, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return FA_OK;
}

int bwd_entry(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
              float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
              int impl, int stage, void* stream)
{
    int rc = check_common(B, H, N, d, scale, causal, dtype);
    if (rc) return rc;
    if (impl != 0 && impl != 1) return fail(FA_ERR_INVALID_ARG, "impl must be 0 or 1");
    if (stage < -1 || stage > 2) return fail(FA_ERR_INVALID_ARG, "stage must be 0, 1 or 2");
    if (stage >= 0 && (dtype != FA_BF16 || impl != 0))
        return fail(FA_ERR_INVALID_ARG, "staged backward is the bf16 tensor-core path only");
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
        return fail(FA_ERR_INVALID_ARG, "every tensor pointer must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(FA_ERR_MISALIGNED, "tensors must be 16-byte aligned (lse 4-byte)");
    const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
    if (!workspace || workspace_bytes < need)
        return fail(FA_ERR_WORKSPACE, "workspace must hold " + std::to_string(need) + " bytes");
    if (!aligned16(workspace)) return fail(FA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    {
        const size_t tb = static_cast<size_t>(B) * H * N * d * (dtype == FA_F32 ? 4 : 2);
        const size_t sb = static_cast<size_t>(B) * H * N * 4;
        const Span outs[3] = {{dq, tb}, {dk, tb}, {dv, tb}};
        const Span ins[7] = {{q, tb}, {k, tb}, {v, tb}, {o, tb}, {dout, tb}, {lse, sb},
                             {workspace, need}};
        if (outputs_overlap(outs, 3, ins, 7)) return fail(FA_ERR_INVALID_ARG, kOverlapMsg);
    }
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    fa::BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    const size_t rows = static_cast<size_t>(B) * H * N;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.delta = reinterpret_cast<float*>(ws);
    p.lse2 = reinterpret_cast<float*>(ws + align256(rows * 4));
    p.N = N; p.BH = B * H; p.scale = scale; p.scale_log2 = scale * fa::kLog2e;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    p.L = fixed_layout(B, H, N, d);
    p.L.order_group = order_group(N, d, causal);
    const int is_f32 = dtype == FA_F32;
    cudaError_t e = cudaSuccess;
    if (stage <= 0) {
        e = fa::launch_bwd_preprocess(d, is_f32, p, st, di->sms);
        if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
        if (stage == 0) return FA_OK;
    }
    if (is_f32 || impl == 1) {
        e = fa::launch_bwd_simt(d, is_f32, p, st);
    } else {
        // maps: q, k, v, dout (all 128-row boxes)
        CUtensorMap maps[4];
        if ((rc = make_maps(maps, q, k, v, dout, p.L, d, fixed_strides(N, d)))) return rc;
        if (stage < 0 || stage == 1) e = fa::launch_bwd_dkv_tc(d, maps, p, st);
        if (e == cudaSuccess && (stage < 0 || stage == 2)) e = fa::launch_bwd_dq_tc(d, maps, p, st, stage < 0);
    }
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, int dtype, void* stream)
{
    return fwd_entry(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, 0, stream);
}

int fa_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, float scale, int causal, int dtype, int impl, void* stream)
{
    return fwd_entry(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, impl, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d)
{
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    const size_t rows = static_cast<size_t>(B) * H * N;
    return 2 * align256(rows * 4) + 256;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
           void* stream)
{
    return bwd_entry(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                     workspace, workspace_bytes, 0, -1, stream);
}

int fa_bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                int impl, void* stream)
{
    return bwd_entry(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                     workspace, workspace_bytes, impl, -1, stream);
}

int fa_bwd_stage(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                 int stage, void* stream)
{
    if (stage < 0 || stage > 2) return fail(FA_ERR_INVALID_ARG, "stage must be 0, 1 or 2");
    return bwd_entry(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                     workspace, workspace_bytes, 0, stage, stream);
}

int fa_device_status(void* stream)
{
    DeviceInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int word = 0;
    if ((e = cudaMemcpy(&word, di->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "reading the status word");
    if (word == 0) return FA_OK;
    const int zero = 0;
    if ((e = cudaMemcpy(di->status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "clearing the status word");
    if (word == fa::kStatusOutOfBounds)
        return fail(FA_ERR_OUT_OF_BOUNDS, "a bounds check failed; the access was skipped");
    return fail(FA_ERR_DEVICE_TIMEOUT, "bounded device wait expired at site " + std::to_string(word));
}

void fa_set_wait_limit_ns(unsigned long long ns)
{
    g_wait_limit_ns = ns < 1000000ull ? 1000000ull : ns;
}

void fa_debug_set_flags(int flags) { g_debug_flags = flags; }

int fa_checked_build(void)
{
#ifdef FA_CHECKED
    return 1;
#else
    return 0;
#endif
}

const char* fa_status_string(int code)
{
    switch (code) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED_D: return "FA_ERR_UNSUPPORTED_D";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
        case FA_ERR_TOO_LARGE: return "FA_ERR_TOO_LARGE";
        case FA_ERR_UNSUPPORTED_DEVICE: return "FA_ERR_UNSUPPORTED_DEVICE";
        case FA_ERR_OUT_OF_BOUNDS: return "FA_ERR_OUT_OF_BOUNDS";
        default: return "FA_ERR_UNKNOWN";
    }
}

const char* fa_last_error(void) { return t_last_error.c_str(); }

int fa_causal_block_counts(int q_block, int Br, int Bc, int N, int* n_full, int* n_masked)
{
    if (q_block < 0 || Br < 1 || Bc < 1 || N < 1 || !n_full || !n_masked ||
        static_cast<long long>(q_block) * Br >= N)
        return fail(FA_ERR_INVALID_ARG, "bad block arguments");
    const int q0 = q_block * Br, q1 = (q0 + Br < N) ? q0 + Br : N;
    int nf = 0, nm = 0;
    for (int k0 = 0; k0 < N; k0 += Bc) {
        const int k1 = (k0 + Bc < N) ? k0 + Bc : N;
        const int c = fa::causal_tile_class(q0, q1, k0, k1);
        nf += c == fa::kTileFull;
        nm += c == fa::kTileMasked;
    }
    *n_full = nf;
    *n_masked = nm;
    return FA_OK;
}

int fa_tile_order(int id, int heads, int nblk, int gsize, int* head, int* rank)
{
    if (heads < 1 || nblk < 1 || gsize < 1 || id < 0 ||
        static_cast<long long>(id) >= static_cast<long long>(heads) * nblk || !head || !rank)
        return fail(FA_ERR_INVALID_ARG, "bad tile-order arguments");
    fa::tile_order(id, heads, nblk, gsize, *head, *rank);
    return FA_OK;
}

int fa_order_group(int N, int d, int causal) { return order_group(N, d, causal); }

const char* fa_version(void) { return "fa-gb300 0.1 (sm_103a)"; }

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Fixed-length batches with grouped key/value heads and Nq != Nk (fa_fwd_gqa, fa_bwd_gqa).
// ---------------------------------------------------------------------------------------
namespace {

int check_gqa(int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal)
{
    if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1)
        return fail(FA_ERR_INVALID_ARG, "B, H, Hkv, Nq and Nk must be >= 1");
    if (H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H must be a multiple of Hkv");
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED_D, "d must be 64 or 128");
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    if (static_cast<long long>(B) * H * Nq * d >= (1LL << 31) ||
        static_cast<long long>(B) * Hkv * Nk * d >= (1LL << 31))
        return fail(FA_ERR_TOO_LARGE, "B*H*Nq*d and B*Hkv*Nk*d must be < 2^31");
    return FA_OK;
}

// [B, H, Nq, d] queries, [B, Hkv, Nk, d] keys and values, [B, H, Nq] statistics.
fa::Layout gqa_layout(int B, int H, int Hkv, int Nq, int Nk, int d, Strides* st)
{
    for (int t = 0; t < 8; ++t) {
        const bool kside = t == kK || t == kV || t == kDK || t == kDV;
        st->rs[t] = d;
        st->hs[t] = static_cast<long long>(kside ? Nk : Nq) * d;
    }
    fa::Layout L{};
    L.cu_q = L.cu_k = nullptr;
    L.B = B; L.H = H; L.Hkv = Hkv;
    L.Nq = Nq; L.Nk = Nk;
    L.Rq = Nq; L.Rk = Nk;
    L.order_group = 1;
    put_strides(L, *st, d);
    return L;
}

}  // namespace

extern "C" int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                          void* stream)
{
    int rc = check_gqa(B, H, Hkv, Nq, Nk, d, scale, causal);
    if (rc) return rc;
    if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA_ERR_MISALIGNED, "q, k, v, o must be 16-byte aligned (lse 4-byte)");
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    fa::FwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    p.N = Nq; p.BH = B * H; p.scale = scale; p.scale_log2 = scale * fa::kLog2e;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    Strides st;
    p.L = gqa_layout(B, H, Hkv, Nq, Nk, d, &st);
    p.L.order_group = order_group(Nk, d, causal);
    CUtensorMap maps[4];
    if ((rc = make_maps(maps, q, k, v, nullptr, p.L, d, st))) return rc;
    cudaError_t e = fa::launch_fwd_tc(d, maps[0], maps[1], maps[2], p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return FA_OK;
}

extern "C" int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                          int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                          void* workspace, size_t workspace_bytes, void* stream)
{
    int rc = check_gqa(B, H, Hkv, Nq, Nk, d, scale, causal);
    if (rc) return rc;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
        return fail(FA_ERR_INVALID_ARG, "every tensor pointer must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(FA_ERR_MISALIGNED, "tensors must be 16-byte aligned (lse 4-byte)");
    const size_t need = fa_bwd_workspace_bytes(B, H, Nq, d);
    if (!workspace || workspace_bytes < need)
        return fail(FA_ERR_WORKSPACE, "workspace must hold " + std::to_string(need) + " bytes");
    if (!aligned16(workspace)) return fail(FA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    {
        const size_t tq = static_cast<size_t>(B) * H * Nq * d * 2;
        const size_t tk = static_cast<size_t>(B) * Hkv * Nk * d * 2;
        const size_t sb = static_cast<size_t>(B) * H * Nq * 4;
        const Span outs[3] = {{dq, tq}, {dk, tk}, {dv, tk}};
        const Span ins[7] = {{q, tq}, {k, tk}, {v, tk}, {o, tq}, {dout, tq}, {lse, sb},
                             {workspace, need}};
        if (outputs_overlap(outs, 3, ins, 7)) return fail(FA_ERR_INVALID_ARG, kOverlapMsg);
    }
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    fa::BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    const size_t rows = static_cast<size_t>(B) * H * Nq;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.delta = reinterpret_cast<float*>(ws);
    p.lse2 = reinterpret_cast<float*>(ws + align256(rows * 4));
    p.N = Nq; p.BH = B * H; p.scale = scale; p.scale_log2 = scale * fa::kLog2e;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    Strides st;
    p.L = gqa_layout(B, H, Hkv, Nq, Nk, d, &st);
    p.L.order_group = order_group(Nk, d, causal);
    CUtensorMap maps[4];
    if ((rc = make_maps(maps, q, k, v, dout, p.L, d, st))) return rc;
    cudaError_t e = fa::launch_bwd_preprocess(d, 0, p, cs, di->sms);
    if (e == cudaSuccess) e = fa::launch_bwd_dkv_tc(d, maps, p, cs);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_tc(d, maps, p, cs, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return FA_OK;
}

// ---------------------------------------------------------------------------------------
// Packed variable-length batches with grouped key/value heads (fa_fwd_varlen, fa_bwd_varlen).
// ---------------------------------------------------------------------------------------
namespace {

int check_varlen(const int* cu_q, const int* cu_k, int B, int* max_q, int* max_k, int total_q,
                 int total_k, int H, int Hkv, int d, float scale, int causal)
{
    if (B < 1 || H < 1 || Hkv < 1) return fail(FA_ERR_INVALID_ARG, "B, H and Hkv must be >= 1");
    if (H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H must be a multiple of Hkv");
    if (total_q < 1 || total_k < 1 || *max_q < 1 || *max_k < 1)
        return fail(FA_ERR_INVALID_ARG, "total_q, total_k, max_seqlen_q and max_seqlen_k must be >= 1");
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED_D, "d must be 64 or 128");
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    if (!cu_q || !cu_k) return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must be non-null");
    if ((reinterpret_cast<uintptr_t>(cu_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_k) & 3u))
        return fail(FA_ERR_MISALIGNED, "cu_seqlens_q and cu_seqlens_k must be 4-byte aligned");
    if (static_cast<long long>(total_q) * H * d >= (1LL << 31) ||
        static_cast<long long>(total_k) * Hkv * d >= (1LL << 31))
        return fail(FA_ERR_TOO_LARGE, "total_q*H*d and total_k*Hkv*d must be < 2^31");
    // no sequence is longer than its packed tensor
    if (*max_q > total_q) *max_q = total_q;
    if (*max_k > total_k) *max_k = total_k;
    if (static_cast<long long>(B) * H * ((*max_q + 127) / 128) >= (1LL << 31) ||
        static_cast<long long>(B) * Hkv * ((*max_k + 127) / 128) >= (1LL << 31))
        return fail(FA_ERR_TOO_LARGE, "B*H*ceil(max_seqlen/128) must be < 2^31");
    return FA_OK;
}

// Contiguous packed tensors: q-side [total_q, H, d], k-side [total_k, Hkv, d].
Strides packed_strides(int H, int Hkv, int d)
{
    Strides st;
    for (int t = 0; t < 8; ++t) {
        const bool kside = t == kK || t == kV || t == kDK || t == kDV;
        st.rs[t] = static_cast<long long>(kside ? Hkv : H) * d;
        st.hs[t] = d;
    }
    return st;
}

// Caller strides: `n` (row, head) pairs in the order q, k, v, o[, dout, dq, dk, dv].  Each must
// be positive and a multiple of 8 elements (16 bytes, for the tensor maps and the 16-byte
// stores), and a head must not be wider than its row step (tensors stored token by token).
int read_strides(const long long* user, int n, int H, int Hkv, int d, Strides* st)
{
    *st = packed_strides(H, Hkv, d);
    if (!user) return fail(FA_ERR_INVALID_ARG, "strides must be non-null");
    for (int t = 0; t < n; ++t) {
        const long long rs = user[2 * t], hs = user[2 * t + 1];
        if (rs <= 0 || hs <= 0 || (rs % 8) || (hs % 8))
            return fail(FA_ERR_MISALIGNED, "strides must be positive multiples of 8 elements");
        if (hs < d || rs < hs)
            return fail(FA_ERR_INVALID_ARG, "each head's d elements must fit within its head step, "
                                            "and the head step within the row step");
        st->rs[t] = rs;
        st->hs[t] = hs;
    }
    return FA_OK;
}

fa::Layout packed_layout(const int* cu_q, const int* cu_k, int B, int max_q, int max_k,
                         int total_q, int total_k, int H, int Hkv, int d, const Strides& st)
{
    fa::Layout L{};
    L.cu_q = cu_q; L.cu_k = cu_k;
    L.B = B; L.H = H; L.Hkv = Hkv;
    L.Nq = max_q; L.Nk = max_k;
    L.Rq = total_q; L.Rk = total_k;
    L.order_group = 1;  // sequences of different lengths: head-major
    put_strides(L, st, d);
    return L;
}

int fwd_varlen_entry(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_q, const int* cu_k, int B, int max_q, int max_k, int total_q,
                     int total_k, int H, int Hkv, int d, float scale, int causal,
                     const long long* user_strides, void* stream)
{
    int rc = check_varlen(cu_q, cu_k, B, &max_q, &max_k, total_q, total_k, H, Hkv, d, scale,
                          causal);
    if (rc) return rc;
    if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA_ERR_MISALIGNED, "q, k, v, o must be 16-byte aligned (lse 4-byte)");
    Strides st = packed_strides(H, Hkv, d);
    if (user_strides && (rc = read_strides(user_strides, 4, H, Hkv, d, &st))) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    fa::FwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    p.N = total_q; p.BH = H; p.scale = scale; p.scale_log2 = scale * fa::kLog2e;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    p.L = packed_layout(cu_q, cu_k, B, max_q, max_k, total_q, total_k, H, Hkv, d, st);
    CUtensorMap maps[4];
    if ((rc = make_maps(maps, q, k, v, nullptr, p.L, d, st))) return rc;
    cudaError_t e = fa::launch_fwd_tc(d, maps[0], maps[1], maps[2], p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return FA_OK;
}

int bwd_varlen_entry(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, const int* cu_q,
                     const int* cu_k, int B, int max_q, int max_k, int total_q, int total_k,
                     int H, int Hkv, int d, float scale, int causal,
                     const long long* user_strides, void* workspace, size_t workspace_bytes,
                     void* stream)
{
    int rc = check_varlen(cu_q, cu_k, B, &max_q, &max_k, total_q, total_k, H, Hkv, d, scale,
                          causal);
    if (rc) return rc;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
        return fail(FA_ERR_INVALID_ARG, "every tensor pointer must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(FA_ERR_MISALIGNED, "tensors must be 16-byte aligned (lse 4-byte)");
    Strides st = packed_strides(H, Hkv, d);
    if (user_strides && (rc = read_strides(user_strides, 8, H, Hkv, d, &st))) return rc;
    const size_t need = fa_bwd_varlen_workspace_bytes(total_q, H, d);
    if (!workspace || workspace_bytes < need)
        return fail(FA_ERR_WORKSPACE, "workspace must hold " + std::to_string(need) + " bytes");
    if (!aligned16(workspace)) return fail(FA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    if (!user_strides) {  // (strided views may interleave in one buffer: not checked)
        const size_t tq = static_cast<size_t>(total_q) * H * d * 2;
        const size_t tk = static_cast<size_t>(total_k) * Hkv * d * 2;
        const size_t sb = static_cast<size_t>(total_q) * H * 4;
        const Span outs[3] = {{dq, tq}, {dk, tk}, {dv, tk}};
        const Span ins[7] = {{q, tq}, {k, tk}, {v, tk}, {o, tq}, {dout, tq}, {lse, sb},
                             {workspace, need}};
        if (outputs_overlap(outs, 3, ins, 7)) return fail(FA_ERR_INVALID_ARG, kOverlapMsg);
    }
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    fa::BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    const size_t rows = static_cast<size_t>(H) * total_q;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.delta = reinterpret_cast<float*>(ws);
    p.lse2 = reinterpret_cast<float*>(ws + align256(rows * 4));
    p.N = total_q; p.BH = H; p.scale = scale; p.scale_log2 = scale * fa::kLog2e;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    p.L = packed_layout(cu_q, cu_k, B, max_q, max_k, total_q, total_k, H, Hkv, d, st);
    CUtensorMap maps[4];
    if ((rc = make_maps(maps, q, k, v, dout, p.L, d, st))) return rc;
    cudaError_t e = fa::launch_bwd_preprocess(d, 0, p, cs, di->sms);
    if (e == cudaSuccess) e = fa::launch_bwd_dkv_tc(d, maps, p, cs);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_tc(d, maps, p, cs, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                             int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int H,
                             int Hkv, int d, float scale, int causal, void* stream)
{
    return fwd_varlen_entry(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, max_seqlen_q,
                            max_seqlen_k, total_q, total_k, H, Hkv, d, scale, causal, nullptr,
                            stream);
}

extern "C" int fa_fwd_varlen_strided(const void* q, const void* k, const void* v, void* o,
                                     float* lse, const long long* strides,
                                     const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                                     int max_seqlen_q, int max_seqlen_k, int total_q,
                                     int total_k, int H, int Hkv, int d, float scale, int causal,
                                     void* stream)
{
    if (!strides) return fail(FA_ERR_INVALID_ARG, "strides must be non-null");
    return fwd_varlen_entry(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, max_seqlen_q,
                            max_seqlen_k, total_q, total_k, H, Hkv, d, scale, causal, strides,
                            stream);
}

extern "C" size_t fa_bwd_varlen_workspace_bytes(int total_q, int H, int d)
{
    if (total_q < 1 || H < 1 || (d != 64 && d != 128)) return 0;
    const size_t rows = static_cast<size_t>(H) * total_q;
    return 2 * align256(rows * 4) + 256;
}

extern "C" int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                             int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int H,
                             int Hkv, int d, float scale, int causal, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    return bwd_varlen_entry(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B,
                            max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale,
                            causal, nullptr, workspace, workspace_bytes, stream);
}

extern "C" int fa_bwd_varlen_strided(const void* q, const void* k, const void* v, const void* o,
                                     const void* dout, const float* lse, void* dq, void* dk,
                                     void* dv, const long long* strides, const int* cu_seqlens_q,
                                     const int* cu_seqlens_k, int B, int max_seqlen_q,
                                     int max_seqlen_k, int total_q, int total_k, int H, int Hkv,
                                     int d, float scale, int causal, void* workspace,
                                     size_t workspace_bytes, void* stream)
{
    if (!strides) return fail(FA_ERR_INVALID_ARG, "strides must be non-null");
    return bwd_varlen_entry(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B,
                            max_seqlen_q, max_seqlen_k, total_q, total_k, H, Hkv, d, scale,
                            causal, strides, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------------------
// Split-KV decode (fa_decode_num_splits, fa_decode_workspace_bytes, fa_fwd_decode).
// ---------------------------------------------------------------------------------------
namespace {

constexpr int kDecodeMaxSplits = 256;

size_t decode_part_o_bytes(int total_q, int H, int d, int splits)
{
    return align256(static_cast<size_t>(splits) * total_q * H * d * 4);
}

}  // namespace

extern "C" int fa_decode_splits_for(int B, int Hkv, int max_seqlen_k, int num_sms)
{
    if (B < 1 || Hkv < 1 || max_seqlen_k < 1 || num_sms < 1)
        return fail(FA_ERR_INVALID_ARG, "B, Hkv, max_seqlen_k and num_sms must be >= 1");
    // One wave: the largest split count whose CTAs (B * Hkv * splits, one per SM) all run at
    // once, keeping at least 8 key blocks per split.  Once enough CTAs stream (each keeps about
    // 200 KB of loads in flight), the HBM time is the same for any split count; a second wave
    // costs its CTAs their set-up and pipeline fill again, and every extra range costs the
    // combine a partial result.  Measured on GB300 (B = 8, Hkv = 8, d = 128): 2 splits over
    // 8 K, 16 K and 32 K keys ran 10-18 % faster than the 7-19 that filled whole waves.
    const long long units = static_cast<long long>(B) * Hkv;
    const int nblk = static_cast<int>((static_cast<long long>(max_seqlen_k) + 127) / 128);
    const int smax = std::max(1, std::min(kDecodeMaxSplits, nblk / 8));
    const long long fit = std::max(1LL, static_cast<long long>(num_sms) / units);
    return static_cast<int>(std::min<long long>(smax, fit));
}

extern "C" int fa_decode_num_splits(int B, int Hkv, int max_seqlen_k)
{
    if (B < 1 || Hkv < 1 || max_seqlen_k < 1) return fail(FA_ERR_INVALID_ARG, "B, Hkv and max_seqlen_k must be >= 1");
    DeviceInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc) return rc;
    return fa_decode_splits_for(B, Hkv, max_seqlen_k, di->sms);
}

extern "C" size_t fa_decode_workspace_bytes(int total_q, int H, int d, int num_splits)
{
    if (total_q < 1 || H < 1 || (d != 64 && d != 128) || num_splits < 1 ||
        num_splits > kDecodeMaxSplits)
        return 0;
    if (num_splits == 1) return 0;
    return decode_part_o_bytes(total_q, H, d, num_splits) +
           align256(static_cast<size_t>(num_splits) * H * total_q * 4) + 256;
}

extern "C" int fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                             int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int H,
                             int Hkv, int d, float scale, int causal, int num_splits,
                             void* workspace, size_t workspace_bytes, void* stream)
{
    int rc = check_varlen(cu_seqlens_q, cu_seqlens_k, B, &max_seqlen_q, &max_seqlen_k, total_q,
                          total_k, H, Hkv, d, scale, causal);
    if (rc) return rc;
    // The rows of a CTA are G query heads of a group times max_seqlen_q queries, at most 128:
    // G is the largest divisor of the group size H / Hkv that fits.
    if (max_seqlen_q > 128)
        return fail(FA_ERR_INVALID_ARG, "max_seqlen_q must be <= 128 for the decode kernel; use "
                                        "fa_fwd_varlen");
    const int group = H / Hkv;
    int G = 1;
    for (int g = 1; g <= group; ++g)
        if (group % g == 0 && g * max_seqlen_q <= 128) G = g;
    if (num_splits < 1 || num_splits > kDecodeMaxSplits)
        return fail(FA_ERR_INVALID_ARG, "num_splits must be in [1, " +
                                            std::to_string(kDecodeMaxSplits) + "]");
    if (static_cast<long long>(B) * Hkv * (group / G) * num_splits >= (1LL << 31))
        return fail(FA_ERR_TOO_LARGE, "B * H / G * num_splits must be < 2^31");
    if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA_ERR_MISALIGNED, "q, k, v, o must be 16-byte aligned (lse 4-byte)");
    const size_t need = fa_decode_workspace_bytes(total_q, H, d, num_splits);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return fail(FA_ERR_WORKSPACE, "workspace must hold " + std::to_string(need) + " bytes");
        if (!aligned16(workspace)) return fail(FA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    }
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    fa::DecodeParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    if (need > 0) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        p.o_part = reinterpret_cast<float*>(ws);
        p.lse_part = reinterpret_cast<float*>(ws + decode_part_o_bytes(total_q, H, d, num_splits));
    }
    p.splits = num_splits; p.G = G; p.head_chunks = group / G; p.q_box = max_seqlen_q;
    p.scale_log2 = scale * fa::kLog2e; p.causal = causal;
    p.status = di->status; p.wait_limit_ns = g_wait_limit_ns; p.debug_flags = g_debug_flags;
    p.part_ext = need > 0 ? static_cast<long long>(num_splits) * total_q * H * d -
                                ((g_debug_flags & fa::kDebugShrinkExtents) ? d : 0)
                          : 0;
    const Strides st = packed_strides(H, Hkv, d);
    p.L = packed_layout(cu_seqlens_q, cu_seqlens_k, B, max_seqlen_q, max_seqlen_k, total_q,
                        total_k, H, Hkv, d, st);
    if ((rc = get_encoder())) return rc;
    // Q: (d, H, total_q) with a box of (64 columns, G heads, max_seqlen_q tokens), so one copy
    // brings the G x nq query rows of a CTA; K, V as fa_fwd_varlen.
    CUtensorMap maps[4];
    {
        const cuuint64_t dd = static_cast<cuuint64_t>(d);
        cuuint64_t dims[3] = {dd, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(total_q)};
        cuuint64_t strides[2] = {dd * 2, static_cast<cuuint64_t>(H) * dd * 2};
        cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(max_seqlen_q)};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = g_encode(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed with code " + std::to_string(r));
    }
    if ((rc = make_map(&maps[1], k, Hkv, total_k, d, 128, true, st.rs[kK], st.hs[kK])) ||
        (rc = make_map(&maps[2], v, Hkv, total_k, d, 128, true, st.rs[kV], st.hs[kV])))
        return rc;
    cudaError_t e = fa::launch_decode(d, maps[0], maps[1], maps[2], p,
                                      static_cast<cudaStream_t>(stream), di->sms);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return FA_OK;
}

// ---------------------------------------------------------------------------------------
// fa_bwd_noalloc: the backward with its scratch in a fixed device array of this library.
// ---------------------------------------------------------------------------------------
namespace {

constexpr long long kNoallocMaxRows = 1LL << 20;  // largest B*H*N accepted
constexpr size_t kNoallocBytes = 2 * static_cast<size_t>(kNoallocMaxRows) * 4 + 256;

// Delta and the base-2 LSE for up to kNoallocMaxRows rows, in the layout of fa_bwd's
// workspace.  Every device that loads the library holds these 8 MiB until the process exits.
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoallocBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev_ptr[64] = {};

// Device address of g_bwd_scratch on the current device, looked up once per device.  In host
// code the symbol names a host-side shadow, not device memory, so it is never passed as is.
int scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(FA_ERR_LAUNCH, "device index out of range");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_dev_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return cuda_fail(e, "cudaGetSymbolAddress(backward scratch)");
        g_scratch_dev_ptr[dev] = ptr;
    }
    *out = g_scratch_dev_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, int dtype,
                              void* stream)
{
    int rc = check_common(B, H, N, d, scale, causal, dtype);
    if (rc) return rc;
    const long long rows = static_cast<long long>(B) * H * N;
    if (rows > kNoallocMaxRows)
        return fail(FA_ERR_TOO_LARGE, "fa_bwd_noalloc supports B*H*N <= " +
                                          std::to_string(kNoallocMaxRows) + " rows (got " +
                                          std::to_string(rows) + "); use fa_bwd with a workspace");
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;
    return bwd_entry(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                     scratch, kNoallocBytes, 0, -1, stream);
}

// ---------------------------------------------------------------------------------------
// e4m3 forward
// ---------------------------------------------------------------------------------------
namespace {

long long fp8_pad_keys(int N) { return (static_cast<long long>(N) + 15) / 16 * 16; }

// 3-D map of 8-bit codes, dimensions (x, y, z) with byte strides for y and z; box 128 bytes x
// by_ x bz (128 rows of one 128-byte swizzle panel: by_ = 128, bz = 1, or bz = 128 rows along
// z for tensors stored token by token).
int make_map_u8(CUtensorMap* m, const void* base, cuuint64_t x, cuuint64_t y, cuuint64_t z,
                cuuint64_t y_stride, cuuint64_t z_stride, cuuint32_t by_ = 128, cuuint32_t bz = 1)
{
    cuuint64_t dims[3] = {x, y, z};
    cuuint64_t strides[2] = {y_stride, z_stride};
    cuuint32_t box[3] = {128, by_, bz};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed with code " + std::to_string(r));
    return FA_OK;
}

bool finite(float x) { return x == x && x != INFINITY && x != -INFINITY; }

}  // namespace

extern "C" size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d)
{
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return align256(static_cast<size_t>(B) * H * d * static_cast<size_t>(fp8_pad_keys(N)));
}

extern "C" int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int N, int d, float scale, float q_descale,
                          float k_descale, float v_descale, int causal, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    int rc = check_common(B, H, N, d, scale, causal, FA_BF16);
    if (rc) return rc;
    if (d != 128) return fail(FA_ERR_UNSUPPORTED_D, "the e4m3 forward takes d = 128 only");
    if (!finite(q_descale) || !finite(k_descale) || !finite(v_descale) ||
        !finite(scale * q_descale * k_descale))
        return fail(FA_ERR_INVALID_ARG, "descale factors (and their product with scale) must be finite");
    if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA_ERR_MISALIGNED, "q, k, v, o must be 16-byte aligned (lse 4-byte)");
    const size_t need = fa_fwd_fp8_workspace_bytes(B, H, N, d);
    if (!workspace || workspace_bytes < need)
        return fail(FA_ERR_WORKSPACE, "workspace must hold " + std::to_string(need) + " bytes");
    if (!aligned16(workspace)) return fail(FA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    if ((rc = get_encoder())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long Npad = fp8_pad_keys(N);
    const cuuint64_t BH = static_cast<cuuint64_t>(B) * H, n = static_cast<cuuint64_t>(N);
    CUtensorMap maps[3];
    // Q, K: (d, N, B*H) bytes; V^T: (Npad keys, d, B*H)
    if ((rc = make_map_u8(&maps[0], q, 128, n, BH, 128, n * 128)) ||
        (rc = make_map_u8(&maps[1], k, 128, n, BH, 128, n * 128)) ||
        (rc = make_map_u8(&maps[2], workspace, static_cast<cuuint64_t>(Npad), 128, BH,
                          static_cast<cuuint64_t>(Npad), static_cast<cuuint64_t>(Npad) * 128)))
        return rc;
    fa::FwdParams p{};
    p.q = q; p.k = k; p.v = workspace; p.o = o; p.lse = lse;
    p.N = N; p.BH = B * H; p.scale = scale;
    p.scale_log2 = scale * q_descale * k_descale * fa::kLog2e;
    p.v_descale = v_descale;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    p.L = fixed_layout(B, H, N, d);
    p.L.order_group = order_group(N, d, causal);
    cudaError_t e = fa::launch_vt_transpose(v, workspace, p.L, static_cast<int>(Npad), di->status, st);
    if (e != cudaSuccess) return cuda_fail(e, "V transpose launch");
    e = fa::launch_fwd_fp8_tc(maps[0], maps[1], maps[2], p, st);
    if (e != cudaSuccess) return cuda_fail(e, "e4m3 forward launch");
    return FA_OK;
}

extern "C" size_t fa_fwd_fp8_varlen_workspace_bytes(int B, int max_seqlen_k, int Hkv, int d)
{
    if (B < 1 || max_seqlen_k < 1 || Hkv < 1 || d < 1) return 0;
    return align256(static_cast<size_t>(B) * Hkv * d * static_cast<size_t>(fp8_pad_keys(max_seqlen_k)));
}

extern "C" int fa_fwd_fp8_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                                 int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                                 int H, int Hkv, int d, float scale, float q_descale,
                                 float k_descale, float v_descale, int causal, void* workspace,
                                 size_t workspace_bytes, void* stream)
{
    int max_q = max_seqlen_q, max_k = max_seqlen_k;
    int rc = check_varlen(cu_seqlens_q, cu_seqlens_k, B, &max_q, &max_k, total_q, total_k, H, Hkv,
                          d, scale, causal);
    if (rc) return rc;
    if (d != 128) return fail(FA_ERR_UNSUPPORTED_D, "the e4m3 forward takes d = 128 only");
    if (!finite(q_descale) || !finite(k_descale) || !finite(v_descale) ||
        !finite(scale * q_descale * k_descale))
        return fail(FA_ERR_INVALID_ARG, "descale factors (and their product with scale) must be finite");
    if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return fail(FA_ERR_MISALIGNED, "q, k, v, o must be 16-byte aligned (lse 4-byte)");
    const long long Kpad = fp8_pad_keys(max_k);
    if (static_cast<long long>(B) * Hkv * ((Kpad + 63) / 64) >= (1LL << 31))
        return fail(FA_ERR_TOO_LARGE, "B * Hkv * ceil(max_seqlen_k / 64) must be < 2^31");
    const size_t need = fa_fwd_fp8_varlen_workspace_bytes(B, max_k, Hkv, d);
    if (!workspace || workspace_bytes < need)
        return fail(FA_ERR_WORKSPACE, "workspace must hold " + std::to_string(need) + " bytes");
    if (!aligned16(workspace)) return fail(FA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    if ((rc = get_encoder())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap maps[3];
    // Q: (d, H, total_q), K: (d, Hkv, total_k) bytes, boxes of 128 tokens of one head;
    // V^T: (Kpad keys, d, B*Hkv)
    const cuuint64_t hq = static_cast<cuuint64_t>(H), hk = static_cast<cuuint64_t>(Hkv);
    if ((rc = make_map_u8(&maps[0], q, 128, hq, static_cast<cuuint64_t>(total_q), 128, hq * 128, 1, 128)) ||
        (rc = make_map_u8(&maps[1], k, 128, hk, static_cast<cuuint64_t>(total_k), 128, hk * 128, 1, 128)) ||
        (rc = make_map_u8(&maps[2], workspace, static_cast<cuuint64_t>(Kpad), 128,
                          static_cast<cuuint64_t>(B) * hk, static_cast<cuuint64_t>(Kpad),
                          static_cast<cuuint64_t>(Kpad) * 128)))
        return rc;
    fa::FwdParams p{};
    p.q = q; p.k = k; p.v = workspace; p.o = o; p.lse = lse;
    p.N = total_q; p.BH = H; p.scale = scale;
    p.scale_log2 = scale * q_descale * k_descale * fa::kLog2e;
    p.v_descale = v_descale;
    p.causal = causal; p.status = di->status; p.wait_limit_ns = g_wait_limit_ns;
    p.debug_flags = g_debug_flags;
    p.L = packed_layout(cu_seqlens_q, cu_seqlens_k, B, max_q, max_k, total_q, total_k, H, Hkv, d,
                        packed_strides(H, Hkv, d));
    cudaError_t e = fa::launch_vt_transpose(v, workspace, p.L, static_cast<int>(Kpad), di->status, st);
    if (e != cudaSuccess) return cuda_fail(e, "V transpose launch");
    e = fa::launch_fwd_fp8_tc(maps[0], maps[1], maps[2], p, st);
    if (e != cudaSuccess) return cuda_fail(e, "e4m3 forward launch");
    return FA_OK;
}
