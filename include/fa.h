/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * What it computes.  Exact scaled-dot-product attention for each of B*H independent heads:
 *     S = scale * Q K^T,  P = softmax(S) row-wise (optionally with the causal mask),  O = P V,
 * as in "Standard Attention Implementation" (Algorithm 0) of the review "[논문 리뷰]
 * FlashAttention: Fast and Memory-Efficient Exact Attention with IO-Awareness", computed
 * tile by tile with the online softmax of its Algorithm 1 and of the "Tiling" section of
 * "Flash Attention IO-awareness principle", so S and P never reach device memory.  The
 * backward pass follows "Backward 구현" of "Triton 06: Flash Attention v2": Delta =
 * rowsum(dO o O), then dK, dV and dQ recomputed from the stored log-sum-exp.
 *
 * Entry-point families.
 *   - Fixed length (fa_fwd, fa_bwd and their variants): every tensor is contiguous row-major
 *     [B, H, N, d]; lse is [B, H, N] float32; dtype FA_BF16 (bfloat16 tensors, fp32
 *     accumulation, tensor cores) or FA_F32 (all fp32, SIMT kernels); B*H*N*d < 2^31.
 *   - Packed (fa_fwd_varlen, fa_bwd_varlen, their _strided forms, fa_fwd_decode): sequences of
 *     different lengths back to back, [total, heads, d], grouped key/value heads, bf16; their
 *     conventions are stated with them below.
 *
 * Conventions shared by every entry point.
 *   - d (head dimension) is 64 or 128; sizes are >= 1.
 *   - Causal mask: key index j <= query index i (top-left aligned, square), the condition
 *     offs_m >= offs_n of "개선 3" in "Triton 06: Flash Attention v2"; the packed calls align
 *     it to the bottom-right corner, which is the same mask when queries and keys are equal
 *     in number.
 *   - lse receives, per query row, the natural log of sum_j exp(scale * q_i . k_j) over the
 *     visible keys (the base-2 value the kernels keep is converted, as that post describes).
 *   - Pointers are device pointers, 16-byte aligned.  The caller allocates and owns every
 *     buffer; the library allocates no device memory on these paths.
 *   - Outputs must not overlap one another, an input or the workspace: the backward's kernels
 *     run concurrently (dQ in the tail of dK/dV).  The backward entry points with contiguous
 *     tensors check this on the host (FA_ERR_INVALID_ARG); strided views are not checked.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous on it.
 *   - Return value: FA_OK (0) or a negative FA_ERR_* code.  Argument errors are detected on
 *     the host before anything is launched; nothing throws across the ABI.  Device-side
 *     watchdog failures are reported by fa_device_status().
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum fa_dtype { FA_BF16 = 0, FA_F32 = 1 };

enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,     /* null pointer, non-positive size, bad flag or dtype     */
    FA_ERR_UNSUPPORTED_D = -2,   /* head dimension other than 64 or 128                    */
    FA_ERR_MISALIGNED = -3,      /* a pointer is not 16-byte aligned                       */
    FA_ERR_WORKSPACE = -4,       /* workspace missing or smaller than fa_bwd_workspace_bytes */
    FA_ERR_LAUNCH = -5,          /* a CUDA call failed; fa_last_error() has its text       */
    FA_ERR_DEVICE_TIMEOUT = -6,  /* a bounded on-device wait expired (watchdog)            */
    FA_ERR_TOO_LARGE = -7,       /* a tensor has 2^31 or more elements                     */
    FA_ERR_UNSUPPORTED_DEVICE = -8, /* bf16 tensor-core path needs compute capability 10.3 */
    FA_ERR_OUT_OF_BOUNDS = -9    /* checked builds: an access fell outside its buffer      */
};

/* Forward.  q, k, v: inputs [B,H,N,d]; o: output [B,H,N,d] (same dtype); lse: output
 * [B,H,N] fp32 (may be NULL when the caller does not need it).  scale is any finite float
 * (1/sqrt(d) in the usual case).  causal is 0 or 1. */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, int dtype, void* stream);

/* Bytes of device workspace fa_bwd needs for this shape (Delta and a base-2 copy of lse,
 * both fp32 [B,H,N], plus alignment).  Returns 0 for invalid sizes. */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/* Backward of fa_fwd.  q, k, v, o, dout: [B,H,N,d] inputs (o and lse from fa_fwd with the
 * same q, k, v, scale, causal); dq, dk, dv: outputs [B,H,N,d]; workspace: caller-owned
 * device buffer of at least fa_bwd_workspace_bytes(B,H,N,d) bytes, overwritten.
 * Gradients are of L = sum(dout o O): dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO with
 * dS = P o (dP - Delta), dP = dO V^T, Delta = rowsum(dO o O).  Deterministic.
 * The dK/dV and dQ kernels of the tensor-core path are launched as programmatic dependents
 * (CUDA's programmatic stream serialization): their set-up may overlap the kernel before them,
 * and dQ may run in the tail of dK/dV (the two read the same inputs and write disjoint
 * outputs), but nothing reads an input before the work that precedes fa_bwd on the stream has
 * completed, and fa_bwd's last kernel completes only after all of its kernels have. */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
           void* stream);

/* One stage of fa_bwd, for callers that schedule or time the stages separately:
 * stage 0 = preprocess (Delta and the base-2 LSE into the workspace), 1 = dK and dV,
 * 2 = dQ.  Running stages 0, 1, 2 in order on one stream is exactly fa_bwd; stages 1 and 2
 * read the workspace stage 0 wrote and may run in either order after it.  Arguments and
 * errors as fa_bwd, plus FA_ERR_INVALID_ARG for another stage value.  bf16 only. */
int fa_bwd_stage(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                 int stage, void* stream);

/* Same as fa_fwd but forces an implementation: 0 = default dispatch, 1 = the portable SIMT
 * kernel (fp32 math; accepts bf16 or fp32 tensors).  For cross-checking the tensor-core
 * path on the device; the default path is what fa_fwd runs. */
int fa_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, float scale, int causal, int dtype, int impl, void* stream);

/* Same as fa_bwd but forces an implementation (0 = default, 1 = portable SIMT kernels). */
int fa_bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                int impl, void* stream);

/* Fixed-length batches with grouped key/value heads and possibly different query and key
 * lengths (bf16, tensor-core path): q, o, dout, dq are [B, H, Nq, d], k, v, dk, dv are
 * [B, Hkv, Nk, d], lse is [B, H, Nq] fp32, all contiguous.  Query head h reads key/value head
 * h / (H / Hkv) and the causal mask is aligned to the bottom-right corner (query i sees key
 * j iff j <= i + Nk - Nq), as for fa_fwd_varlen; rows that see no key get O = 0, lse = -inf.
 * H % Hkv == 0; B*H*Nq*d and B*Hkv*Nk*d < 2^31.  The backward's workspace is
 * fa_bwd_workspace_bytes(B, H, Nq, d); dk and dv of a shared head sum over its group.
 * Ownership, alignment, streams and errors as fa_fwd / fa_bwd. */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream);

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
               const float* lse, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq,
               int Nk, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
               void* stream);

/* e4m3 (FP8) forward, per-tensor scaling (the FP8 mode of FlashAttention-3 named in the
 * "FA2·FA3" section of "Flash Attention IO-awareness principle"; the page gives no
 * algorithm, so the plainest reading is taken).
 *
 * What it computes.  q, k, v hold e4m3 codes (1 byte each, OCP FP8 E4M3: bias 7, no
 * infinities, largest finite 448) standing for the values Q = q_descale * q, K = k_descale * k,
 * V = v_descale * v.  The result is exact attention on those values, as fa_fwd computes it:
 * O = softmax(scale * Q K^T [+ causal mask]) V in bf16 and lse (natural log of the scaled
 * logits) in fp32.  Q K^T accumulates exactly (every e4m3 product is exact in fp32); the
 * probabilities enter the P V product rounded to e4m3, so |O - O_exact| is bounded, element
 * by element, by v_descale * sum_j max(2^-4 P_ij, 2^-10 max_j P_ij) |v_jc| plus bf16
 * rounding of O.  O is divided by the fp32 sum of the unrounded probabilities.
 *
 *   - Layout: q, k, v [B, H, N, 128] contiguous bytes; o [B, H, N, 128] bf16; lse [B, H, N]
 *     fp32 (may be null).  d must be 128 (else FA_ERR_UNSUPPORTED_D).
 *   - workspace: at least fa_fwd_fp8_workspace_bytes(B, H, N, d) bytes, 16-byte aligned,
 *     owned by the caller; it receives a transposed copy of v (each head's 128 x N codes,
 *     keys padded to a multiple of 16) that the tensor-core kernel reads as a K-major
 *     operand.  Its contents need no initialisation and mean nothing after the call.
 *   - scale, q_descale, k_descale, v_descale: finite floats (else FA_ERR_INVALID_ARG);
 *     scale * q_descale * k_descale multiplies the dot products of the stored e4m3 values.
 *   - Errors, streams and ownership as fa_fwd; two kernels run on `stream` (the transpose,
 *     then the forward).  Needs compute capability 10.3. */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d);

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, float q_descale, float k_descale, float v_descale,
               int causal, void* workspace, size_t workspace_bytes, void* stream);

/* e4m3 forward on packed variable-length batches with grouped key/value heads: what
 * fa_fwd_fp8 computes, with the sequences, head grouping, bottom-right causal mask and
 * empty-row rules of fa_fwd_varlen (see there).
 *   - q [total_q, H, 128], k and v [total_k, Hkv, 128] e4m3 codes, contiguous; o
 *     [total_q, H, 128] bf16; lse [H, total_q] fp32 (may be null); cu_seqlens_* int32 [B + 1]
 *     on the device, read by the kernels (malformed offsets are clamped to the tensors).
 *   - workspace: at least fa_fwd_fp8_varlen_workspace_bytes(B, max_seqlen_k, Hkv, d) bytes,
 *     16-byte aligned; it receives V^T per (sequence, key/value head), each padded to
 *     max_seqlen_k rounded up to 16 keys, so it grows with B * max_seqlen_k rather than
 *     total_k.
 *   - Errors as fa_fwd_varlen and fa_fwd_fp8, plus FA_ERR_TOO_LARGE when
 *     B * Hkv * ceil(max_seqlen_k / 64) >= 2^31. */
size_t fa_fwd_fp8_varlen_workspace_bytes(int B, int max_seqlen_k, int Hkv, int d);

int fa_fwd_fp8_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                      const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int max_seqlen_q,
                      int max_seqlen_k, int total_q, int total_k, int H, int Hkv, int d,
                      float scale, float q_descale, float k_descale, float v_descale, int causal,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Packed variable-length batches with grouped key/value heads (bf16, tensor-core path).
 *
 * What it computes.  B independent sequences; sequence b has the query rows
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]) and the key/value rows [cu_seqlens_k[b],
 * cu_seqlens_k[b+1]), so nq_b queries and nk_b keys, which may differ.  Query head h attends to
 * key/value head h / (H / Hkv): Hkv = H is multi-head attention, 1 < Hkv < H grouped-query
 * attention and Hkv = 1 multi-query attention (the GQA / MQA models of "서빙에서 Flash
 * Attention 이득이 예상보다 작은 경우" in "Flash Attention IO-awareness principle").  The
 * causal mask is aligned to the bottom-right corner: query i sees key j iff
 * j <= i + (nk_b - nq_b), so a chunk of the last nq_b queries of a prompt sees every earlier
 * key, as chunked prefill needs ("PagedAttention·Chunked Prefill과의 위치", same page); with
 * nq_b == nk_b this is the square mask of fa_fwd.  A query row that sees no key (nq_b > nk_b
 * under the causal mask, or nk_b == 0) gets O = 0, lse = -inf and zero gradient.
 *
 * Layout (token by token, no padding between sequences):
 *   q, o, dout, dq: [total_q, H, d] bf16;  k, v, dk, dv: [total_k, Hkv, d] bf16;
 *   lse: [H, total_q] fp32 (may be NULL in the forward);
 *   cu_seqlens_q, cu_seqlens_k: device int32 arrays of B+1 non-decreasing offsets, [0] = 0,
 *   [B] = total_q (total_k).  The library cannot read them on the host: offsets outside
 *   [0, total] are clamped on the device and lengths are clamped to max_seqlen_q /
 *   max_seqlen_k (an upper bound the caller passes; larger values only cost idle CTAs), so
 *   inconsistent offsets give wrong values but never touch memory outside the buffers.
 * d is 64 or 128; H % Hkv == 0; total_q*H*d and total_k*Hkv*d < 2^31.  Ownership, alignment,
 * streams and error codes as for fa_fwd / fa_bwd. */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int max_seqlen_q,
                  int max_seqlen_k, int total_q, int total_k, int H, int Hkv, int d, float scale,
                  int causal, void* stream);

/* Bytes of device workspace fa_bwd_varlen needs (Delta and the base-2 LSE, fp32 [H, total_q],
 * plus alignment).  Returns 0 for invalid sizes. */
size_t fa_bwd_varlen_workspace_bytes(int total_q, int H, int d);

/* Backward of fa_fwd_varlen (o and lse from it with the same arguments).  Gradients as for
 * fa_bwd; dk and dv of a shared key/value head are the sums over the query heads of its group.
 * Deterministic (no atomics). */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int max_seqlen_q, int max_seqlen_k, int total_q,
                  int total_k, int H, int Hkv, int d, float scale, int causal, void* workspace,
                  size_t workspace_bytes, void* stream);

/* fa_fwd_varlen / fa_bwd_varlen on tensors with caller-chosen element strides, so that views
 * need no copy: for example q, k and v taken from one fused projection [total, 3, H, d], or
 * outputs written into slices of larger buffers.  strides is a host array of (row, head)
 * element-stride pairs, one pair per tensor in argument order: q, k, v, o for the forward
 * (8 values); q, k, v, o, dout, dq, dk, dv for the backward (16 values).  Row i, head h of a
 * tensor starts at base + i * row + h * head elements; its d elements are contiguous.
 * Each stride must be a positive multiple of 8 elements (16 bytes; else FA_ERR_MISALIGNED),
 * head >= d and row >= head (tensors stored token by token; else FA_ERR_INVALID_ARG).
 * Output views must not overlap one another or an input view (not checked).  Everything
 * else as fa_fwd_varlen / fa_bwd_varlen. */
int fa_fwd_varlen_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                          const long long* strides, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, int B, int max_seqlen_q, int max_seqlen_k,
                          int total_q, int total_k, int H, int Hkv, int d, float scale,
                          int causal, void* stream);

int fa_bwd_varlen_strided(const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          const long long* strides, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, int B, int max_seqlen_q, int max_seqlen_k,
                          int total_q, int total_k, int H, int Hkv, int d, float scale,
                          int causal, void* workspace, size_t workspace_bytes, void* stream);

/* Split-KV decode: the forward of fa_fwd_varlen (same arguments, layout, mask, results up to
 * rounding) laid out for few queries per sequence against a long key/value history, the
 * decoding case that "서빙에서 Flash Attention 이득이 예상보다 작은 경우" in "Flash Attention
 * IO-awareness principle" hands to decoding kernels.  The query heads of a group (H / Hkv)
 * and the sequence's queries share one 128-row tile, so they read their K and V once (when
 * the group times max_seqlen_q exceeds 128 rows, the group's heads are split into the fewest
 * equal chunks that fit, one tile each); each sequence's key blocks are split into num_splits
 * ranges processed in parallel, whose partial results (O and log-sum-exp per range) a second
 * kernel merges.
 *   - Requires max_seqlen_q <= 128 (else FA_ERR_INVALID_ARG: use fa_fwd_varlen).
 *   - num_splits in [1, 256]; fa_decode_num_splits suggests one for this GPU.  Ranges with no
 *     key block (num_splits larger than the blocks of a sequence) contribute nothing.
 *   - workspace: caller-owned device buffer of fa_decode_workspace_bytes(total_q, H, d,
 *     num_splits) bytes (0 for num_splits = 1, when workspace may be NULL); overwritten.
 *   - Its kernels are launched as programmatic dependents (CUDA's programmatic stream
 *     serialization): their set-up may overlap the end of the work before them on the stream,
 *     but they read no input and write no output before that work has completed, so stream
 *     order is kept.
 * bf16 only, forward only.  Errors as fa_fwd_varlen, plus FA_ERR_WORKSPACE. */
int fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int max_seqlen_q,
                  int max_seqlen_k, int total_q, int total_k, int H, int Hkv, int d, float scale,
                  int causal, int num_splits, void* workspace, size_t workspace_bytes,
                  void* stream);

/* Bytes of workspace fa_fwd_decode needs: the partial O (fp32 [num_splits, total_q, H, d]) and
 * log-sum-exp (fp32 [num_splits, H, total_q]) of every range, plus alignment; 0 for
 * num_splits = 1 or invalid sizes. */
size_t fa_decode_workspace_bytes(int total_q, int H, int d, int num_splits);

/* A split count for fa_fwd_decode on the current device: the largest one whose B * Hkv *
 * num_splits CTAs fit on the device's SMs at one per SM (at least 1), at most
 * max(1, blocks / 8) (blocks = ceil(max_seqlen_k / 128)).  Returns it (>= 1) or a negative
 * FA_ERR_* code. */
int fa_decode_num_splits(int B, int Hkv, int max_seqlen_k);

/* Backward for callers that cannot allocate device memory.  This entry point has no
 * counterpart on the pages; it exists for code that is not allowed to call cudaMalloc or any
 * allocating routine, for example a plugin running inside a host framework that owns every
 * byte of device memory, or a latency-critical loop that must not take the device-wide
 * synchronisation an allocation can imply.  It computes exactly what fa_bwd computes (the
 * same kernels, so the same bits), with the same arguments except the workspace: its scratch
 * (Delta and the base-2 LSE) lives in a fixed 8 MiB array inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   - Limit: B*H*N <= 1048576 rows (1 << 20); larger shapes return FA_ERR_TOO_LARGE and must
 *     use fa_bwd with a workspace.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, with that device current).  The CUDA runtime
 *     may load the library's device code, and with it back the array, at the first call of
 *     any entry point on a device; make that first call, and the first fa_bwd_noalloc call,
 *     before any stream capture.  Every later fa_bwd_noalloc call allocates nothing.
 *   - The looked-up address is kept for the life of the process: the library must not be
 *     used on a device after cudaDeviceReset (the same holds for every entry point, which
 *     keep the device's status-word address and kernel attributes).
 *   - Every call shares the one array and overwrites all of it that it uses before reading
 *     it, so nothing carries over between calls; calls that overlap on the GPU (for example
 *     on two streams at once) race on the array and must be serialised by the caller. */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, int dtype, void* stream);

/* Synchronises `stream`, then reads and clears the device status word that bounded waits
 * inside the kernels write when they give up.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT (the
 * wait site is appended to fa_last_error()), FA_ERR_OUT_OF_BOUNDS (checked builds only) or
 * FA_ERR_LAUNCH if the synchronisation failed. */
int fa_device_status(void* stream);

/* Upper bound, in nanoseconds, on every on-device wait (default 2e9).  Values below 1e6 are
 * clamped to 1e6.  Applies to launches made after the call. */
void fa_set_wait_limit_ns(unsigned long long ns);

/* Test hook for the watchdog: flags = 1 makes the tensor-core kernels announce their first
 * streamed tile without copying it, so the wait for it can only end by expiring; each CTA then
 * aborts cleanly (frees Tensor Memory, returns) and fa_device_status() reports
 * FA_ERR_DEVICE_TIMEOUT.  0 (the default) restores normal operation.  Not for production use;
 * applies to launches made after the call. */
void fa_debug_set_flags(int flags);

/* 1 if this library is the checked build (libfa_checked.so, compiled with FA_CHECKED), else 0.
 * A checked build tests every element that the tensor-core, decode, backward-preprocess and
 * e4m3-transpose kernels read or write directly in global memory (outputs, gradients,
 * statistics, decode partials, V and its transposed copy; tiles moved by TMA are bounded by
 * their tensor maps; the fp32 SIMT kernels index only from their grid and take no offsets)
 * against the extent of its buffer implied by the call's sizes and strides:
 * an access outside it is skipped and fa_device_status() then returns FA_ERR_OUT_OF_BOUNDS.
 * Its results are otherwise identical to the regular build's.  With fa_debug_set_flags(2)
 * the checked build takes every extent one row short, so the check must fire (test hook). */
int fa_checked_build(void);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(int code);

/* Text of the last error seen by this thread (empty string if none). */
const char* fa_last_error(void);

/* Causal block schedule of query block `q_block` (rows [q_block*Br, min(N,(q_block+1)*Br)))
 * against key blocks of Bc keys: number of blocks visited without a mask (*n_full) and with
 * the element-wise mask (*n_masked); the rest are skipped.  This is the host copy of the
 * classification every kernel uses ("개선 3", two-stage causal split).  Host-only. */
int fa_causal_block_counts(int q_block, int Br, int Bc, int N, int* n_full, int* n_masked);

/* Order of the work tiles of the tensor-core kernels, host copy (tests and schedulers).  A
 * launch over `heads` heads of `nblk` tiles each runs tile index `id` (its CTA index, or the index
 * of a CTA whose launch it took over) as (*head, *rank), rank 0 being a head's heaviest tile
 * under the causal mask.  Heads go in groups of `gsize`: within a group the tiles go by rank, the
 * group's heads interleaved, so a group's heaviest tiles start first and its light ones fill the
 * end; gsize = 1 is head-major order.  Returns FA_OK, or FA_ERR_INVALID_ARG for arguments out of
 * range.  Host-only. */
int fa_tile_order(int id, int heads, int nblk, int gsize, int* head, int* rank);

/* The group size the fixed-length entry points pass to their kernels for sequences of N rows and
 * head dimension d: 1 without the causal mask (every tile costs the same); under it, as many
 * heads as keep one head's streamed rows (4 N d bytes) within 32 MB of L2, at most 16.
 * Host-only. */
int fa_order_group(int N, int d, int causal);

/* The split count fa_decode_num_splits gives on a device with num_sms SMs (host copy, for tests
 * and schedulers): min(max(1, blocks / 8), max(1, num_sms / (B * Hkv))), blocks =
 * ceil(max_seqlen_k / 128), capped at 256.  Returns it, or FA_ERR_INVALID_ARG for a size or
 * num_sms below 1.  Host-only. */
int fa_decode_splits_for(int B, int Hkv, int max_seqlen_k, int num_sms);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
