// Parameter block of the split-KV decode kernels (fa_decode_tc.cu), shared with the host side
// of the ABI.
#pragma once
#include "fa_common.cuh"

namespace fa {

// Parameters of the split-KV decode kernels (packed layout only).  One CTA owns the query rows
// of one (sequence, key/value head, head chunk): G consecutive query heads of the group
// (the group's H / Hkv heads are split into head_chunks chunks of G when the group times the
// sequence's nq <= q_box queries exceeds 128 rows) times the queries, row r = i * G + g (query
// i, head hk * (H / Hkv) + chunk * G + g), at most 128.
// Its keys are split into `splits` contiguous ranges of 128-key blocks; with splits > 1 every
// range writes a partial result (O normalised by its own weights, fp32, and its natural-log
// LSE) and the combine kernel merges them.
struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;           // bf16 [total_q, H, d]
    float* lse;        // fp32 [H, total_q] (may be null)
    float* o_part;     // workspace: fp32 [splits, total_q, H, d]
    float* lse_part;   // workspace: fp32 [splits, H, total_q]
    int splits;
    int G;             // query heads per CTA (a divisor of H / Hkv)
    int head_chunks;   // (H / Hkv) / G
    int q_box;         // queries per sequence covered by the Q tile (max_seqlen_q)
    float scale_log2;
    int causal;
    int* status;
    unsigned long long wait_limit_ns;
    int debug_flags;
    long long part_ext;  // elements of o_part (checked builds)
    Layout L;
};

}  // namespace fa
