// Internal launch interface between the C ABI (kda_api.cu) and the kernels.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

struct DecodeParams {
    const void *q, *k, *v;
    const float *g;
    const void *b;
    const int32_t *slot_ids;
    float *pool;
    int64_t num_slots;
    void *out;
    int32_t *err_flag;
    int32_t batch, H, dv;
    float eps, scale;
};

// Fused decode (ShortConv + decode step + RMS norm and sigmoid gate).
struct DecodeFusedParams {
    const void *q, *k, *v;
    const float *g;
    const void *b;
    const int32_t *slot_ids;
    float *pool;
    int64_t num_slots;
    void *conv_state;     // dtype [num_slots][H][3][2 dk + dv]
    const float *conv_w;  // f32 [H][2 dk + dv][4]
    const void *z;        // dtype [batch][H][dv]
    const float *norm_w;  // f32 [dv]
    void *out;
    int32_t *err_flag;
    int32_t batch, H, dv;
    float eps, scale, eps_o;
};

struct VerifyParams {
    const void *q, *k, *v;
    const float *g;
    const void *b;
    const int32_t *slot_ids;
    const float *pool;
    int64_t num_slots;
    void *out;
    float *rec_k_hat;
    void *rec_v;
    float *rec_g;
    float *rec_beta;
    void *workspace;  // scratch of verify_workspace_bytes(...) bytes, or null when that is 0
    int32_t *err_flag;
    int32_t batch, D, H, dv;
    float eps, scale;
    // u-record variant: u_j = beta_j (v_j - S'_j k^_j) per value row, fp32
    // [B][D][H][dv] (null: not written; rec_v and rec_beta may then be null)
    float *rec_u;
    // commit first: before this window, the accepted prefix of the previous
    // window's u records is applied to the committed state, which is written
    // back (prev_accepted null: no commit; the CUDA-core verify kernel does it
    // in the same launch, the tensor-core path as a launch of its own)
    const float *prev_k_hat, *prev_g, *prev_u;
    const int32_t *prev_accepted;
    int32_t prev_D;
};

struct ReplayParams {
    const float *rec_k_hat;
    const void *rec_v;
    const float *rec_g;
    const float *rec_beta;
    const float *rec_u;  // u-record commit (rec_v and rec_beta unused)
    const int32_t *num_accepted;
    const int32_t *slot_ids;
    float *pool;
    int64_t num_slots;
    int32_t *err_flag;
    int32_t batch, D, H, dv;
};

struct PrefillParams {
    const int32_t *cu_seqlens;
    int64_t total_tokens;
    const void *q, *k, *v;
    const float *g;
    const void *b;
    const int32_t *slot_ids;
    float *pool;
    int64_t num_slots;
    int32_t init_from_pool;
    void *out;
    void *workspace;
    size_t workspace_bytes;
    int32_t *err_flag;
    int32_t num_seqs, H, dk, dv;
    float eps, scale;
    // state snapshots at chunk boundaries (num_snaps = 0: none); requests
    // sorted by sequence, then by token count
    int32_t num_snaps;
    const int32_t *snap_seq, *snap_tokens, *snap_slot;
    // fused ShortConv + gated RMS norm (conv_w null: the plain prefill);
    // tensor-core path only
    void *conv_state;     // dtype [num_slots][H][3][2 dk + dv]
    const float *conv_w;  // f32 [H][2 dk + dv][4]
    const void *z;        // dtype [total_tokens][H][dv]
    const float *norm_w;  // f32 [dv]
    float eps_o;
};

// Snapshot requests of sequence s: [lo, hi) of the sorted request list.
__device__ __forceinline__ void snap_range(const PrefillParams &p, int s, int &lo, int &hi) {
    int a = 0, b = p.num_snaps;  // first request with sequence >= s
    while (a < b) {
        const int m = (a + b) >> 1;
        if (p.snap_seq[m] < s) a = m + 1; else b = m;
    }
    lo = a;
    b = p.num_snaps;  // first request with sequence > s
    while (a < b) {
        const int m = (a + b) >> 1;
        if (p.snap_seq[m] <= s) a = m + 1; else b = m;
    }
    hi = a;
}

// The snapshot requests due once `done` tokens of the sequence are in the
// state: calls store(slot) for each valid one and returns the next pending
// request.  A request that can no longer be met (its token count is not a
// positive multiple of the chunk length, it is out of order, or its slot is
// out of range) is skipped and flagged in `bad`.
template <typename F>
__device__ __forceinline__ int snap_due(const PrefillParams &p, int ptr, int hi, int64_t done, int chunk_len,
                                        bool &bad, F &&store) {
    while (ptr < hi && (int64_t)p.snap_tokens[ptr] <= done) {
        const int64_t t = p.snap_tokens[ptr];
        const int slot = p.snap_slot[ptr];
        if (t == done && t > 0 && t % chunk_len == 0 && (int64_t)slot < p.num_slots) {
            if (slot >= 0) store(slot);
        } else {
            bad = true;
        }
        ++ptr;
    }
    return ptr;
}

// The driver's cuTensorMapEncodeTiled (looked up once through the runtime),
// or nullptr when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn();

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_decode(const DecodeParams &p, int dk, int dtype, cudaStream_t s);
cudaError_t launch_decode_fused(const DecodeFusedParams &p, int dk, int dtype, cudaStream_t s);
cudaError_t launch_verify(const VerifyParams &p, int dk, int dtype, cudaStream_t s);
// Verify for bf16, dk = dv = 128, D <= 8 (window kernel + tensor-core state
// kernel): the scratch it needs (0 for every other shape), whether it applies
// to these parameters, and its launcher.
size_t verify_workspace_bytes(int H, int dk, int dv, int dtype, int64_t batch, int D);
bool verify_tc_supported(const VerifyParams &p, int dk, int dtype);
cudaError_t launch_verify_tc(const VerifyParams &p, cudaStream_t st);
cudaError_t launch_replay(const ReplayParams &p, int dk, int dtype, cudaStream_t s);
// Commit from u records: S <- S diag(exp g_j) + u_j k^_j^T for the accepted prefix.
cudaError_t launch_replay_u(const ReplayParams &p, int dk, cudaStream_t s);
cudaError_t launch_prefill(const PrefillParams &p, int dtype, cudaStream_t s);
size_t prefill_workspace_bytes(int H, int dk, int dv, int dtype, int32_t num_seqs, int64_t total_tokens);

// Tensor-core prefill (dk = dv = 128, bf16): a prep kernel over all chunks
// writes per-(chunk, head) operand images, a chain kernel walks the chunks.
bool prefill_tc_supported(int dk, int dv, int dtype);
size_t prefill_tc_workspace_bytes(int H, int32_t num_seqs, int64_t total_tokens);
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s);

}  // namespace kda
