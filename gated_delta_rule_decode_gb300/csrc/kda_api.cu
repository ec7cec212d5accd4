// C ABI of libkda.so: argument validation, dispatch and status strings.
// Every entry point checks its arguments on the host, returns a negative
// kda_status without launching anything on a host-detectable error, and
// otherwise enqueues its kernels on the caller's stream without synchronising.
#include <math.h>
#include <stdint.h>

#include "kda.h"
#include "kda_internal.h"

namespace {

bool head_size_ok(int32_t d) { return d == 32 || d == 64 || d == 128; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Common checks on kda_dims; returns KDA_OK or the status to report.
int check_dims(const kda_dims *d) {
    if (d == nullptr) return KDA_ERR_INVALID_ARG;
    if (d->num_heads < 1) return KDA_ERR_INVALID_ARG;
    if (d->dtype != KDA_DT_F32 && d->dtype != KDA_DT_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_size_ok(d->dk) || !head_size_ok(d->dv)) return KDA_ERR_UNSUPPORTED;
    if (!(d->eps >= 0.f) || isinf(d->eps)) return KDA_ERR_INVALID_ARG;
    if (isnan(d->scale) || isinf(d->scale)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

float resolve_scale(const kda_dims *d) {
    return d->scale > 0.f ? d->scale : 1.0f / sqrtf((float)d->dk);
}

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    return KDA_ERR_CUDA;
}

bool all_aligned(std::initializer_list<const void *> ps) {
    for (const void *p : ps)
        if (p == nullptr || !aligned16(p)) return false;
    return true;
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

// The checked build's precondition check: a slot id named twice in one call
// (two CTAs would update the same state) sets KDA_DEVERR_DUPLICATE.  O(n^2)
// comparisons, before the call's kernels, on its stream; nothing in the
// normal build.
#ifdef KDA_CHECKED
static __global__ void duplicate_slots_kernel(const int32_t *slots, int32_t n, int32_t *flag) {
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int32_t si = slots[i];
        if (si < 0) continue;
        for (int32_t j = i + 1; j < n; ++j)
            if (slots[j] == si) {
                atomicOr(flag, KDA_DEVERR_DUPLICATE);
                break;
            }
    }
}
#endif

static int check_unique_slots(const int32_t *slots, int32_t n, int32_t *err_flag, void *stream) {
#ifdef KDA_CHECKED
    if (slots == nullptr || err_flag == nullptr || n < 2) return KDA_OK;
    const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
    duplicate_slots_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(slots, n, err_flag);
    return from_cuda(cudaGetLastError());
#else
    (void)slots, (void)n, (void)err_flag, (void)stream;
    return KDA_OK;
#endif
}

int kda_checked_build(void) {
#ifdef KDA_CHECKED
    return 1;
#else
    return 0;
#endif
}

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported head size or dtype";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        default: return "unknown status";
    }
}

size_t kda_records_bytes(const kda_dims *dims, int32_t batch, int32_t draft_len) {
    if (check_dims(dims) != KDA_OK || batch < 0 || draft_len < 1) return 0;
    const size_t tokens = (size_t)batch * (size_t)draft_len * (size_t)dims->num_heads;
    const size_t esz = dims->dtype == KDA_DT_BF16 ? 2 : 4;
    return tokens * ((size_t)dims->dk * 4 * 2 + (size_t)dims->dv * esz + 4);
}

int kda_decode(const kda_dims *dims, int32_t batch, const void *q, const void *k,
               const void *v, const float *g, const void *b, const int32_t *slot_ids,
               float *pool, int64_t num_slots, void *out, int32_t *err_flag, void *stream) {
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (batch == 0) return KDA_OK;
    if (!all_aligned({q, k, v, g, out}) || b == nullptr || slot_ids == nullptr)
        return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool})) return KDA_ERR_INVALID_ARG;
    kda::DecodeParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.b = b;
    p.slot_ids = slot_ids; p.pool = pool; p.num_slots = num_slots;
    p.out = out; p.err_flag = err_flag;
    p.batch = batch; p.H = dims->num_heads; p.dv = dims->dv;
    p.eps = dims->eps; p.scale = resolve_scale(dims);
    if (const int cs = check_unique_slots(slot_ids, batch, err_flag, stream)) return cs;
    return from_cuda(kda::launch_decode(p, dims->dk, dims->dtype, (cudaStream_t)stream));
}

int kda_decode_fused(const kda_dims *dims, int32_t batch, const void *q, const void *k,
                     const void *v, const float *g, const void *b, const int32_t *slot_ids,
                     float *pool, int64_t num_slots, const kda_fused_io *io, void *out,
                     int32_t *err_flag, void *stream) {
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_slots < 0 || io == nullptr) return KDA_ERR_INVALID_ARG;
    if (!(io->eps_o >= 0.f) || isinf(io->eps_o)) return KDA_ERR_INVALID_ARG;
    if (batch == 0) return KDA_OK;
    if (!all_aligned({q, k, v, g, out, io->conv_w, io->z, io->norm_w}) || b == nullptr ||
        slot_ids == nullptr)
        return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool, io->conv_state})) return KDA_ERR_INVALID_ARG;
    kda::DecodeFusedParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.b = b;
    p.slot_ids = slot_ids; p.pool = pool; p.num_slots = num_slots;
    p.conv_state = io->conv_state; p.conv_w = io->conv_w; p.z = io->z; p.norm_w = io->norm_w;
    p.out = out; p.err_flag = err_flag;
    p.batch = batch; p.H = dims->num_heads; p.dv = dims->dv;
    p.eps = dims->eps; p.scale = resolve_scale(dims); p.eps_o = io->eps_o;
    if (const int cs = check_unique_slots(slot_ids, batch, err_flag, stream)) return cs;
    return from_cuda(kda::launch_decode_fused(p, dims->dk, dims->dtype, (cudaStream_t)stream));
}

size_t kda_verify_workspace_bytes(const kda_dims *dims, int32_t batch, int32_t draft_len) {
    if (check_dims(dims) != KDA_OK || batch < 0 || draft_len < 1 || draft_len > 16) return 0;
    return kda::verify_workspace_bytes(dims->num_heads, dims->dk, dims->dv, dims->dtype, batch, draft_len);
}

int kda_verify_record(const kda_dims *dims, int32_t batch, int32_t draft_len, const void *q,
                      const void *k, const void *v, const float *g, const void *b,
                      const int32_t *slot_ids, const float *pool, int64_t num_slots, void *out,
                      const kda_records *rec, void *workspace, size_t workspace_bytes,
                      int32_t *err_flag, void *stream) {
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_slots < 0 || draft_len < 1 || draft_len > 16) return KDA_ERR_INVALID_ARG;
    if (batch == 0) return KDA_OK;
    if (rec == nullptr) return KDA_ERR_INVALID_ARG;
    if (!all_aligned({q, k, v, g, out, rec->k_hat, rec->v, rec->g}) || b == nullptr ||
        slot_ids == nullptr || rec->beta == nullptr)
        return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool})) return KDA_ERR_INVALID_ARG;
    const size_t need = kda::verify_workspace_bytes(dims->num_heads, dims->dk, dims->dv, dims->dtype,
                                                    batch, draft_len);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return KDA_ERR_WORKSPACE;
    kda::VerifyParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.b = b;
    p.workspace = need > 0 ? workspace : nullptr;
    p.slot_ids = slot_ids; p.pool = pool; p.num_slots = num_slots; p.out = out;
    p.rec_k_hat = rec->k_hat; p.rec_v = rec->v; p.rec_g = rec->g; p.rec_beta = rec->beta;
    p.err_flag = err_flag;
    p.batch = batch; p.D = draft_len; p.H = dims->num_heads; p.dv = dims->dv;
    p.eps = dims->eps; p.scale = resolve_scale(dims);
    if (const int cs = check_unique_slots(slot_ids, batch, err_flag, stream)) return cs;
    return from_cuda(kda::launch_verify(p, dims->dk, dims->dtype, (cudaStream_t)stream));
}

size_t kda_records_u_bytes(const kda_dims *dims, int32_t batch, int32_t draft_len) {
    if (check_dims(dims) != KDA_OK || batch < 0 || draft_len < 1) return 0;
    const size_t tokens = (size_t)batch * (size_t)draft_len * (size_t)dims->num_heads;
    return tokens * ((size_t)dims->dk * 4 * 2 + (size_t)dims->dv * 4);
}

// Verify into u records, optionally after committing the previous window's
// accepted u records (prev != NULL).
static int verify_u_impl(const kda_dims *dims, int32_t batch, int32_t prev_draft_len,
                         const kda_records_u *prev, const int32_t *prev_accepted, int32_t draft_len,
                         const void *q, const void *k, const void *v, const float *g, const void *b,
                         const int32_t *slot_ids, const float *pool, int64_t num_slots, void *out,
                         const kda_records_u *rec, void *workspace, size_t workspace_bytes,
                         int32_t *err_flag, void *stream) {
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_slots < 0 || draft_len < 1 || draft_len > 16) return KDA_ERR_INVALID_ARG;
    if (prev != nullptr && (prev_draft_len < 1 || prev_draft_len > 16 || prev_accepted == nullptr ||
                            !all_aligned({prev->k_hat, prev->g, prev->u})))
        return KDA_ERR_INVALID_ARG;
    if (batch == 0) return KDA_OK;
    if (rec == nullptr) return KDA_ERR_INVALID_ARG;
    if (!all_aligned({q, k, v, g, out, rec->k_hat, rec->g, rec->u}) || b == nullptr || slot_ids == nullptr)
        return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool})) return KDA_ERR_INVALID_ARG;
    const size_t need = kda::verify_workspace_bytes(dims->num_heads, dims->dk, dims->dv, dims->dtype,
                                                    batch, draft_len);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return KDA_ERR_WORKSPACE;
    kda::VerifyParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.b = b;
    p.workspace = need > 0 ? workspace : nullptr;
    p.slot_ids = slot_ids; p.pool = pool; p.num_slots = num_slots; p.out = out;
    p.rec_k_hat = rec->k_hat; p.rec_g = rec->g; p.rec_u = rec->u;
    p.err_flag = err_flag;
    p.batch = batch; p.D = draft_len; p.H = dims->num_heads; p.dv = dims->dv;
    p.eps = dims->eps; p.scale = resolve_scale(dims);
    if (prev != nullptr) {
        p.prev_k_hat = prev->k_hat; p.prev_g = prev->g; p.prev_u = prev->u;
        p.prev_accepted = prev_accepted; p.prev_D = prev_draft_len;
    }
    if (const int cs = check_unique_slots(slot_ids, batch, err_flag, stream)) return cs;
    return from_cuda(kda::launch_verify(p, dims->dk, dims->dtype, (cudaStream_t)stream));
}

int kda_verify_record_u(const kda_dims *dims, int32_t batch, int32_t draft_len, const void *q,
                        const void *k, const void *v, const float *g, const void *b,
                        const int32_t *slot_ids, const float *pool, int64_t num_slots, void *out,
                        const kda_records_u *rec, void *workspace, size_t workspace_bytes,
                        int32_t *err_flag, void *stream) {
    return verify_u_impl(dims, batch, 0, nullptr, nullptr, draft_len, q, k, v, g, b, slot_ids, pool,
                         num_slots, out, rec, workspace, workspace_bytes, err_flag, stream);
}

int kda_commit_verify_u(const kda_dims *dims, int32_t batch, int32_t prev_draft_len,
                        const kda_records_u *prev, const int32_t *prev_accepted, int32_t draft_len,
                        const void *q, const void *k, const void *v, const float *g, const void *b,
                        const int32_t *slot_ids, float *pool, int64_t num_slots, void *out,
                        const kda_records_u *rec, void *workspace, size_t workspace_bytes,
                        int32_t *err_flag, void *stream) {
    if (prev == nullptr) return KDA_ERR_INVALID_ARG;
    return verify_u_impl(dims, batch, prev_draft_len, prev, prev_accepted, draft_len, q, k, v, g, b, slot_ids,
                         pool, num_slots, out, rec, workspace, workspace_bytes, err_flag, stream);
}

int kda_replay_commit_u(const kda_dims *dims, int32_t batch, int32_t draft_len, const kda_records_u *rec,
                        const int32_t *num_accepted, const int32_t *slot_ids, float *pool,
                        int64_t num_slots, int32_t *err_flag, void *stream) {
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_slots < 0 || draft_len < 1 || draft_len > 16) return KDA_ERR_INVALID_ARG;
    if (batch == 0) return KDA_OK;
    if (rec == nullptr || num_accepted == nullptr || slot_ids == nullptr) return KDA_ERR_INVALID_ARG;
    if (!all_aligned({rec->k_hat, rec->g, rec->u})) return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool})) return KDA_ERR_INVALID_ARG;
    kda::ReplayParams p{};
    p.rec_k_hat = rec->k_hat; p.rec_g = rec->g; p.rec_u = rec->u;
    p.num_accepted = num_accepted; p.slot_ids = slot_ids;
    p.pool = pool; p.num_slots = num_slots; p.err_flag = err_flag;
    p.batch = batch; p.D = draft_len; p.H = dims->num_heads; p.dv = dims->dv;
    if (const int cs = check_unique_slots(slot_ids, batch, err_flag, stream)) return cs;
    return from_cuda(kda::launch_replay_u(p, dims->dk, (cudaStream_t)stream));
}

int kda_replay_commit(const kda_dims *dims, int32_t batch, int32_t draft_len,
                      const kda_records *rec, const int32_t *num_accepted,
                      const int32_t *slot_ids, float *pool, int64_t num_slots,
                      int32_t *err_flag, void *stream) {
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_slots < 0 || draft_len < 1 || draft_len > 16) return KDA_ERR_INVALID_ARG;
    if (batch == 0) return KDA_OK;
    if (rec == nullptr || num_accepted == nullptr || slot_ids == nullptr) return KDA_ERR_INVALID_ARG;
    if (!all_aligned({rec->k_hat, rec->v, rec->g}) || rec->beta == nullptr) return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool})) return KDA_ERR_INVALID_ARG;
    kda::ReplayParams p{};
    p.rec_k_hat = rec->k_hat; p.rec_v = rec->v; p.rec_g = rec->g; p.rec_beta = rec->beta;
    p.num_accepted = num_accepted; p.slot_ids = slot_ids;
    p.pool = pool; p.num_slots = num_slots; p.err_flag = err_flag;
    p.batch = batch; p.D = draft_len; p.H = dims->num_heads; p.dv = dims->dv;
    if (const int cs = check_unique_slots(slot_ids, batch, err_flag, stream)) return cs;
    return from_cuda(kda::launch_replay(p, dims->dk, dims->dtype, (cudaStream_t)stream));
}

size_t kda_prefill_workspace_bytes(const kda_dims *dims, int32_t num_seqs, int64_t total_tokens) {
    if (check_dims(dims) != KDA_OK || num_seqs < 0 || total_tokens < 0) return 0;
    return kda::prefill_workspace_bytes(dims->num_heads, dims->dk, dims->dv, dims->dtype, num_seqs,
                                        total_tokens);
}

static int prefill_impl(const kda_dims *dims, int32_t num_seqs, const int32_t *cu_seqlens,
                        int64_t total_tokens, const void *q, const void *k, const void *v,
                        const float *g, const void *b, const int32_t *slot_ids, float *pool,
                        int64_t num_slots, int32_t init_from_pool, void *out, int32_t num_snaps,
                        const int32_t *snap_seq, const int32_t *snap_tokens, const int32_t *snap_slot,
                        void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream,
                        const kda_fused_io *io = nullptr) {
    if (num_snaps < 0) return KDA_ERR_INVALID_ARG;
    if (num_snaps > 0 && (snap_seq == nullptr || snap_tokens == nullptr || snap_slot == nullptr))
        return KDA_ERR_INVALID_ARG;
    int st = check_dims(dims);
    if (st != KDA_OK) return st;
    if (num_seqs < 0 || total_tokens < 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return KDA_OK;
    if (cu_seqlens == nullptr || slot_ids == nullptr) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!all_aligned({q, k, v, g, out}) || b == nullptr))
        return KDA_ERR_INVALID_ARG;
    if (num_slots > 0 && !all_aligned({pool})) return KDA_ERR_INVALID_ARG;
    if (total_tokens > (int64_t)0x7fffffff) return KDA_ERR_INVALID_ARG;
    if (io != nullptr) {
        // the fused prefill exists on the tensor-core path only
        if (!kda::prefill_tc_supported(dims->dk, dims->dv, dims->dtype)) return KDA_ERR_UNSUPPORTED;
        if (!(io->eps_o >= 0.f) || isinf(io->eps_o)) return KDA_ERR_INVALID_ARG;
        if (!all_aligned({io->conv_w, io->norm_w})) return KDA_ERR_INVALID_ARG;
        if (total_tokens > 0 && !all_aligned({io->z})) return KDA_ERR_INVALID_ARG;
        if (num_slots > 0 && !all_aligned({io->conv_state})) return KDA_ERR_INVALID_ARG;
    }
    const size_t need = kda::prefill_workspace_bytes(dims->num_heads, dims->dk, dims->dv, dims->dtype,
                                                     num_seqs, total_tokens);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return KDA_ERR_WORKSPACE;
    kda::PrefillParams p{};
    p.cu_seqlens = cu_seqlens; p.total_tokens = total_tokens;
    p.q = q; p.k = k; p.v = v; p.g = g; p.b = b;
    p.slot_ids = slot_ids; p.pool = pool; p.num_slots = num_slots;
    p.init_from_pool = init_from_pool ? 1 : 0; p.out = out;
    p.workspace = workspace; p.workspace_bytes = workspace_bytes; p.err_flag = err_flag;
    p.num_seqs = num_seqs; p.H = dims->num_heads; p.dk = dims->dk; p.dv = dims->dv;
    p.eps = dims->eps; p.scale = resolve_scale(dims);
    p.num_snaps = num_snaps; p.snap_seq = snap_seq; p.snap_tokens = snap_tokens; p.snap_slot = snap_slot;
    if (io != nullptr) {
        p.conv_state = io->conv_state; p.conv_w = io->conv_w; p.z = io->z; p.norm_w = io->norm_w;
        p.eps_o = io->eps_o;
    }
    if (const int cs = check_unique_slots(slot_ids, num_seqs, err_flag, stream)) return cs;
    return from_cuda(kda::launch_prefill(p, dims->dtype, (cudaStream_t)stream));
}

int kda_prefill_chunked(const kda_dims *dims, int32_t num_seqs, const int32_t *cu_seqlens,
                        int64_t total_tokens, const void *q, const void *k, const void *v,
                        const float *g, const void *b, const int32_t *slot_ids, float *pool,
                        int64_t num_slots, int32_t init_from_pool, void *out, void *workspace,
                        size_t workspace_bytes, int32_t *err_flag, void *stream) {
    return prefill_impl(dims, num_seqs, cu_seqlens, total_tokens, q, k, v, g, b, slot_ids, pool, num_slots,
                        init_from_pool, out, 0, nullptr, nullptr, nullptr, workspace, workspace_bytes, err_flag,
                        stream);
}

int kda_prefill_chunked_snapshots(const kda_dims *dims, int32_t num_seqs, const int32_t *cu_seqlens,
                                  int64_t total_tokens, const void *q, const void *k, const void *v,
                                  const float *g, const void *b, const int32_t *slot_ids, float *pool,
                                  int64_t num_slots, int32_t init_from_pool, void *out, int32_t num_snaps,
                                  const int32_t *snap_seq, const int32_t *snap_tokens,
                                  const int32_t *snap_slot, void *workspace, size_t workspace_bytes,
                                  int32_t *err_flag, void *stream) {
    return prefill_impl(dims, num_seqs, cu_seqlens, total_tokens, q, k, v, g, b, slot_ids, pool, num_slots,
                        init_from_pool, out, num_snaps, snap_seq, snap_tokens, snap_slot, workspace,
                        workspace_bytes, err_flag, stream);
}

int kda_prefill_fused(const kda_dims *dims, int32_t num_seqs, const int32_t *cu_seqlens, int64_t total_tokens,
                      const void *q, const void *k, const void *v, const float *g, const void *b,
                      const int32_t *slot_ids, float *pool, int64_t num_slots, int32_t init_from_pool,
                      const kda_fused_io *io, void *out, void *workspace, size_t workspace_bytes,
                      int32_t *err_flag, void *stream) {
    if (io == nullptr) return KDA_ERR_INVALID_ARG;
    return prefill_impl(dims, num_seqs, cu_seqlens, total_tokens, q, k, v, g, b, slot_ids, pool, num_slots,
                        init_from_pool, out, 0, nullptr, nullptr, nullptr, workspace, workspace_bytes, err_flag,
                        stream, io);
}

}  // extern "C"
