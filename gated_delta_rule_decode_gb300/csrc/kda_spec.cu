// ReplaySSM speculative verify (record) and commit (replay) kernels.
//
// "2.8x faster Kimi K3 inference on CANN", section 04 "ReplaySSM": while the
// draft tokens are verified only the per-token update records needed for a
// replay are kept; once the accepted length is known, the commit starts from
// the committed state and applies the accepted records in order, so no full
// state is ever stored per candidate token.
//
// verify_kernel: a CTA owns one (sequence, head, block of 16*R state rows),
// reads those rows once into registers, runs the D draft tokens over them in
// order (emitting every token's output), writes the records, and never writes
// the pool.  replay_kernel: a CTA owns the same tile, skips it without any
// memory access when a = 0, else reads the rows once, applies a records and
// writes them back.  Both use the row math of the decode kernel, so replaying
// a records reproduces a decode calls bit for bit.
#include "kda.h"
#include "kda_internal.h"
#include "kda_rowmath.cuh"

namespace kda {

constexpr int kSpecWarps = 4;
constexpr int kRowStride = kSpecWarps * kGroupsPerWarp;  // 16

constexpr int kMaxDraft = 16;

// Per-token coefficients of all draft tokens, staged in shared memory so that
// the sequential token loop never waits on global memory.  Each 8-lane group
// computes one token with the decode kernel's routine (same lane mapping,
// same bits) and stores it at channel positions.
template <int DK, int ROWS>
struct SpecSmem {
    float kh[kMaxDraft][DK];
    float qh[kMaxDraft][DK];
    float al[kMaxDraft][DK];
    float beta[kMaxDraft];
    float kq[kMaxDraft];
    float v[kMaxDraft][ROWS];
};

template <int DK, typename T, int R>
__global__ void __launch_bounds__(kSpecWarps * 32) verify_kernel(const VerifyParams p) {
    constexpr int ROWS = kRowStride * R;
    __shared__ __align__(16) SpecSmem<DK, ROWS> sm;
    const int nblk = p.dv / ROWS;
    const int64_t item = blockIdx.x;
    const int blk = (int)(item % nblk);
    const int64_t sh = item / nblk;
    const int h = (int)(sh % p.H);
    const int n = (int)(sh / p.H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int gid = warp * kGroupsPerWarp + grp;  // 0..15
    const int row0 = blk * ROWS + gid;

    const int slot = __ldg(p.slot_ids + n);
    const bool valid = slot >= 0 && (int64_t)slot < p.num_slots;
    if (slot >= 0 && !valid && blk == 0 && threadIdx.x == 0 && p.err_flag)
        atomicOr(p.err_flag, KDA_DEVERR_SLOT);

    LaneVec<DK> s[R];
    if (valid) {
        const float *S = p.pool + ((int64_t)slot * p.H + h) * (int64_t)p.dv * DK;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) load_row<DK>(S + (int64_t)(row0 + rr * kRowStride) * DK, l, s[rr]);
    }

    // Phase 1: group gid prepares draft token gid (all tokens in parallel).
    // Every lane of the warp runs make_coeffs, whose reductions are full-warp
    // shuffles: groups past the last draft token recompute the last token
    // and discard the result.
    {
        const bool mine = gid < p.D;
        const int j = mine ? gid : p.D - 1;
        const int64_t tk = ((int64_t)n * p.D + j) * p.H + h;
        TokenCoeffs<DK> tc;
        const float bb = Elem<T>::load1(static_cast<const T *>(p.b) + tk);
        make_coeffs<DK, T>(tc, static_cast<const T *>(p.q) + tk * DK,
                           static_cast<const T *>(p.k) + tk * DK, p.g + tk * DK, bb, p.eps, l);
        if (mine) {
            store_lane_vec<DK>(sm.kh[j], l, tc.kh);
            store_lane_vec<DK>(sm.qh[j], l, tc.qh);
            store_lane_vec<DK>(sm.al[j], l, tc.alpha);
            if (l == 0) {
                sm.beta[j] = tc.beta;
                sm.kq[j] = tc.kq;
            }
            if (blk == 0) {  // the key, gate and beta records (one writer per token)
                float *kr = p.rec_k_hat + tk * DK;
                float *gr = p.rec_g + tk * DK;
                const float *gi = p.g + tk * DK;
                store_lane_vec<DK>(kr, l, tc.kh);
#pragma unroll
                for (int jj = 0; jj < DK / 32; ++jj)
                    *reinterpret_cast<float4 *>(gr + 4 * l + 32 * jj) =
                        __ldg(reinterpret_cast<const float4 *>(gi + 4 * l + 32 * jj));
                if (l == 0) p.rec_beta[tk] = tc.beta;
            }
        }
    }
    // this CTA's value rows of every draft token; value records are bit copies
    for (int idx = threadIdx.x; idx < p.D * ROWS; idx += kSpecWarps * 32) {
        const int j = idx / ROWS, r = idx % ROWS;
        const int64_t tk = ((int64_t)n * p.D + j) * p.H + h;
        const int64_t off = tk * p.dv + blk * ROWS + r;
        const T raw = static_cast<const T *>(p.v)[off];
        static_cast<T *>(p.rec_v)[off] = raw;
        sm.v[j][r] = Elem<T>::to_f(raw);
    }
    __syncthreads();

    // Phase 2: the draft tokens in order over the rows held in registers.
    for (int j = 0; j < p.D; ++j) {
        const int64_t tk = ((int64_t)n * p.D + j) * p.H + h;
        T *orow = static_cast<T *>(p.out) + tk * p.dv;
        TokenCoeffs<DK> tc;
        load_lane_vec_smem<DK>(sm.kh[j], l, tc.kh);
        load_lane_vec_smem<DK>(sm.qh[j], l, tc.qh);
        load_lane_vec_smem<DK>(sm.al[j], l, tc.alpha);
        tc.beta = sm.beta[j];
        tc.kq = sm.kq[j];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int row = row0 + rr * kRowStride;
            float o = 0.f;
            if (valid) {
                float u;
                const float c = row_update<DK, true>(s[rr], tc, sm.v[j][gid + rr * kRowStride], &u);
                o = row_output(c, u, tc.kq, p.scale);
            }
            if (l == 0) Elem<T>::store1(orow + row, o);
        }
    }
}

template <int DK, typename T, int R>
__global__ void __launch_bounds__(kSpecWarps * 32) replay_kernel(const ReplayParams p) {
    constexpr int ROWS = kRowStride * R;
    __shared__ __align__(16) SpecSmem<DK, ROWS> sm;
    const int nblk = p.dv / ROWS;
    const int64_t item = blockIdx.x;
    const int blk = (int)(item % nblk);
    const int64_t sh = item / nblk;
    const int h = (int)(sh % p.H);
    const int n = (int)(sh / p.H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int gid = warp * kGroupsPerWarp + grp;
    const int row0 = blk * ROWS + gid;

    const int a = __ldg(p.num_accepted + n);
    const int slot = __ldg(p.slot_ids + n);
    const bool report = (blk == 0 && h == 0 && threadIdx.x == 0 && p.err_flag);
    if (a < 0 || a > p.D) {
        if (report) atomicOr(p.err_flag, KDA_DEVERR_ACCEPTED);
        return;
    }
    if (slot < 0) return;
    if ((int64_t)slot >= p.num_slots) {
        if (report) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    if (a == 0) return;  // nothing accepted: no memory access at all

    float *S = p.pool + ((int64_t)slot * p.H + h) * (int64_t)p.dv * DK;
    LaneVec<DK> s[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) load_row<DK>(S + (int64_t)(row0 + rr * kRowStride) * DK, l, s[rr]);

    // Phase 1: group gid loads record gid (all accepted records in parallel).
    if (gid < a) {
        const int64_t tk = ((int64_t)n * p.D + gid) * p.H + h;
        TokenCoeffs<DK> tc;
        coeffs_from_record<DK>(tc, p.rec_k_hat + tk * DK, p.rec_g + tk * DK, __ldg(p.rec_beta + tk), l);
        store_lane_vec<DK>(sm.kh[gid], l, tc.kh);
        store_lane_vec<DK>(sm.al[gid], l, tc.alpha);
        if (l == 0) sm.beta[gid] = tc.beta;
    }
    for (int idx = threadIdx.x; idx < a * ROWS; idx += kSpecWarps * 32) {
        const int j = idx / ROWS, r = idx % ROWS;
        const int64_t tk = ((int64_t)n * p.D + j) * p.H + h;
        sm.v[j][r] = Elem<T>::load1(static_cast<const T *>(p.rec_v) + tk * p.dv + blk * ROWS + r);
    }
    __syncthreads();

    for (int j = 0; j < a; ++j) {
        TokenCoeffs<DK> tc;
        load_lane_vec_smem<DK>(sm.kh[j], l, tc.kh);
        load_lane_vec_smem<DK>(sm.al[j], l, tc.alpha);
        tc.beta = sm.beta[j];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            float u;
            row_update<DK, false>(s[rr], tc, sm.v[j][gid + rr * kRowStride], &u);
        }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) store_row<DK>(S + (int64_t)(row0 + rr * kRowStride) * DK, l, s[rr]);
}

template <int DK, typename T>
static cudaError_t launch_verify_t(const VerifyParams &p, cudaStream_t st) {
    // 64 state rows per CTA where dv allows (measured faster than 32 or 16:
    // the per-token coefficients are computed once per CTA, so larger row
    // blocks amortise them), else 32.
    if (p.dv % (kRowStride * 4) == 0) {
        const int64_t grid = (int64_t)p.batch * p.H * (p.dv / (kRowStride * 4));
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        verify_kernel<DK, T, 4><<<(unsigned)grid, kSpecWarps * 32, 0, st>>>(p);
    } else {
        const int64_t grid = (int64_t)p.batch * p.H * (p.dv / (kRowStride * 2));
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        verify_kernel<DK, T, 2><<<(unsigned)grid, kSpecWarps * 32, 0, st>>>(p);
    }
    return cudaGetLastError();
}

template <int DK, typename T>
static cudaError_t launch_replay_t(const ReplayParams &p, cudaStream_t st) {
    // 64 rows per CTA where dv allows (each lane keeps 4 rows, more bytes in
    // flight), else 32
    if (p.dv % (kRowStride * 4) == 0) {
        const int64_t grid = (int64_t)p.batch * p.H * (p.dv / (kRowStride * 4));
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        replay_kernel<DK, T, 4><<<(unsigned)grid, kSpecWarps * 32, 0, st>>>(p);
    } else {
        const int64_t grid = (int64_t)p.batch * p.H * (p.dv / (kRowStride * 2));
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        replay_kernel<DK, T, 2><<<(unsigned)grid, kSpecWarps * 32, 0, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_verify(const VerifyParams &p, int dk, int dtype, cudaStream_t st) {
    if (dtype == KDA_DT_BF16) {
        if (dk == 128) return launch_verify_t<128, __nv_bfloat16>(p, st);
        if (dk == 64) return launch_verify_t<64, __nv_bfloat16>(p, st);
        return launch_verify_t<32, __nv_bfloat16>(p, st);
    }
    if (dk == 128) return launch_verify_t<128, float>(p, st);
    if (dk == 64) return launch_verify_t<64, float>(p, st);
    return launch_verify_t<32, float>(p, st);
}

cudaError_t launch_replay(const ReplayParams &p, int dk, int dtype, cudaStream_t st) {
    if (dtype == KDA_DT_BF16) {
        if (dk == 128) return launch_replay_t<128, __nv_bfloat16>(p, st);
        if (dk == 64) return launch_replay_t<64, __nv_bfloat16>(p, st);
        return launch_replay_t<32, __nv_bfloat16>(p, st);
    }
    if (dk == 128) return launch_replay_t<128, float>(p, st);
    if (dk == 64) return launch_replay_t<64, float>(p, st);
    return launch_replay_t<32, float>(p, st);
}

}  // namespace kda
