// ReplaySSM speculative verify (record) and commit (replay) kernels.
//
// "2.8x faster Kimi K3 inference on CANN", section 04 "ReplaySSM": while the
// draft tokens are verified only the per-token update records needed for a
// replay are kept; once the accepted length is known, the commit starts from
// the committed state and applies the accepted records in order, so no full
// state is ever stored per candidate token.
//
// verify_kernel: a CTA owns one (sequence, head).  It reads the committed
// state once, computes every draft token's output in chunk form over that
// state (the algebra is in kda_window.cuh), writes the records, and never
// writes the pool.  The records come from the decode kernel's coefficient
// routine, bit for bit.  This is the general path; bf16 windows of up to 8
// tokens at dk = dv = 128 take the window + tensor-core state kernels of
// kda_spec_tc.cu (they need the caller's workspace).
// replay_kernel: a CTA owns one (sequence, head, block of 16*R state rows).
// It skips the tile without any memory access when a = 0.  Otherwise it
// reads the rows once, applies a records with the decode kernel's row math
// and writes them back, so replaying a records reproduces a decode calls bit
// for bit.
#include "kda.h"
#include "kda_internal.h"
#include "kda_bulk.cuh"
#include "kda_check.cuh"
#include "kda_rowmath.cuh"
#include "kda_window.cuh"

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

// ------------------------------------------------------------------ verify kernel
//
// One CTA of 2 * dv threads per (sequence, head): the token coefficients, the
// window products and the row phase, separated by CTA barriers; the state's
// bulk copy and the value rows are in flight from the start.

template <int DK, int DMAX>
struct VerifySmem {
    float kh[DMAX][DK];   // k^_j
    float qh[DMAX][DK];   // q^_j
    float al[DMAX][DK];   // alpha_j
    float kt[DMAX][DK];   // K~_j
    float qt[DMAX][DK];   // Q~_j
    float A[DMAX][DMAX];  // a_jm, m < j
    float P[DMAX][DMAX];  // p_jm, m <= j
    float beta[DMAX];
    float v[DMAX][kMaxDv];
    float rt[DMAX][kMaxDv];  // S0[i] . K~_j
    float ct[DMAX][kMaxDv];  // S0[i] . Q~_j
    float o[DMAX][kMaxDv];
    uint64_t bar;            // completion of the state copy
};

// The committed state block (dv x dk fp32) follows the struct, 128-byte aligned.
template <int DK, int DMAX>
__host__ __device__ constexpr size_t verify_state_offset() {
    return (sizeof(VerifySmem<DK, DMAX>) + 127) / 128 * 128;
}

template <int DK, typename T, int DMAX>
__global__ void __launch_bounds__(256, (DMAX <= 8 ? 2 : 1)) verify_kernel(const VerifyParams p) {
    extern __shared__ __align__(128) unsigned char verify_smem[];
    VerifySmem<DK, DMAX> &sm = *reinterpret_cast<VerifySmem<DK, DMAX> *>(verify_smem);
    float *st = reinterpret_cast<float *>(verify_smem + verify_state_offset<DK, DMAX>());
    const int ngroups = (blockDim.x >> 5) * kGroupsPerWarp;  // dv / 4
    const int64_t sh = blockIdx.x;                            // (sequence, head)
    const int h = (int)(sh % p.H);
    const int n = (int)(sh / p.H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int gid = warp * kGroupsPerWarp + grp;
    const int D = p.D;

    // checked build: the window's token-heads (inputs, outputs, records) and
    // the previous window's records
    if (!in_bounds((int64_t)n * D * p.H + h, (int64_t)(D - 1) * p.H + 1, (int64_t)p.batch * D * p.H, p.err_flag) ||
        (p.prev_accepted != nullptr &&
         !in_bounds((int64_t)n * p.prev_D * p.H + h, (int64_t)(p.prev_D - 1) * p.H + 1,
                    (int64_t)p.batch * p.prev_D * p.H, p.err_flag)))
        return;
    const int slot = __ldg(p.slot_ids + n);
    const bool valid = slot >= 0 && (int64_t)slot < p.num_slots;
    if (slot >= 0 && !valid && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
    if (valid && !in_bounds(((int64_t)slot * p.H + h) * p.dv * DK, (int64_t)p.dv * DK,
                            p.num_slots * p.H * (int64_t)p.dv * DK, p.err_flag))
        return;

    // S0 is requested first, as one bulk copy into shared memory, so that the
    // coefficient phases overlap the load and hold no state registers
    const uint32_t state_bytes = (uint32_t)p.dv * DK * 4;
    if (valid && threadIdx.x == 0) {
        mbar_init(&sm.bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&sm.bar, state_bytes);
        bulk_g2s(st, p.pool + ((int64_t)slot * p.H + h) * (int64_t)p.dv * DK, state_bytes, &sm.bar);
    }

    ValueVecs<T> vv;
    window_values_load<T>(p, n, h, threadIdx.x, blockDim.x, vv);
    for (int base = 0; base < 3 * D; base += ngroups) {
        if (base + warp * kGroupsPerWarp >= 3 * D) break;  // warp-uniform
        window_coeffs<DK, T>(p, n, h, base + gid, base + gid < 3 * D, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0],
                             sm.beta);
    }
    window_values_store<T>(p, n, h, threadIdx.x, blockDim.x, vv, &sm.v[0][0]);
    __syncthreads();
    const int ntasks = D + D * (D - 1) / 2;
    auto store_kq = [&](float *kt, float *qt, int j, int ll, const LaneVec<DK> &kj, const LaneVec<DK> &qj) {
        store_lane_vec<DK>(kt + j * DK, ll, kj);
        store_lane_vec<DK>(qt + j * DK, ll, qj);
    };
    for (int base = 0; base < ntasks; base += ngroups) {
        if (base + warp * kGroupsPerWarp >= ntasks) break;  // warp-uniform
        window_pair<DK>(base + gid, base + gid < ntasks, D, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0],
                        &sm.kt[0][0], &sm.qt[0][0], &sm.A[0][0], &sm.P[0][0], DMAX, store_kq);
    }
    __syncthreads();
    float *urec = p.rec_u ? p.rec_u + ((int64_t)n * D * p.H + h) * p.dv : nullptr;
    const int64_t ustride = (int64_t)p.H * p.dv;
    if (valid) {
        // the outcome is made CTA-uniform so that no thread skips a barrier
        if (__syncthreads_and(mbar_wait(&sm.bar, 0)) == 0) {
            if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            mbar_wait_drain(&sm.bar, 0);  // the copy still in flight
            return;
        }
        // fused commit of the previous window's accepted u records: each
        // group updates its rows in shared memory and writes them back to
        // the pool before the window reads them
        if (p.prev_accepted) {
            const int a = __ldg(p.prev_accepted + n);
            if (a < 0 || a > p.prev_D) {
                if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_ACCEPTED);
            } else if (a > 0) {
                // (the fused call writes the committed state: its pool is not read-only)
                float *Sp = const_cast<float *>(p.pool) + ((int64_t)slot * p.H + h) * (int64_t)p.dv * DK;
#pragma unroll 1
                for (int rr = 0; rr < kVerifyRows; ++rr) {
                    const int row = gid + rr * ngroups;
                    LaneVec<DK> sr;
                    load_lane_vec_smem<DK>(st + row * DK, l, sr);
#pragma unroll 1
                    for (int j = 0; j < a; ++j) {
                        const int64_t tk = ((int64_t)n * p.prev_D + j) * p.H + h;
                        commit_u_row<DK>(sr, p.prev_k_hat + tk * DK, p.prev_g + tk * DK, __ldg(p.prev_u + tk * p.dv + row), l);
                    }
                    store_lane_vec<DK>(st + row * DK, l, sr);
                    store_row<DK>(Sp + (int64_t)row * DK, l, sr);
                }
                __syncthreads();
            }
        }
        window_rows<DK, DMAX>(st, ngroups, gid, l, D, p.scale, &sm.kt[0][0], &sm.qt[0][0], &sm.A[0][0], &sm.P[0][0],
                              sm.beta, &sm.v[0][0], &sm.rt[0][0], &sm.ct[0][0], &sm.o[0][0], urec, ustride);
    } else if (urec) {
        // a skipped entry's u records are zero
        for (int idx = threadIdx.x; idx < D * p.dv; idx += blockDim.x)
            urec[(idx / p.dv) * ustride + idx % p.dv] = 0.f;
    }
    __syncthreads();
    window_store<T>(p, n, h, threadIdx.x, blockDim.x, &sm.o[0][0], valid);
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
    // checked build: this CTA's state rows and the sequence's records
    if (!in_bounds(((int64_t)slot * p.H + h) * p.dv * DK + (int64_t)blk * ROWS * DK, (int64_t)ROWS * DK,
                   p.num_slots * p.H * (int64_t)p.dv * DK, p.err_flag) ||
        !in_bounds((int64_t)n * p.D * p.H + h, (int64_t)(p.D - 1) * p.H + 1, (int64_t)p.batch * p.D * p.H,
                   p.err_flag))
        return;

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
    // this tile's value records in 16-byte vectors, at most two per thread
    // (D <= 16, 4-byte elements), all in flight at once
    {
        constexpr int E = 16 / sizeof(T);
        constexpr int VPT = ROWS / E;  // vectors per token
        const int total = a * VPT;
        uint4 vbuf[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = threadIdx.x + u * kSpecWarps * 32;
            if (idx < total) {
                const int j = idx / VPT, c = (idx % VPT) * E;
                const int64_t tk = ((int64_t)n * p.D + j) * p.H + h;
                vbuf[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const T *>(p.rec_v) + tk * p.dv +
                                                                blk * ROWS + c));
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = threadIdx.x + u * kSpecWarps * 32;
            if (idx < total) {
                const int j = idx / VPT, c = (idx % VPT) * E;
                const T *e = reinterpret_cast<const T *>(&vbuf[u]);
#pragma unroll
                for (int i = 0; i < E; ++i) sm.v[j][c + i] = Elem<T>::to_f(e[i]);
            }
        }
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

// Commit from u records (the ReplaySSM variant that stores u = beta (v - S'k^)):
// per accepted token j, S <- S diag(exp g_j) + u_j k^_j^T.  The same tiles as
// replay_kernel; no dot products.  The element arithmetic (one multiply by
// alpha, then one fused multiply-add) is the fused commit's, bit for bit.
template <int DK, int R>
__global__ void __launch_bounds__(kSpecWarps * 32) replay_u_kernel(const ReplayParams p) {
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
    // checked build: this CTA's state rows and the sequence's records
    if (!in_bounds(((int64_t)slot * p.H + h) * p.dv * DK + (int64_t)blk * ROWS * DK, (int64_t)ROWS * DK,
                   p.num_slots * p.H * (int64_t)p.dv * DK, p.err_flag) ||
        !in_bounds((int64_t)n * p.D * p.H + h, (int64_t)(p.D - 1) * p.H + 1, (int64_t)p.batch * p.D * p.H,
                   p.err_flag))
        return;

    float *S = p.pool + ((int64_t)slot * p.H + h) * (int64_t)p.dv * DK;
    LaneVec<DK> s[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) load_row<DK>(S + (int64_t)(row0 + rr * kRowStride) * DK, l, s[rr]);
    // group gid stages record gid's k^ and alpha; the tile's u values
    if (gid < a) {
        const int64_t tk = ((int64_t)n * p.D + gid) * p.H + h;
        LaneVec<DK> kh, al;
        load_lane_vec<DK, float>(p.rec_k_hat + tk * DK, l, kh);
        load_lane_vec<DK, float>(p.rec_g + tk * DK, l, al);
        exp_lane<DK>(al);
        store_lane_vec<DK>(sm.kh[gid], l, kh);
        store_lane_vec<DK>(sm.al[gid], l, al);
    }
    for (int idx = threadIdx.x; idx < a * ROWS; idx += kSpecWarps * 32) {
        const int j = idx / ROWS, c = idx % ROWS;
        sm.v[j][c] = __ldg(p.rec_u + (((int64_t)n * p.D + j) * p.H + h) * p.dv + blk * ROWS + c);
    }
    __syncthreads();
    for (int j = 0; j < a; ++j) {
        LaneVec<DK> kh, al;
        load_lane_vec_smem<DK>(sm.kh[j], l, kh);
        load_lane_vec_smem<DK>(sm.al[j], l, al);
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const float u = sm.v[j][gid + rr * kRowStride];
            const float2 u2 = make_float2(u, u);
#pragma unroll
            for (int i = 0; i < DK / 16; ++i) s[rr].v[i] = __ffma2_rn(u2, kh.v[i], __fmul2_rn(s[rr].v[i], al.v[i]));
        }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) store_row<DK>(S + (int64_t)(row0 + rr * kRowStride) * DK, l, s[rr]);
}

template <int DK, typename T, int DMAX>
static cudaError_t launch_verify_d(const VerifyParams &p, cudaStream_t st) {
    const size_t smem = verify_state_offset<DK, DMAX>() + (size_t)p.dv * DK * 4;
    const cudaError_t e = cudaFuncSetAttribute(verify_kernel<DK, T, DMAX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)p.batch * p.H;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    verify_kernel<DK, T, DMAX><<<(unsigned)grid, 2 * p.dv, smem, st>>>(p);
    return cudaGetLastError();
}

template <int DK, typename T>
static cudaError_t launch_verify_t(const VerifyParams &p, cudaStream_t st) {
    // dv in {32, 64, 128}: dv / 16 warps own 4 rows per 8-lane group; the
    // window length picks the size of the per-row register arrays
    if (p.dv % (kVerifyRows * kGroupsPerWarp) != 0 || p.dv > kMaxDv || (p.dv & (p.dv - 1)) != 0)
        return cudaErrorNotSupported;
    if (p.D <= 8) return launch_verify_d<DK, T, 8>(p, st);
    if (p.D <= kMaxDraft) return launch_verify_d<DK, T, kMaxDraft>(p, st);
    return cudaErrorNotSupported;
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
    if (verify_tc_supported(p, dk, dtype)) {
        if (p.prev_accepted == nullptr) return launch_verify_tc(p, st);
        // A commit before the verify on the tensor-core shape: the commit's
        // own launch (replay_u_kernel), then the verify from the committed
        // state, in stream order.  One launch doing both (the state kernel
        // committing its staged tile, storing it back and then verifying)
        // was slower, 174 us against 157 us at 128 x 7 x 32 heads: with the
        // previous window's staging it held two CTAs per SM instead of three
        // and ran its stages one after another.  Running the commit beside
        // the window kernel (which does not read the state) took 162 us.
        ReplayParams r{};
        r.rec_k_hat = p.prev_k_hat;
        r.rec_g = p.prev_g;
        r.rec_u = p.prev_u;
        r.num_accepted = p.prev_accepted;
        r.slot_ids = p.slot_ids;
        r.pool = const_cast<float *>(p.pool);
        r.num_slots = p.num_slots;
        r.err_flag = p.err_flag;
        r.batch = p.batch;
        r.D = p.prev_D;
        r.H = p.H;
        r.dv = p.dv;
        const cudaError_t e = launch_replay_u(r, dk, st);
        if (e != cudaSuccess) return e;
        VerifyParams v = p;
        v.prev_k_hat = v.prev_g = v.prev_u = nullptr;
        v.prev_accepted = nullptr;
        v.prev_D = 0;
        return launch_verify_tc(v, st);
    }
    if (dtype == KDA_DT_BF16) {
        if (dk == 128) return launch_verify_t<128, __nv_bfloat16>(p, st);
        if (dk == 64) return launch_verify_t<64, __nv_bfloat16>(p, st);
        return launch_verify_t<32, __nv_bfloat16>(p, st);
    }
    if (dk == 128) return launch_verify_t<128, float>(p, st);
    if (dk == 64) return launch_verify_t<64, float>(p, st);
    return launch_verify_t<32, float>(p, st);
}

template <int DK>
static cudaError_t launch_replay_u_t(const ReplayParams &p, cudaStream_t st) {
    if (p.dv % (kRowStride * 4) == 0) {
        const int64_t grid = (int64_t)p.batch * p.H * (p.dv / (kRowStride * 4));
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        replay_u_kernel<DK, 4><<<(unsigned)grid, kSpecWarps * 32, 0, st>>>(p);
    } else {
        const int64_t grid = (int64_t)p.batch * p.H * (p.dv / (kRowStride * 2));
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        replay_u_kernel<DK, 2><<<(unsigned)grid, kSpecWarps * 32, 0, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_replay_u(const ReplayParams &p, int dk, cudaStream_t st) {
    if (dk == 128) return launch_replay_u_t<128>(p, st);
    if (dk == 64) return launch_replay_u_t<64>(p, st);
    return launch_replay_u_t<32>(p, st);
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
