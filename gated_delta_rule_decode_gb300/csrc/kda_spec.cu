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
// state (below), writes the records, and never writes the pool.  The records
// come from the decode kernel's coefficient routine, bit for bit.
// replay_kernel: a CTA owns one (sequence, head, block of 16*R state rows).
// It skips the tile without any memory access when a = 0.  Otherwise it
// reads the rows once, applies a records with the decode kernel's row math
// and writes them back, so replaying a records reproduces a decode calls bit
// for bit.
#include "kda.h"
#include "kda_internal.h"
#include "kda_bulk.cuh"
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

// ------------------------------------------------------------------ verify
//
// The D draft tokens of one (sequence, head) are the token recurrence unrolled
// over the window, starting from the committed state S0:
//   E_j   = prod_{l<=j} alpha_l                  (per key channel)
//   K~_j  = k^_j E_j,   Q~_j = q^_j E_j
//   a_jm  = sum_c k^_m[c] k^_j[c] prod_{l=m+1..j} alpha_l[c]   (m < j)
//   p_jm  = sum_c k^_m[c] q^_j[c] prod_{l=m+1..j} alpha_l[c]   (m <= j)
// and for every state row i
//   u_j[i] = beta_j (v_j[i] - S0[i].K~_j - sum_{m<j} a_jm u_m[i])
//   o_j[i] = scale (S0[i].Q~_j + sum_{m<=j} p_jm u_m[i]).
// A row then needs 2D independent dot products with S0, instead of D
// dependent read-modify-write passes, plus a D x D triangular recurrence of
// scalars.  The decay factors are running products of alpha = exp(g), so a
// strongly decaying channel underflows towards zero and nothing overflows.

constexpr int kVerifyRows = 4;   // state rows per 8-lane group
constexpr int kMaxDv = 128;

template <int DK>
__device__ __forceinline__ void set_ones(LaneVec<DK> &x) {
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) x.v[i] = make_float2(1.f, 1.f);
}

template <int DK>
__device__ __forceinline__ void mul_lane(LaneVec<DK> &x, const LaneVec<DK> &y) {
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) x.v[i] = __fmul2_rn(x.v[i], y.v[i]);
}

// Token coefficients: one 8-lane group prepares draft token j0 of (n, h) with
// the decode kernel's routine (same bits, so the key records replay exactly
// like decode) and writes its records.  The routine's reductions are
// full-warp shuffles: every lane of the warp calls this, and a group with
// j0 >= D recomputes token D-1 and discards it.  P has leading dimension ldp.
template <int DK, typename T>
__device__ __forceinline__ void window_token(const VerifyParams &p, int n, int h, int j0, int l, float *kh,
                                             float *qh, float *al, float *beta, float *P, int ldp) {
    const int D = p.D;
    const bool mine = j0 < D;
    const int j = mine ? j0 : D - 1;
    const int64_t tk = ((int64_t)n * D + j) * p.H + h;
    TokenCoeffs<DK> tc;
    const float bb = Elem<T>::load1(static_cast<const T *>(p.b) + tk);
    make_coeffs<DK, T>(tc, static_cast<const T *>(p.q) + tk * DK, static_cast<const T *>(p.k) + tk * DK,
                       p.g + tk * DK, bb, p.eps, l);
    if (mine) {
        store_lane_vec<DK>(kh + j * DK, l, tc.kh);
        store_lane_vec<DK>(qh + j * DK, l, tc.qh);
        store_lane_vec<DK>(al + j * DK, l, tc.alpha);
        store_lane_vec<DK>(p.rec_k_hat + tk * DK, l, tc.kh);
        const float *gi = p.g + tk * DK;
        float *gr = p.rec_g + tk * DK;
#pragma unroll
        for (int jj = 0; jj < DK / 32; ++jj)
            *reinterpret_cast<float4 *>(gr + 4 * l + 32 * jj) =
                __ldg(reinterpret_cast<const float4 *>(gi + 4 * l + 32 * jj));
        if (l == 0) {
            beta[j] = tc.beta;
            P[j * ldp + j] = tc.kq;  // p_jj = k^_j . q^_j
            p.rec_beta[tk] = tc.beta;
        }
    }
}

// Value rows of every draft token: bit copies into the records, fp32 into
// v[j][r] (leading dimension kMaxDv), in 16-byte vectors.  A CTA of 2 * dv
// threads holds at most two vectors per thread (D <= 16, 4-byte elements),
// so the loads are all issued first and stored after the caller's other work.
template <typename T>
struct ValueVecs {
    uint4 x[2];
};

template <typename T>
__device__ __forceinline__ int64_t value_vec_offset(const VerifyParams &p, int n, int h, int idx) {
    constexpr int E = 16 / sizeof(T);
    const int sh = __ffs(p.dv / E) - 1;  // log2(vectors per token row)
    const int j = idx >> sh, col = (idx & ((p.dv / E) - 1)) * E;
    return (((int64_t)n * p.D + j) * p.H + h) * p.dv + col;
}

template <typename T>
__device__ __forceinline__ void window_values_load(const VerifyParams &p, int n, int h, int tid, int nthreads,
                                                   ValueVecs<T> &vv) {
    const int total = p.D * p.dv * (int)sizeof(T) / 16;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int idx = tid + u * nthreads;
        if (idx < total)
            vv.x[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const T *>(p.v) +
                                                            value_vec_offset<T>(p, n, h, idx)));
    }
}

template <typename T>
__device__ __forceinline__ void window_values_store(const VerifyParams &p, int n, int h, int tid, int nthreads,
                                                    const ValueVecs<T> &vv, float *v) {
    constexpr int E = 16 / sizeof(T);
    const int total = p.D * p.dv * (int)sizeof(T) / 16;
    const int sh = __ffs(p.dv / E) - 1;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int idx = tid + u * nthreads;
        if (idx < total) {
            *reinterpret_cast<uint4 *>(static_cast<T *>(p.rec_v) + value_vec_offset<T>(p, n, h, idx)) = vv.x[u];
            const int j = idx >> sh, col = (idx & ((p.dv / E) - 1)) * E;
            const T *e = reinterpret_cast<const T *>(&vv.x[u]);
#pragma unroll
            for (int i = 0; i < E; ++i) v[j * kMaxDv + col + i] = Elem<T>::to_f(e[i]);
        }
    }
}

// Window products as independent tasks, one per group: task t < D is
// (m = -1, j = t) and yields K~_j and Q~_j; the others enumerate the pairs
// m < j and yield a_jm and p_jm.  A task forms w = prod_{l=m+1..j} alpha_l
// in that order, then x = k^_m w (k^_m taken as all ones for m = -1).  Every
// lane of a warp takes part (full-warp reductions); `act` marks a real task.
template <int DK>
__device__ __forceinline__ void window_pair(int t, bool act, int D, int l, const float *kh, const float *qh,
                                            const float *al, float *kt, float *qt, float *A, float *P, int ldp) {
    int m = -1, j = 0;
    if (!act) {
        j = 0;
    } else if (t < D) {
        j = t;
    } else {
        int r = t - D;
        m = 0;
        while (r >= D - 1 - m) {  // pairs (m, m+1 .. D-1) come in runs of D - 1 - m
            r -= D - 1 - m;
            ++m;
        }
        j = m + 1 + r;
    }
    LaneVec<DK> w, x, kj, qj;
    set_ones<DK>(w);
    for (int sidx = 0; sidx < D; ++sidx) {  // warp-uniform trip count
        const int li = m + 1 + sidx;
        if (li <= j) {
            LaneVec<DK> a;
            load_lane_vec_smem<DK>(al + li * DK, l, a);
            mul_lane<DK>(w, a);
        }
    }
    if (m >= 0) {
        load_lane_vec_smem<DK>(kh + m * DK, l, x);
        mul_lane<DK>(x, w);
    } else {
        x = w;
    }
    load_lane_vec_smem<DK>(kh + j * DK, l, kj);
    load_lane_vec_smem<DK>(qh + j * DK, l, qj);
    const float a = group_sum(lane_dot<DK>(x, kj));
    const float pp = group_sum(lane_dot<DK>(x, qj));
    if (act) {
        if (m < 0) {
            mul_lane<DK>(kj, x);
            mul_lane<DK>(qj, x);
            store_lane_vec<DK>(kt + j * DK, l, kj);
            store_lane_vec<DK>(qt + j * DK, l, qj);
        } else if (l == 0) {
            A[j * ldp + m] = a;
            P[j * ldp + m] = pp;
        }
    }
}

// Window rows: the group's rows gid + rr * ngroups of S0 (fp32 in shared
// memory, row length DK).  Per row the 2D dot products with K~ and Q~,
// reduced over the 8 lanes in transposed form (lanes l and l ^ 4 end with row
// l & 3) and parked in rt/ct, then the triangular recurrence for u and the
// outputs o[j][row].  The token loop of the dot products stays rolled:
// unrolled, the compiler hoists the next token's operands and spills.
template <int DK, int DMAX>
__device__ __forceinline__ void window_rows(const float *st, int ngroups, int gid, int l, int D, float scale,
                                            const float *kt, const float *qt, const float *A, const float *P,
                                            const float *beta, const float *v, float *rt, float *ct, float *o) {
    LaneVec<DK> s[kVerifyRows];
#pragma unroll
    for (int rr = 0; rr < kVerifyRows; ++rr) load_lane_vec_smem<DK>(st + (gid + rr * ngroups) * DK, l, s[rr]);
    const bool b0 = (l & 1) != 0, b1 = (l & 2) != 0;
    const int row = gid + (l & 3) * ngroups;
#pragma unroll 1
    for (int j = 0; j < D; ++j) {
        LaneVec<DK> kj, qj;
        load_lane_vec_smem<DK>(kt + j * DK, l, kj);
        load_lane_vec_smem<DK>(qt + j * DK, l, qj);
        float x[kVerifyRows][2];
#pragma unroll
        for (int rr = 0; rr < kVerifyRows; ++rr) {
            x[rr][0] = lane_dot<DK>(s[rr], kj);
            x[rr][1] = lane_dot<DK>(s[rr], qj);
        }
        float y[2][2];
#pragma unroll
        for (int hi = 0; hi < 2; ++hi)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float keep = b0 ? x[2 * hi + 1][c] : x[2 * hi][c];
                const float send = b0 ? x[2 * hi][c] : x[2 * hi + 1][c];
                y[hi][c] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 1));
            }
        float z[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const float keep = b1 ? y[1][c] : y[0][c];
            const float send = b1 ? y[0][c] : y[1][c];
            z[c] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 2));
            z[c] = __fadd_rn(z[c], __shfl_xor_sync(0xffffffffu, z[c], 4));
        }
        if (l < 4) {
            rt[j * kMaxDv + row] = z[0];
            ct[j * kMaxDv + row] = z[1];
        }
    }
    __syncwarp();
    float u[DMAX];
#pragma unroll
    for (int j = 0; j < DMAX; ++j) {
        u[j] = 0.f;
        if (j < D) {
            float r = rt[j * kMaxDv + row];
#pragma unroll
            for (int m = 0; m < j; ++m) r = __fmaf_rn(A[j * DMAX + m], u[m], r);
            u[j] = __fmul_rn(beta[j], __fsub_rn(v[j * kMaxDv + row], r));
            float c = ct[j * kMaxDv + row];
#pragma unroll
            for (int m = 0; m <= j; ++m) c = __fmaf_rn(P[j * DMAX + m], u[m], c);
            if (l < 4) o[j * kMaxDv + row] = __fmul_rn(scale, c);
        }
    }
}

// Outputs of one (sequence, head): o[j][r] (zeros for a skipped slot).
template <typename T>
__device__ __forceinline__ void window_store(const VerifyParams &p, int n, int h, int tid, int nthreads,
                                             const float *o, bool valid) {
    const int sh = __ffs(p.dv) - 1;
    for (int idx = tid; idx < (p.D << sh); idx += nthreads) {
        const int j = idx >> sh, r = idx & (p.dv - 1);
        T *orow = static_cast<T *>(p.out) + (((int64_t)n * p.D + j) * p.H + h) * p.dv;
        Elem<T>::store1(orow + r, valid ? o[j * kMaxDv + r] : 0.f);
    }
}

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

    const int slot = __ldg(p.slot_ids + n);
    const bool valid = slot >= 0 && (int64_t)slot < p.num_slots;
    if (slot >= 0 && !valid && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);

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
    for (int base = 0; base < D; base += ngroups) {
        if (base + warp * kGroupsPerWarp >= D) break;  // warp-uniform
        window_token<DK, T>(p, n, h, base + gid, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0], sm.beta,
                            &sm.P[0][0], DMAX);
    }
    window_values_store<T>(p, n, h, threadIdx.x, blockDim.x, vv, &sm.v[0][0]);
    __syncthreads();
    const int ntasks = D + D * (D - 1) / 2;
    for (int base = 0; base < ntasks; base += ngroups) {
        if (base + warp * kGroupsPerWarp >= ntasks) break;  // warp-uniform
        window_pair<DK>(base + gid, base + gid < ntasks, D, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0],
                        &sm.kt[0][0], &sm.qt[0][0], &sm.A[0][0], &sm.P[0][0], DMAX);
    }
    __syncthreads();
    if (valid) {
        // the outcome is made CTA-uniform so that no thread skips a barrier
        if (__syncthreads_and(mbar_wait(&sm.bar, 0)) == 0) {
            if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            mbar_wait(&sm.bar, 0);  // bounded second chance for the copy in flight
            return;
        }
        window_rows<DK, DMAX>(st, ngroups, gid, l, D, p.scale, &sm.kt[0][0], &sm.qt[0][0], &sm.A[0][0], &sm.P[0][0],
                              sm.beta, &sm.v[0][0], &sm.rt[0][0], &sm.ct[0][0], &sm.o[0][0]);
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
