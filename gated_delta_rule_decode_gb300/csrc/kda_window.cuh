// Draft-window pieces shared by the ReplaySSM verify kernels (CUDA-core and
// tensor-core row phases): token coefficients, value rows, window products,
// the per-row recurrence and the output store.
#pragma once

#include "kda.h"
#include "kda_internal.h"
#include "kda_rowmath.cuh"

namespace kda {

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

// Token coefficients as group tasks: task t = kind * D + j prepares draft
// token j's normalised key (kind 0, with the decode kernel's routine, so the
// key and beta records replay exactly like decode), normalised query
// (kind 1) or decay alpha = exp(g) (kind 2, with the gate record).  The norm's
// reduction is a full-warp shuffle: every lane of the warp calls this, and a
// group without a task (act false) computes a dummy and stores nothing.
template <int DK, typename T>
__device__ __forceinline__ void window_coeffs(const VerifyParams &p, int n, int h, int t, bool act, int l, float *kh,
                                              float *qh, float *al, float *beta) {
    const int D = p.D;
    const int tt = act ? t : 0;
    const int kind = tt / D, j = tt - kind * D;
    const int64_t tk = ((int64_t)n * D + j) * p.H + h;
    LaneVec<DK> x;
    if (kind == 0)
        load_lane_vec<DK, T>(static_cast<const T *>(p.k) + tk * DK, l, x);
    else if (kind == 1)
        load_lane_vec<DK, T>(static_cast<const T *>(p.q) + tk * DK, l, x);
    else
        load_lane_vec<DK, float>(p.g + tk * DK, l, x);
    LaneVec<DK> xn = x;
    l2norm_lane<DK>(xn, p.eps);
    if (!act) return;
    if (kind == 0) {
        store_lane_vec<DK>(kh + j * DK, l, xn);
        store_lane_vec<DK>(p.rec_k_hat + tk * DK, l, xn);
        if (l == 0) {
            const float bt = sigmoid_f(Elem<T>::load1(static_cast<const T *>(p.b) + tk));
            beta[j] = bt;
            if (p.rec_beta) p.rec_beta[tk] = bt;
        }
    } else if (kind == 1) {
        store_lane_vec<DK>(qh + j * DK, l, xn);
    } else {
        store_lane_vec<DK>(p.rec_g + tk * DK, l, x);
        exp_lane<DK>(x);
        store_lane_vec<DK>(al + j * DK, l, x);
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
            if (p.rec_v)
                *reinterpret_cast<uint4 *>(static_cast<T *>(p.rec_v) + value_vec_offset<T>(p, n, h, idx)) = vv.x[u];
            const int j = idx >> sh, col = (idx & ((p.dv / E) - 1)) * E;
            const T *e = reinterpret_cast<const T *>(&vv.x[u]);
#pragma unroll
            for (int i = 0; i < E; ++i) v[j * kMaxDv + col + i] = Elem<T>::to_f(e[i]);
        }
    }
}

// Window products as independent tasks, one per group: task t < D is
// (m = -1, j = t) and yields K~_j and Q~_j (written by store_kq, which picks
// the layout) and p_jj; the others enumerate the pairs m < j and yield a_jm
// and p_jm.  A task forms w = prod_{l=m+1..j} alpha_l
// in that order, then x = k^_m w (k^_m taken as all ones for m = -1).  Every
// lane of a warp takes part (full-warp reductions); `act` marks a real task.
template <int DK, typename StoreKQ>
__device__ __forceinline__ void window_pair(int t, bool act, int D, int l, const float *kh, const float *qh,
                                            const float *al, float *kt, float *qt, float *A, float *P, int ldp,
                                            StoreKQ store_kq) {
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
    const float kq = group_sum(lane_dot<DK>(kj, qj));  // p_jj (used by the m = -1 task)
    if (act) {
        if (m < 0) {
            if (l == 0) P[j * ldp + j] = kq;
            mul_lane<DK>(kj, x);
            mul_lane<DK>(qj, x);
            store_kq(kt, qt, j, l, kj, qj);
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
                                            const float *beta, const float *v, float *rt, float *ct, float *o,
                                            float *urec = nullptr, int64_t ustride = 0) {
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
            if (urec && l < 4) urec[j * ustride + row] = u[j];  // u record of (token j, row)
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

}  // namespace kda
