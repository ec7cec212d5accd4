// Row-parallel KDA token math shared by the decode, verify and replay kernels.
//
// Rows of the V x K state (value channels) are independent for one token:
// row i needs only its own dk entries s_i, the normalised key k^, the
// normalised query q^, alpha = exp(g), beta and v_i.  Each row is owned by an
// 8-lane group of a warp; lane l of the group holds the dk/8 entries at key
// channels {4l + 32j + e : j < dk/32, e < 4}, so that one float4 access per
// j by the group covers 128 contiguous bytes of the row.  A lane keeps its
// entries as float2 pairs (channels 4l+32j+{0,1} and 4l+32j+{2,3}) and does
// the element-wise work with the paired fp32 instructions of sm_100
// (fma.rn.f32x2 and friends): each half is an ordinary round-to-nearest fp32
// operation, at half the instruction count.
//
// All arithmetic uses explicit round-to-nearest operations in one fixed order,
// so every kernel that calls these functions produces the same bits for the
// same token: replaying a record equals the decode step, bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kLanesPerRow = 8;
constexpr int kGroupsPerWarp = 32 / kLanesPerRow;

// ------------------------------------------------------------------ element io

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    // 4 consecutive elements starting at p (16-byte aligned)
    static __device__ __forceinline__ float4 load4(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ float load1(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ void store1(float *p, float x) { *p = x; }
    static __device__ __forceinline__ float to_f(float x) { return x; }
};

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
        uint2 raw = __ldg(reinterpret_cast<const uint2 *>(p));
        float4 r;
        r.x = __uint_as_float(raw.x << 16);
        r.y = __uint_as_float(raw.x & 0xffff0000u);
        r.z = __uint_as_float(raw.y << 16);
        r.w = __uint_as_float(raw.y & 0xffff0000u);
        return r;
    }
    static __device__ __forceinline__ float load1(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store1(__nv_bfloat16 *p, float x) {
        *p = __float2bfloat16_rn(x);
    }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// Streaming state access (each state block is touched once per call).
__device__ __forceinline__ float4 ld_state(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_state(float *p, float4 x) {
    __stcs(reinterpret_cast<float4 *>(p), x);
}

// Sum over the 8 lanes of a row group; every lane of the group receives the
// same bits (IEEE addition is commutative).
__device__ __forceinline__ float group_sum(float x) {
    x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 1));
    x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 2));
    x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 4));
    return x;
}

// ------------------------------------------------------------------ lane vectors

// A lane's dk/8 entries as dk/16 float2 pairs: v[2j] = channels 4l+32j+{0,1},
// v[2j+1] = channels 4l+32j+{2,3}.
template <int DK>
struct LaneVec {
    static constexpr int P = DK / 16;
    float2 v[P];
};

__device__ __forceinline__ void split4(float4 t, float2 &lo, float2 &hi) {
    lo = make_float2(t.x, t.y);
    hi = make_float2(t.z, t.w);
}

// Loads this lane's entries of a dk-vector of element type T.
template <int DK, typename T>
__device__ __forceinline__ void load_lane_vec(const T *p, int l, LaneVec<DK> &x) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) split4(Elem<T>::load4(p + 4 * l + 32 * j), x.v[2 * j], x.v[2 * j + 1]);
}

// Stores this lane's entries (fp32) to global or shared memory.
template <int DK>
__device__ __forceinline__ void store_lane_vec(float *p, int l, const LaneVec<DK> &x) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j)
        *reinterpret_cast<float4 *>(p + 4 * l + 32 * j) =
            make_float4(x.v[2 * j].x, x.v[2 * j].y, x.v[2 * j + 1].x, x.v[2 * j + 1].y);
}

// Loads this lane's entries from fp32 shared memory.
template <int DK>
__device__ __forceinline__ void load_lane_vec_smem(const float *p, int l, LaneVec<DK> &x) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j)
        split4(*reinterpret_cast<const float4 *>(p + 4 * l + 32 * j), x.v[2 * j], x.v[2 * j + 1]);
}

// Partial dot product of the lane's entries in a fixed association order:
// two paired accumulators (channels {0,1} and {2,3} of each float4 slot) run
// over the slots j in order, then are folded as ((a.x + b.x) + (a.y + b.y)).
template <int DK>
__device__ __forceinline__ float lane_dot(const LaneVec<DK> &s, const LaneVec<DK> &w) {
    float2 a = __fmul2_rn(s.v[0], w.v[0]);
    float2 b = __fmul2_rn(s.v[1], w.v[1]);
#pragma unroll
    for (int j = 1; j < DK / 32; ++j) {
        a = __ffma2_rn(s.v[2 * j], w.v[2 * j], a);
        b = __ffma2_rn(s.v[2 * j + 1], w.v[2 * j + 1], b);
    }
    const float2 t = __fadd2_rn(a, b);
    return __fadd_rn(t.x, t.y);
}

// ------------------------------------------------------------------ per-token coefficients

template <int DK>
struct TokenCoeffs {
    LaneVec<DK> kh;     // normalised key at this lane's channels
    LaneVec<DK> qh;     // normalised query at this lane's channels
    LaneVec<DK> alpha;  // exp(g) at this lane's channels
    float beta;         // sigmoid(b)
    float kq;           // k^ . q^ over all dk channels
};

// x^ = x * rsqrt(sum x^2 + eps) over the group's dk entries.
template <int DK>
__device__ __forceinline__ void l2norm_lane(LaneVec<DK> &x, float eps) {
    const float ss = group_sum(lane_dot<DK>(x, x));
    const float inv = rsqrtf(__fadd_rn(ss, eps));
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) x.v[i] = __fmul2_rn(x.v[i], inv2);
}

__device__ __forceinline__ float sigmoid_f(float b) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-b)));
}

template <int DK>
__device__ __forceinline__ void exp_lane(LaneVec<DK> &x) {
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) x.v[i] = make_float2(expf(x.v[i].x), expf(x.v[i].y));
}

// Q/K L2Norm, gate and beta processing for one token (decode and verify).
template <int DK, typename T>
__device__ __forceinline__ void make_coeffs(TokenCoeffs<DK> &tc, const T *q, const T *k,
                                            const float *g, float b, float eps, int l) {
    load_lane_vec<DK, T>(k, l, tc.kh);
    load_lane_vec<DK, T>(q, l, tc.qh);
    load_lane_vec<DK, float>(g, l, tc.alpha);
    l2norm_lane<DK>(tc.kh, eps);
    l2norm_lane<DK>(tc.qh, eps);
    exp_lane<DK>(tc.alpha);
    tc.beta = sigmoid_f(b);
    tc.kq = group_sum(lane_dot<DK>(tc.kh, tc.qh));
}

// The same coefficients rebuilt from a ReplaySSM record (no query needed).
template <int DK>
__device__ __forceinline__ void coeffs_from_record(TokenCoeffs<DK> &tc, const float *k_hat,
                                                   const float *g, float beta, int l) {
    load_lane_vec<DK, float>(k_hat, l, tc.kh);
    load_lane_vec<DK, float>(g, l, tc.alpha);
    exp_lane<DK>(tc.alpha);
    tc.beta = beta;
}

// ------------------------------------------------------------------ one row, one token

// Decay, delta rule and outer-product update of one state row (in place).
// Returns c = s'.q^ (the pre-update query dot, group-reduced) when WANT_OUT,
// and writes u to *u_out.
template <int DK, bool WANT_OUT>
__device__ __forceinline__ float row_update(LaneVec<DK> &s, const TokenCoeffs<DK> &tc, float v_i,
                                            float *u_out) {
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) s.v[i] = __fmul2_rn(s.v[i], tc.alpha.v[i]);
    const float r = group_sum(lane_dot<DK>(s, tc.kh));
    float c = 0.f;
    if constexpr (WANT_OUT) c = group_sum(lane_dot<DK>(s, tc.qh));
    const float u = __fmul_rn(tc.beta, __fsub_rn(v_i, r));
    const float2 u2 = make_float2(u, u);
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) s.v[i] = __ffma2_rn(u2, tc.kh.v[i], s.v[i]);
    *u_out = u;
    return c;
}

// One u record on one state row: s = s diag(exp g) + u k^ (element by
// element, s * alpha first, then one fused multiply-add).  No dot product:
// u already holds beta (v - s' . k^).
template <int DK>
__device__ __forceinline__ void commit_u_row(LaneVec<DK> &s, const float *k_hat, const float *g, float u, int l) {
    LaneVec<DK> kh, al;
    load_lane_vec<DK, float>(k_hat, l, kh);
    load_lane_vec<DK, float>(g, l, al);
    exp_lane<DK>(al);
    const float2 u2 = make_float2(u, u);
#pragma unroll
    for (int i = 0; i < DK / 16; ++i) s.v[i] = __ffma2_rn(u2, kh.v[i], __fmul2_rn(s.v[i], al.v[i]));
}

// o_i = scale * (S_t q^)_i computed as scale * (s'.q^ + u (k^.q^)).
__device__ __forceinline__ float row_output(float c, float u, float kq, float scale) {
    return __fmul_rn(scale, __fmaf_rn(u, kq, c));
}

// State row io: this lane's float4 slots of a row that starts at `row`.
template <int DK>
__device__ __forceinline__ void load_row(const float *row, int l, LaneVec<DK> &s) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) split4(ld_state(row + 4 * l + 32 * j), s.v[2 * j], s.v[2 * j + 1]);
}

template <int DK>
__device__ __forceinline__ void store_row(float *row, int l, const LaneVec<DK> &s) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j)
        st_state(row + 4 * l + 32 * j, make_float4(s.v[2 * j].x, s.v[2 * j].y, s.v[2 * j + 1].x, s.v[2 * j + 1].y));
}

}  // namespace kda
