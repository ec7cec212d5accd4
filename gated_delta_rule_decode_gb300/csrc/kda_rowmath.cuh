// Row-parallel KDA token math shared by the decode, verify and replay kernels.
//
// Rows of the V x K state (value channels) are independent for one token:
// row i needs only its own dk entries s_i, the normalised key k^, the
// normalised query q^, alpha = exp(g), beta and v_i.  Each row is owned by an
// 8-lane group of a warp; lane l of the group holds the dk/8 entries at key
// channels {4l + 32j + e : j < dk/32, e < 4}, so that one float4 access per
// j by the group covers 128 contiguous bytes of the row.
//
// All arithmetic uses explicit round-to-nearest intrinsics in one fixed order,
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

// ------------------------------------------------------------------ per-token coefficients

template <int DK>
struct TokenCoeffs {
    static constexpr int E = DK / kLanesPerRow;  // entries per lane
    float kh[E];      // normalised key at this lane's channels
    float qh[E];      // normalised query at this lane's channels
    float alpha[E];   // exp(g) at this lane's channels
    float beta;       // sigmoid(b)
    float kq;         // k^ . q^ over all dk channels
};

// Channel index of entry e of lane l.
template <int DK>
__device__ __forceinline__ int lane_channel(int l, int e) {
    return 4 * l + 32 * (e >> 2) + (e & 3);
}

// Loads this lane's entries of a dk-vector of element type T.
template <int DK, typename T>
__device__ __forceinline__ void load_lane_vec(const T *p, int l, float (&x)[DK / kLanesPerRow]) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) {
        float4 t = Elem<T>::load4(p + 4 * l + 32 * j);
        x[4 * j + 0] = t.x;
        x[4 * j + 1] = t.y;
        x[4 * j + 2] = t.z;
        x[4 * j + 3] = t.w;
    }
}

// x^ = x * rsqrt(sum x^2 + eps) over the group's dk entries.
template <int DK>
__device__ __forceinline__ void l2norm_lane(float (&x)[DK / kLanesPerRow], float eps) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) ss = __fmaf_rn(x[e], x[e], ss);
    ss = group_sum(ss);
    const float inv = rsqrtf(__fadd_rn(ss, eps));
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) x[e] = __fmul_rn(x[e], inv);
}

__device__ __forceinline__ float sigmoid_f(float b) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-b)));
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
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) tc.alpha[e] = expf(tc.alpha[e]);
    tc.beta = sigmoid_f(b);
    float kq = 0.f;
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) kq = __fmaf_rn(tc.kh[e], tc.qh[e], kq);
    tc.kq = group_sum(kq);
}

// The same coefficients rebuilt from a ReplaySSM record (no query needed).
template <int DK>
__device__ __forceinline__ void coeffs_from_record(TokenCoeffs<DK> &tc, const float *k_hat,
                                                   const float *g, float beta, int l) {
    load_lane_vec<DK, float>(k_hat, l, tc.kh);
    load_lane_vec<DK, float>(g, l, tc.alpha);
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) tc.alpha[e] = expf(tc.alpha[e]);
    tc.beta = beta;
}

// ------------------------------------------------------------------ one row, one token

// Partial dot product of the lane's entries in a fixed association order:
// a 4-term FMA chain per float4 slot, then the slots summed pairwise.
template <int DK>
__device__ __forceinline__ float lane_dot(const float (&s)[DK / kLanesPerRow],
                                          const float (&w)[DK / kLanesPerRow]) {
    constexpr int J = DK / 32;
    float p[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        float a = __fmul_rn(s[4 * j], w[4 * j]);
        a = __fmaf_rn(s[4 * j + 1], w[4 * j + 1], a);
        a = __fmaf_rn(s[4 * j + 2], w[4 * j + 2], a);
        a = __fmaf_rn(s[4 * j + 3], w[4 * j + 3], a);
        p[j] = a;
    }
    if constexpr (J == 1) {
        return p[0];
    } else if constexpr (J == 2) {
        return __fadd_rn(p[0], p[1]);
    } else {
        return __fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3]));
    }
}

// Decay, delta rule and outer-product update of one state row (in place).
// Returns c = s'.q^ (the pre-update query dot, group-reduced) when WANT_OUT,
// and writes u to *u_out.
template <int DK, bool WANT_OUT>
__device__ __forceinline__ float row_update(float (&s)[DK / kLanesPerRow], const TokenCoeffs<DK> &tc,
                                            float v_i, float *u_out) {
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) s[e] = __fmul_rn(s[e], tc.alpha[e]);
    const float r = group_sum(lane_dot<DK>(s, tc.kh));
    float c = 0.f;
    if constexpr (WANT_OUT) c = group_sum(lane_dot<DK>(s, tc.qh));
    const float u = __fmul_rn(tc.beta, __fsub_rn(v_i, r));
#pragma unroll
    for (int e = 0; e < DK / kLanesPerRow; ++e) s[e] = __fmaf_rn(u, tc.kh[e], s[e]);
    *u_out = u;
    return c;
}

// o_i = scale * (S_t q^)_i computed as scale * (s'.q^ + u (k^.q^)).
__device__ __forceinline__ float row_output(float c, float u, float kq, float scale) {
    return __fmul_rn(scale, __fmaf_rn(u, kq, c));
}

// State row io: this lane's float4 slots of a row that starts at `row`.
template <int DK>
__device__ __forceinline__ void load_row(const float *row, int l, float (&s)[DK / kLanesPerRow]) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) {
        float4 t = ld_state(row + 4 * l + 32 * j);
        s[4 * j + 0] = t.x;
        s[4 * j + 1] = t.y;
        s[4 * j + 2] = t.z;
        s[4 * j + 3] = t.w;
    }
}

template <int DK>
__device__ __forceinline__ void store_row(float *row, int l, const float (&s)[DK / kLanesPerRow]) {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j)
        st_state(row + 4 * l + 32 * j, make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]));
}

}  // namespace kda
