// Tensor-core chunked prefill (tcgen05 + TMEM), dk = dv = 128, bf16 inputs.
//
// One CTA (4 warps) owns one (sequence, head) and walks its 64-token chunks
// in order ("Ascend day-0 support for Kimi K3", section "KDA Prefill and
// Decode dual path": 64-token chunks, with Q/K normalisation, gate
// accumulation and the chunk KDA organised as batched computation).  The
// chunk form (WY/UT, gamma = in-chunk cumulative gate per key channel):
//
//   A = strict-lower( beta_r sum_c k^_r k^_j e^{gamma_r - gamma_j} ),
//   P = lower( sum_c q^_r k^_j e^{gamma_r - gamma_j} ),  T = (I + A)^-1
//   W^T = (beta K~)^T T^T,  U'^T = (beta V)^T T^T            (WY factors)
//   U^T = U'^T - S W^T,  O^T = scale (S Q~^T + U^T P^T),
//   S <- S diag(e^{gamma_C}) + U^T K^                        (chunk step)
//
// The fp32 state S (dv x dk) never leaves tensor memory: it is the A operand
// of the MMAs that read it (TMEM lane = value row, column = key channel) and
// the accumulator of the rank-64 update.  All five products run on tcgen05
// in kind::tf32 with fp32 accumulation; B operands are staged in shared
// memory in the K-major 128-byte-swizzled layout.
//
// TMEM columns (512 allocated, one CTA per SM):
//   [0,128)   S                         [128,256) D1: S W^T | S Q~^T + U^T P^T
//   [256,320) U^T (Q~^T during prep)    [320,384) G = [K+;Q+] K-^T (A' | P)
//   [384,448) W^T                       [448,512) U'^T
//   During prep D1 holds the A operands (beta K~)^T and (beta V)^T.
//
// Decay factors: with ref = gamma at token 31 of the chunk, K+ = k^ e^{gamma-ref},
// Q+ = q^ e^{gamma-ref}, K- = k^ e^{ref-gamma}, so that K+ K-^T carries
// e^{gamma_r - gamma_j}.  A chunk whose gamma spans more than 80 (natural
// units) around ref on some channel would overflow these factors; such a
// chunk computes A and P with one exp per (r, j, c) on the CUDA cores.
#include <stdint.h>

#include "kda.h"
#include "kda_bulk.cuh"
#include "kda_internal.h"
#include "kda_rowmath.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace prefill_tc {

constexpr int C = 64;    // chunk length
constexpr int D = 128;   // dk = dv
constexpr int kThreads = 128;
constexpr int TM_S = 0, TM_D1 = 128, TM_UT = 256, TM_G = 320, TM_WT = 384, TM_UPT = 448;
constexpr int TM_BKT = TM_D1, TM_BVT = TM_D1 + 64, TM_QT = TM_UT;
constexpr uint32_t TM_COLS = 512;
constexpr float kSpanLimit = 80.f;

struct Smem {
    unsigned char bufA[128 * 128 * 4];  // [K+;Q+] then [W;Q~]   (128 rows x K 128)
    unsigned char bufKM[64 * 128 * 4];  // K-                     (64 rows x K 128)
    unsigned char bufT[64 * 64 * 4];    // T                      (64 rows x K 64)
    unsigned char bufP[64 * 64 * 4];    // P                      (64 rows x K 64)
    unsigned char bufKT[128 * 64 * 4];  // K^^T                   (128 rows x K 64)
    float As[C][C + 1];
    float Ts[C][C + 1];
    float Xs[3][16][17];
    float invk[C], invq[C], beta[C];
    float egc[D];
    uint64_t bar;
    uint32_t tmem_base;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

__device__ __forceinline__ void st_sw(unsigned char *tile, int rows, int row, int k, float x) {
    *reinterpret_cast<float *>(tile + tc::sw128_off(row, k, rows)) = x;
}

// Bounded wait on the CTA's MMA barrier; records a timeout.  The result is
// made uniform across the CTA so that every thread leaves the chunk loop
// together.
__device__ __forceinline__ bool wait_mma(Smem &sm, uint32_t &phase, int32_t *err_flag) {
    const bool mine = mbar_wait(&sm.bar, phase & 1);
    phase ^= 1;
    const bool ok = __syncthreads_and(mine) != 0;
    if (!ok && threadIdx.x == 0 && err_flag) atomicOr(err_flag, KDA_DEVERR_TIMEOUT);
    tc::fence_after_sync();
    return ok;
}

__device__ __forceinline__ void sync_for_mma() {
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t *plan = static_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    if (plan[n + 1] == 0) return;
    const int s = blockIdx.x, h = blockIdx.y, H = p.H;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t cs = p.cu_seqlens[s], ce = p.cu_seqlens[s + 1];
    const int slot = p.slot_ids[s];
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *bb = static_cast<const T *>(p.b);
    T *out = static_cast<T *>(p.out);
    const int64_t tok_stride = (int64_t)H * D;

    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        for (int64_t t = cs; t < ce; ++t) Elem<T>::store1(out + t * tok_stride + (int64_t)h * D + tid, 0.f);
        if (slot >= 0 && h == 0 && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }

    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, TM_COLS);
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_barrier_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem_base;
    uint32_t phase = 0;
    bool ok = true;
    float *Sg = p.pool + ((int64_t)slot * H + h) * (int64_t)D * D;

    // initial state: TMEM lane i = value row i
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 16) {
        float vv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) vv[j] = p.init_from_pool ? Sg[(int64_t)tid * D + c0 + j] : 0.f;
        tc::st16(tc::lane_addr(tm, warp, TM_S + c0), vv);
    }
    tc::wait_st();

    const int nchunks = (ce - cs + C - 1) / C;
    for (int ci = 0; ci < nchunks && ok; ++ci) {
        const int64_t t0 = (int64_t)cs + (int64_t)ci * C;
        const int L = (int)((int64_t)ce - t0 < C ? (int64_t)ce - t0 : C);
        const int64_t hoff = (int64_t)h * D;

        // ---- 1a. inverse norms (thread = token row) and beta
        {
            const int r = tid & 63;
            const bool isq = tid >= 64;
            float inv = 0.f;
            if (r < L) {
                const T *row = (isq ? q : k) + (t0 + r) * tok_stride + hoff;
                float ss = 0.f;
#pragma unroll 8
                for (int j = 0; j < D; j += 4) {
                    const float4 x = Elem<T>::load4(row + j);
                    ss = fmaf(x.x, x.x, ss);
                    ss = fmaf(x.y, x.y, ss);
                    ss = fmaf(x.z, x.z, ss);
                    ss = fmaf(x.w, x.w, ss);
                }
                inv = rsqrtf(ss + p.eps);
            }
            if (isq) {
                sm.invq[r] = inv;
            } else {
                sm.invk[r] = inv;
                sm.beta[r] = (r < L) ? sigmoid_f(Elem<T>::load1(bb + (t0 + r) * H + h)) : 0.f;
            }
        }
        __syncthreads();

        // ---- 1b. thread = key channel c: gate cumsum and the chunk operands
        const int c = tid;
        float gam[C];
        {
            float acc = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                if (r < L) acc += __ldg(p.g + (t0 + r) * tok_stride + hoff + c);
                gam[r] = acc;
            }
        }
        float gC = gam[0];
#pragma unroll
        for (int r = 1; r < C; ++r)
            if (r == L - 1) gC = gam[r];
        const float ref = gam[31];
        float span = 0.f;
#pragma unroll
        for (int r = 0; r < C; ++r) span = fmaxf(span, fabsf(gam[r] - ref));
        sm.egc[c] = expf(gC);
        const bool unsafe = __syncthreads_or(span > kSpanLimit) != 0;

        {
            const float eref = expf(ref);
            const float egcref = expf(gC - ref);
            float bkt[16], qt[16], bvt[16];
            float kt4[4];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const bool valid = r < L;
                const int64_t off = (t0 + r) * tok_stride + hoff + c;
                const float kx = valid ? Elem<T>::load1(k + off) * sm.invk[r] : 0.f;
                const float qx = valid ? Elem<T>::load1(q + off) * sm.invq[r] : 0.f;
                const float vx = valid ? Elem<T>::load1(v + off) : 0.f;
                float ktil, qtil, khat_end;
                if (!unsafe) {
                    const float E = __expf(gam[r] - ref);
                    const float Ei = __expf(ref - gam[r]);
                    const float kp = kx * E, qp = qx * E;
                    st_sw(sm.bufA, 128, r, c, kp);
                    st_sw(sm.bufA, 128, 64 + r, c, qp);
                    st_sw(sm.bufKM, 64, r, c, kx * Ei);
                    ktil = kp * eref;
                    qtil = qp * eref;
                    khat_end = kx * Ei * egcref;
                } else {
                    // plain [64][128] copies of k^, q^ and gamma for the exact path
                    reinterpret_cast<float *>(sm.bufA)[r * D + c] = kx;
                    reinterpret_cast<float *>(sm.bufA)[C * D + r * D + c] = qx;
                    reinterpret_cast<float *>(sm.bufKM)[r * D + c] = gam[r];
                    const float eg = expf(gam[r]);
                    ktil = kx * eg;
                    qtil = qx * eg;
                    khat_end = kx * expf(gC - gam[r]);
                }
                kt4[r & 3] = valid ? khat_end : 0.f;
                if ((r & 3) == 3)
                    *reinterpret_cast<float4 *>(sm.bufKT + tc::sw128_off(c, r - 3, 128)) =
                        make_float4(kt4[0], kt4[1], kt4[2], kt4[3]);
                bkt[r & 15] = sm.beta[r] * ktil;
                qt[r & 15] = qtil;
                bvt[r & 15] = sm.beta[r] * vx;  // thread c is also value row i = c
                if ((r & 15) == 15) {
                    tc::st16(tc::lane_addr(tm, warp, TM_BKT + (r - 15)), bkt);
                    tc::st16(tc::lane_addr(tm, warp, TM_QT + (r - 15)), qt);
                    tc::st16(tc::lane_addr(tm, warp, TM_BVT + (r - 15)), bvt);
                }
            }
        }
        tc::wait_st();
        sync_for_mma();

        // ---- 2. A and P
        if (!unsafe) {
            if (tid == 0) {
                constexpr uint32_t id = tc::idesc_tf32(128, 64);
                const uint32_t a0 = tc::smem_u32(sm.bufA), b0 = tc::smem_u32(sm.bufKM);
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_tf32_ss(tm + TM_G, tc::desc_tf32_kstep(a0, 128, ks), tc::desc_tf32_kstep(b0, 64, ks),
                                    id, ks > 0);
                tc::commit(&sm.bar);
            }
            ok = wait_mma(sm, phase, p.err_flag);
            if (!ok) break;
            // lanes 0..63: rows of A' ; lanes 64..127: rows of P
            const int r = tid & 63;
            float g16[16];
#pragma unroll
            for (int j0 = 0; j0 < C; j0 += 16) {
                tc::ld16(tc::lane_addr(tm, warp, TM_G + j0), g16);
                tc::wait_ld();
                if (tid < 64) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        sm.As[r][j] = (j < r) ? sm.beta[r] * g16[jj] : 0.f;
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4) {
                        const int j = j0 + jj;
                        *reinterpret_cast<float4 *>(sm.bufP + tc::sw128_off(r, j, 64)) =
                            make_float4(j <= r ? g16[jj] : 0.f, j + 1 <= r ? g16[jj + 1] : 0.f,
                                        j + 2 <= r ? g16[jj + 2] : 0.f, j + 3 <= r ? g16[jj + 3] : 0.f);
                    }
                }
            }
        } else {
            // exact path: one exp per (r, j, c)
            const float *kh = reinterpret_cast<const float *>(sm.bufA);
            const float *qh = kh + C * D;
            const float *gm = reinterpret_cast<const float *>(sm.bufKM);
            for (int idx = tid; idx < C * C; idx += kThreads) {
                const int r = idx / C, j = idx % C;
                float a = 0.f, pp = 0.f;
                if (j <= r) {
                    for (int cc = 0; cc < D; ++cc) {
                        const float m = kh[j * D + cc] * expf(gm[r * D + cc] - gm[j * D + cc]);
                        a = fmaf(kh[r * D + cc], m, a);
                        pp = fmaf(qh[r * D + cc], m, pp);
                    }
                }
                sm.As[r][j] = (j < r) ? sm.beta[r] * a : 0.f;
                *reinterpret_cast<float *>(sm.bufP + tc::sw128_off(r, j, 64)) = (j <= r) ? pp : 0.f;
            }
        }
        __syncthreads();

        // ---- 2c. T = (I + A)^-1: diagonal 16x16 blocks by forward
        // substitution, then off-diagonal blocks T_IJ = -T_II sum_K A_IK T_KJ
        for (int idx = tid; idx < C * (C + 1); idx += kThreads) (&sm.Ts[0][0])[idx] = 0.f;
        __syncthreads();
        if (tid < 64) {
            const int I = tid >> 4, j = tid & 15, o = 16 * I;
            float col[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    if (m < r && m >= j) acc = fmaf(-sm.As[o + r][o + m], col[m], acc);
                col[r] = (r >= j) ? acc : 0.f;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sm.Ts[o + r][o + j] = col[r];
        }
        __syncthreads();
        for (int dist = 1; dist < 4; ++dist) {
            const int nb = 4 - dist;
            for (int idx = tid; idx < nb * 256; idx += kThreads) {
                const int bi = idx >> 8, e = idx & 255, r = e >> 4, j = e & 15;
                const int I = bi + dist, J = bi;
                float x = 0.f;
                for (int K = J; K < I; ++K)
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        x = fmaf(sm.As[16 * I + r][16 * K + kk], sm.Ts[16 * K + kk][16 * J + j], x);
                sm.Xs[bi][r][j] = x;
            }
            __syncthreads();
            for (int idx = tid; idx < nb * 256; idx += kThreads) {
                const int bi = idx >> 8, e = idx & 255, r = e >> 4, j = e & 15;
                const int I = bi + dist, J = bi;
                float t = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    if (m <= r) t = fmaf(sm.Ts[16 * I + r][16 * I + m], sm.Xs[bi][m][j], t);
                sm.Ts[16 * I + r][16 * J + j] = -t;
            }
            __syncthreads();
        }
        for (int idx = tid; idx < C * C / 4; idx += kThreads) {
            const int r = idx / (C / 4), j = (idx % (C / 4)) * 4;
            *reinterpret_cast<float4 *>(sm.bufT + tc::sw128_off(r, j, 64)) =
                make_float4(sm.Ts[r][j], sm.Ts[r][j + 1], sm.Ts[r][j + 2], sm.Ts[r][j + 3]);
        }
        sync_for_mma();

        // ---- 3. W^T = (beta K~)^T T^T and U'^T = (beta V)^T T^T
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
            const uint32_t b0 = tc::smem_u32(sm.bufT);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const uint64_t bd = tc::desc_tf32_kstep(b0, 64, ks);
                tc::mma_tf32_ts(tm + TM_WT, tm + TM_BKT + 8 * ks, bd, id, ks > 0);
                tc::mma_tf32_ts(tm + TM_UPT, tm + TM_BVT + 8 * ks, bd, id, ks > 0);
            }
            tc::commit(&sm.bar);
        }
        ok = wait_mma(sm, phase, p.err_flag);
        if (!ok) break;
        // [W; Q~] into bufA as the B operand of the chunk step (thread = channel)
        {
            float w16[16];
#pragma unroll
            for (int r0 = 0; r0 < C; r0 += 16) {
                tc::ld16(tc::lane_addr(tm, warp, TM_WT + r0), w16);
                tc::wait_ld();
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) st_sw(sm.bufA, 128, r0 + rr, c, w16[rr]);
                tc::ld16(tc::lane_addr(tm, warp, TM_QT + r0), w16);
                tc::wait_ld();
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) st_sw(sm.bufA, 128, 64 + r0 + rr, c, w16[rr]);
            }
        }
        sync_for_mma();

        // ---- 4. D1 = S [W; Q~]^T
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 128);
            const uint32_t b0 = tc::smem_u32(sm.bufA);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_tf32_ts(tm + TM_D1, tm + TM_S + 8 * ks, tc::desc_tf32_kstep(b0, 128, ks), id, ks > 0);
            tc::commit(&sm.bar);
        }
        ok = wait_mma(sm, phase, p.err_flag);
        if (!ok) break;
        // U^T = U'^T - S W^T (thread = value row i); S <- S diag(e^{gamma_C})
        {
            float a16[16], b16[16];
#pragma unroll
            for (int r0 = 0; r0 < C; r0 += 16) {
                tc::ld16(tc::lane_addr(tm, warp, TM_UPT + r0), a16);
                tc::ld16(tc::lane_addr(tm, warp, TM_D1 + r0), b16);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) a16[j] -= b16[j];
                tc::st16(tc::lane_addr(tm, warp, TM_UT + r0), a16);
            }
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                tc::ld16(tc::lane_addr(tm, warp, TM_S + c0), a16);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) a16[j] *= sm.egc[c0 + j];
                tc::st16(tc::lane_addr(tm, warp, TM_S + c0), a16);
            }
            tc::wait_st();
        }
        sync_for_mma();

        // ---- 5. O^T += U^T P^T ; S += U^T K^
        if (tid == 0) {
            constexpr uint32_t id64 = tc::idesc_tf32(128, 64);
            constexpr uint32_t id128 = tc::idesc_tf32(128, 128);
            const uint32_t bp = tc::smem_u32(sm.bufP), bk = tc::smem_u32(sm.bufKT);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                tc::mma_tf32_ts(tm + TM_D1 + 64, tm + TM_UT + 8 * ks, tc::desc_tf32_kstep(bp, 64, ks), id64, 1);
                tc::mma_tf32_ts(tm + TM_S, tm + TM_UT + 8 * ks, tc::desc_tf32_kstep(bk, 128, ks), id128, 1);
            }
            tc::commit(&sm.bar);
        }
        ok = wait_mma(sm, phase, p.err_flag);
        if (!ok) break;
        {
            float o16[16];
            const float scale = p.scale;
#pragma unroll
            for (int r0 = 0; r0 < C; r0 += 16) {
                tc::ld16(tc::lane_addr(tm, warp, TM_D1 + 64 + r0), o16);
                tc::wait_ld();
#pragma unroll
                for (int rr = 0; rr < 16; ++rr)
                    if (r0 + rr < L)
                        Elem<T>::store1(out + (t0 + r0 + rr) * tok_stride + hoff + tid, scale * o16[rr]);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    if (ok) {
        float s16[16];
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            tc::ld16(tc::lane_addr(tm, warp, TM_S + c0), s16);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(Sg + (int64_t)tid * D + c0 + j) =
                    make_float4(s16[j], s16[j + 1], s16[j + 2], s16[j + 3]);
        }
    } else {
        // bounded: let the MMA group whose wait gave up finish before the
        // tensor memory is released (its phase is the one before `phase`)
        mbar_wait(&sm.bar, (phase ^ 1) & 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TM_COLS);
}

}  // namespace prefill_tc

#ifndef KDA_PREFILL_TC
#define KDA_PREFILL_TC 0
#endif

bool prefill_tc_supported(int dk, int dv, int dtype) {
    return KDA_PREFILL_TC && dtype == KDA_DT_BF16 && dk == 128 && dv == 128;
}

cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t st) {
    using namespace prefill_tc;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.num_seqs, (unsigned)p.H);
    prefill_tc_kernel<__nv_bfloat16><<<grid, kThreads, kSmemBytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
