// Fused single-token KDA decode over the state pool.
//
// One launch performs, for every (sequence, value head): Q/K L2Norm, gate and
// beta processing, state decay, delta rule, outer-product update, output and
// in-place write-back of the final state ("Ascend day-0 support for Kimi K3",
// section "KDA Prefill and Decode dual path", decode kernel paragraph).
//
// Work decomposition: the page assigns one task per logical sequence x value
// head.  Here a CTA of 4 warps owns one (sequence, head, block of 16*R state
// rows); rows are independent, so a (sequence, head) is split over dv/(16R)
// CTAs to keep enough bytes in flight per SM.  Each 8-lane group owns R rows
// and keeps them in registers: every state byte is read once and written
// once with 128-bit streaming accesses, the two row dot products (S'k^ and
// S'q^) are 3-level shuffle reductions, and no __syncthreads is needed.
#include "kda.h"
#include "kda_internal.h"
#include "kda_bulk.cuh"
#include "kda_rowmath.cuh"

// State staging of the decode kernel: 0 = 128-bit loads straight into
// registers, 1 = one bulk (1-D TMA) copy of the CTA's rows into shared memory
// and one bulk copy back.
#ifndef KDA_DECODE_STAGING
#define KDA_DECODE_STAGING 0
#endif
#ifndef KDA_DECODE_BULK_ROWS
#define KDA_DECODE_BULK_ROWS 32
#endif

namespace kda {

constexpr int kWarps = 4;

template <int DK, typename T, int R>
__global__ void __launch_bounds__(kWarps * 32) decode_kernel(const DecodeParams p) {
    constexpr int ROWS = kWarps * kGroupsPerWarp * R;
    const int nblk = p.dv / ROWS;
    const int64_t item = blockIdx.x;
    const int blk = (int)(item % nblk);
    const int64_t sh = item / nblk;  // (sequence, head) flattened = token index
    const int h = (int)(sh % p.H);
    const int n = (int)(sh / p.H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int row0 = blk * ROWS + warp * kGroupsPerWarp + grp;  // + rr * 16

    const T *vrow = static_cast<const T *>(p.v) + sh * p.dv;
    T *orow = static_cast<T *>(p.out) + sh * p.dv;
    const int slot = __ldg(p.slot_ids + n);
    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        if (l == 0) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) Elem<T>::store1(orow + row0 + rr * kWarps * kGroupsPerWarp, 0.f);
        }
        if (slot >= 0 && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    float *S = p.pool + ((int64_t)slot * p.H + h) * (int64_t)p.dv * DK;

    // Issue the state loads first: they do not depend on the token.
    LaneVec<DK> s[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) load_row<DK>(S + (int64_t)(row0 + rr * 16) * DK, l, s[rr]);

    TokenCoeffs<DK> tc;
    const T *qp = static_cast<const T *>(p.q) + sh * DK;
    const T *kp = static_cast<const T *>(p.k) + sh * DK;
    const float bb = Elem<T>::load1(static_cast<const T *>(p.b) + sh);
    make_coeffs<DK, T>(tc, qp, kp, p.g + sh * DK, bb, p.eps, l);

#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int row = row0 + rr * 16;
        const float v_i = Elem<T>::load1(vrow + row);
        float u;
        const float c = row_update<DK, true>(s[rr], tc, v_i, &u);
        const float o = row_output(c, u, tc.kq, p.scale);
        if (l == 0) Elem<T>::store1(orow + row, o);
        store_row<DK>(S + (int64_t)row * DK, l, s[rr]);
    }
}

// Same decomposition and arithmetic, with the CTA's ROWS x dk block of state
// (contiguous in the pool) staged through shared memory by the bulk-copy
// engine: the load is in flight while the token coefficients are computed,
// and the in-flight bytes do not occupy registers.
template <int DK, typename T, int ROWS>
__global__ void __launch_bounds__(kWarps * 32) decode_bulk_kernel(const DecodeParams p) {
    constexpr uint32_t BYTES = ROWS * DK * 4;
    __shared__ __align__(128) float st[ROWS * DK];
    __shared__ __align__(8) uint64_t bar;
    const int nblk = p.dv / ROWS;
    const int64_t item = blockIdx.x;
    const int blk = (int)(item % nblk);
    const int64_t sh = item / nblk;
    const int h = (int)(sh % p.H);
    const int n = (int)(sh / p.H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int gid = warp * kGroupsPerWarp + grp;

    const T *vrow = static_cast<const T *>(p.v) + sh * p.dv + blk * ROWS;
    T *orow = static_cast<T *>(p.out) + sh * p.dv + blk * ROWS;
    const int slot = __ldg(p.slot_ids + n);
    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        for (int r = threadIdx.x; r < ROWS; r += kWarps * 32) Elem<T>::store1(orow + r, 0.f);
        if (slot >= 0 && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    float *S = p.pool + (((int64_t)slot * p.H + h) * (int64_t)p.dv + (int64_t)blk * ROWS) * DK;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar, BYTES);
        bulk_g2s(st, S, BYTES, &bar);
    }
    TokenCoeffs<DK> tc;
    const float bb = Elem<T>::load1(static_cast<const T *>(p.b) + sh);
    make_coeffs<DK, T>(tc, static_cast<const T *>(p.q) + sh * DK, static_cast<const T *>(p.k) + sh * DK,
                       p.g + sh * DK, bb, p.eps, l);
    __syncthreads();  // barrier initialised before anyone waits on it
    // the outcome is made CTA-uniform so that no thread skips a later barrier
    if (__syncthreads_and(mbar_wait(&bar, 0)) == 0) {
        if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
        mbar_wait(&bar, 0);  // bounded second chance for the copy in flight
        return;
    }
#pragma unroll
    for (int rr = 0; rr < ROWS / 16; ++rr) {
        const int row = rr * 16 + gid;
        LaneVec<DK> s;
        float *sp = st + row * DK;
        load_lane_vec_smem<DK>(sp, l, s);
        float u;
        const float c = row_update<DK, true>(s, tc, Elem<T>::load1(vrow + row), &u);
        if (l == 0) Elem<T>::store1(orow + row, row_output(c, u, tc.kq, p.scale));
        store_lane_vec<DK>(sp, l, s);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
        bulk_s2g(S, st, BYTES);
        bulk_commit();
        bulk_wait_read_all();  // shared memory must outlive the store's reads
    }
}

template <int DK, typename T>
static cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t st) {
    // 16*R rows per CTA; R = 2 keeps 8 float4 state loads in flight per lane
    // at dk = 128 and divides every supported dv.
#if KDA_DECODE_STAGING == 1
    constexpr int ROWS = KDA_DECODE_BULK_ROWS < 32 ? KDA_DECODE_BULK_ROWS : 32;
    const int rows = p.dv < KDA_DECODE_BULK_ROWS ? ROWS : KDA_DECODE_BULK_ROWS;
    const int64_t grid = (int64_t)p.batch * p.H * (p.dv / rows);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (rows == 32)
        decode_bulk_kernel<DK, T, 32><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
    else
        decode_bulk_kernel<DK, T, KDA_DECODE_BULK_ROWS><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
#else
    // dk = 128 with dv a multiple of 64 takes R = 4 (64 rows, 16 float4
    // state loads in flight per lane): about 5% faster on the 256 x 32-head
    // pool workload than R = 2, same bits.
    const bool wide = DK == 128 && p.dv % (kWarps * kGroupsPerWarp * 4) == 0;
    const int R = wide ? 4 : 2;
    const int nblk = p.dv / (kWarps * kGroupsPerWarp * R);
    const int64_t grid = (int64_t)p.batch * p.H * nblk;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (wide)
        decode_kernel<DK, T, (DK == 128 ? 4 : 2)><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
    else
        decode_kernel<DK, T, 2><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
#endif
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams &p, int dk, int dtype, cudaStream_t st) {
    if (dtype == KDA_DT_BF16) {
        if (dk == 128) return launch_decode_t<128, __nv_bfloat16>(p, st);
        if (dk == 64) return launch_decode_t<64, __nv_bfloat16>(p, st);
        return launch_decode_t<32, __nv_bfloat16>(p, st);
    }
    if (dk == 128) return launch_decode_t<128, float>(p, st);
    if (dk == 64) return launch_decode_t<64, float>(p, st);
    return launch_decode_t<32, float>(p, st);
}

}  // namespace kda
