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
#include "kda_check.cuh"
#include "kda_internal.h"
#include "kda_rowmath.cuh"

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
    // checked build: this CTA's token vectors and its rows of v and out
    const int64_t tokens = (int64_t)p.batch * p.H;
    if (!in_bounds(sh * DK, DK, tokens * DK, p.err_flag) ||
        !in_bounds(sh * p.dv + blk * ROWS, ROWS, tokens * p.dv, p.err_flag))
        return;
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
    if (!in_bounds(((int64_t)slot * p.H + h) * p.dv * DK + (int64_t)blk * ROWS * DK, (int64_t)ROWS * DK,
                   p.num_slots * p.H * (int64_t)p.dv * DK, p.err_flag))
        return;

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

template <int DK, typename T, int R>
static cudaError_t launch_decode_r(const DecodeParams &p, cudaStream_t st) {
    const int nblk = p.dv / (kWarps * kGroupsPerWarp * R);
    const int64_t grid = (int64_t)p.batch * p.H * nblk;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_kernel<DK, T, R><<<(unsigned)grid, kWarps * 32, 0, st>>>(p);
    return cudaGetLastError();
}

template <int DK, typename T>
static cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t st) {
    // 16*R rows per CTA; every R gives the same bits.  Large batches at
    // dk = 128 take R = 4 (64 rows, 16 float4 state loads in flight per lane:
    // about 5% faster than R = 2 on the 256 x 32-head pool workload).  Small
    // batches, where the grid would not cover the GPU twice over, take fewer
    // rows per CTA so that more CTAs share the latency of one step.
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        sms = 1;
    const int64_t rows = (int64_t)p.batch * p.H * p.dv;  // state rows of the launch
    if (DK == 128 && p.dv % 64 == 0 && rows / 64 >= 2 * (int64_t)sms) return launch_decode_r<DK, T, 4>(p, st);
    if (rows / 32 >= 2 * (int64_t)sms) return launch_decode_r<DK, T, 2>(p, st);
    return launch_decode_r<DK, T, 1>(p, st);
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
