// MegaKDA-style fused decode: ShortConv + KDA decode step + RMS norm and
// sigmoid output gate in one launch.
//
// "2.8x faster Kimi K3 inference on CANN", section 03 "MegaKDA": the input
// side (ShortConv) and the output-side compute are fused with the
// recurrence, so that no intermediate q, k, v or o round-trips through HBM
// and one launch replaces several small ones.  Readings taken here (the
// page names the fusion, not its formulas):
//
//   ShortConv   per channel c of q, k and v: y = silu(w0 x_{t-3} + w1 x_{t-2}
//               + w2 x_{t-1} + w3 x_t), the three earlier raw inputs taken
//               from the sequence's conv state, which is then shifted by one
//   KDA step    as in kda_decode, on the convolved q, k, v (fp32, never
//               rounded to the input dtype)
//   output      o' = o / sqrt(mean(o^2) + eps_o) * w_o * sigmoid(z)
//
// A cluster of two 4-warp CTAs owns one (sequence, head); the RMS norm needs
// the whole output row, so the two halves' sums of squares meet in
// distributed shared memory.  Each 8-lane group owns dv/32 rows; the state
// loads are issued before the convolution so that they are in flight while
// it runs.  The per-row arithmetic is kda_decode's (kda_rowmath.cuh),
// in the same order, so the state equals what kda_decode produces from the
// same convolved inputs held in fp32.
#include "kda.h"
#include "kda_bulk.cuh"
#include "kda_check.cuh"
#include "kda_internal.h"
#include "kda_rowmath.cuh"

namespace kda {

constexpr int kFusedWarps = 4;
constexpr int kFusedThreads = kFusedWarps * 32;
constexpr int kFusedGroups = kFusedWarps * kGroupsPerWarp;  // 16 row groups per CTA

// SiLU with the fast exponential and division (a few ulp)
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Arrive without ordering memory: execution order only.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of `p`'s counterpart in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t pa;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(pa) : "r"(a), "r"(rank));
    return pa;
}

// Writes `v` into CTA `rank`'s copy of `dst` and completes 4 bytes of the
// transaction count of that CTA's copy of `bar`.
__device__ __forceinline__ void st_async_peer(float *dst, uint64_t *bar, float v, uint32_t rank) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                     peer_addr(dst, rank)),
                 "r"(__float_as_uint(v)), "r"(peer_addr(bar, rank))
                 : "memory");
}

// A cluster of two CTAs owns one (sequence, head): CTA r of the pair holds
// value rows [r dv/2, (r+1) dv/2), the same 64-row grain per CTA as kda_decode.
// Both CTAs convolve all q and k channels (each needs the whole k^ and q^)
// and their own half of the v channels.  The RMS norm's sum of squares is
// exchanged through distributed shared memory: each CTA stores its partial
// sum into the other's `peer_part` with st.async, which completes the
// other's `xbar`.  A CTA writes its conv-state channels only after it has
// received the other's partial, which the other sent after its reads of the
// old conv state; and it exits only after that receipt, so neither CTA's
// shared memory is written after it has gone.
template <int DK, typename T, int R>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFusedThreads, 3)
    decode_fused_kernel(const DecodeFusedParams p) {
    constexpr int DV = 2 * kFusedGroups * R;
    constexpr int HV = DV / 2;          // value rows of this CTA
    constexpr int NC = 2 * DK + DV;     // conv channels of the head: q | k | v
    constexpr int NL = 2 * DK + HV;     // channels this CTA convolves
    constexpr int PER = (NL + kFusedThreads - 1) / kFusedThreads;
    __shared__ __align__(16) float xc[NL];  // q~ | k~ | this CTA's v~ rows
    __shared__ float red[kFusedWarps];
    __shared__ float peer_part;             // the other CTA's sum of o_i^2
    __shared__ __align__(8) uint64_t xbar;  // peer_part received

    const uint32_t rank = cluster_rank();
    const int64_t sh = blockIdx.x >> 1;  // (sequence, head) flattened = token index
    const int h = (int)(sh % p.H);
    const int n = (int)(sh / p.H);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int lrow0 = warp * kGroupsPerWarp + grp;  // local row, + rr * 16
    const int vbase = (int)rank * HV;               // first value row of this CTA

    T *orow = static_cast<T *>(p.out) + sh * DV + vbase;
    // checked build: the token's vectors and this CTA's rows of z and out
    // (both CTAs of the pair take the same decision, so neither waits alone)
    const int64_t tokens = (int64_t)p.batch * p.H;
    if (!in_bounds(sh * DK, DK, tokens * DK, p.err_flag) || !in_bounds(sh * DV, DV, tokens * DV, p.err_flag))
        return;
    const int slot = __ldg(p.slot_ids + n);
    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        // uniform over the pair: both CTAs read the same slot id
        for (int i = tid; i < HV; i += kFusedThreads) Elem<T>::store1(orow + i, 0.f);
        if (slot >= 0 && rank == 0 && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    float *S = p.pool + ((int64_t)slot * p.H + h) * (int64_t)DV * DK + (int64_t)vbase * DK;
    if (!in_bounds(((int64_t)slot * p.H + h) * DV * DK, (int64_t)DV * DK, p.num_slots * p.H * (int64_t)DV * DK,
                   p.err_flag) ||
        !in_bounds(((int64_t)slot * p.H + h) * 3 * NC, 3 * NC, p.num_slots * p.H * (int64_t)(3 * NC), p.err_flag))
        return;

    // Every global load of the step is issued here, before any of them is
    // used: the state rows, the token's gate, beta, output gate and norm
    // weight, and the conv inputs, so that one memory latency covers them all.
    LaneVec<DK> s[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) load_row<DK>(S + (int64_t)(lrow0 + rr * kFusedGroups) * DK, l, s[rr]);
    TokenCoeffs<DK> tc;
    load_lane_vec<DK, float>(p.g + sh * DK, l, tc.alpha);
    const float braw = Elem<T>::load1(static_cast<const T *>(p.b) + sh);
    const int orow_l = lrow0 + (l < R ? l : 0) * kFusedGroups;  // the row lane l < R writes
    const float zraw = Elem<T>::load1(static_cast<const T *>(p.z) + sh * DV + vbase + orow_l);
    const float nw = __ldg(p.norm_w + vbase + orow_l);

    // the exchange barrier, initialised before the other CTA can send to it
    // (the cluster wait below comes before this CTA's own send)
    if (tid == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&xbar, 4);
    }
    cluster_arrive_relaxed();

    T *cs = static_cast<T *>(p.conv_state) + ((int64_t)slot * p.H + h) * (3 * NC);
    const float4 *cw = reinterpret_cast<const float4 *>(p.conv_w) + (int64_t)h * NC;
    T cx[PER], c0[PER], c1[PER], c2[PER];
    float4 cwv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int cl = tid + j * kFusedThreads;  // local channel
        if (cl < NL) {
            const int c = cl < 2 * DK ? cl : cl + vbase;  // head channel
            const T *src = c < DK ? static_cast<const T *>(p.q) + sh * DK + c
                         : c < 2 * DK ? static_cast<const T *>(p.k) + sh * DK + (c - DK)
                                      : static_cast<const T *>(p.v) + sh * DV + (c - 2 * DK);
            cx[j] = *src;
            c0[j] = cs[c];
            c1[j] = cs[NC + c];
            c2[j] = cs[2 * NC + c];
            cwv[j] = __ldg(cw + c);
        }
    }

    // ShortConv of this CTA's channels; the raw inputs stay in registers
    // until both CTAs have read the old conv state
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int cl = tid + j * kFusedThreads;
        if (cl < NL) {
            float acc = __fmul_rn(cwv[j].x, Elem<T>::to_f(c0[j]));
            acc = __fmaf_rn(cwv[j].y, Elem<T>::to_f(c1[j]), acc);
            acc = __fmaf_rn(cwv[j].z, Elem<T>::to_f(c2[j]), acc);
            acc = __fmaf_rn(cwv[j].w, Elem<T>::to_f(cx[j]), acc);
            xc[cl] = silu_f(acc);
        }
    }
    __syncthreads();

    load_lane_vec_smem<DK>(xc + DK, l, tc.kh);
    load_lane_vec_smem<DK>(xc, l, tc.qh);
    l2norm_lane<DK>(tc.kh, p.eps);
    l2norm_lane<DK>(tc.qh, p.eps);
    exp_lane<DK>(tc.alpha);
    tc.beta = sigmoid_f(braw);
    tc.kq = group_sum(lane_dot<DK>(tc.kh, tc.qh));

    float o[R];
    float ss = 0.f;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int lrow = lrow0 + rr * kFusedGroups;
        float u;
        const float c = row_update<DK, true>(s[rr], tc, xc[2 * DK + lrow], &u);
        o[rr] = row_output(c, u, tc.kq, p.scale);
        ss = __fmaf_rn(o[rr], o[rr], ss);
    }
    // the updated state leaves first: nothing below waits for these stores
    // (the exchange below is st.async into an mbarrier, with no release)
#pragma unroll
    for (int rr = 0; rr < R; ++rr) store_row<DK>(S + (int64_t)(lrow0 + rr * kFusedGroups) * DK, l, s[rr]);

    // sum of o_i^2: the 4 groups of a warp, the 4 warps in order, then the
    // two CTAs (rank 0's half first, on both CTAs: the same bits)
    ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 8));
    ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 16));
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float mine = red[0];
#pragma unroll
    for (int w = 1; w < kFusedWarps; ++w) mine = __fadd_rn(mine, red[w]);
    cluster_wait();  // the other CTA's exchange barrier is initialised
    // every read of the old conv state has been consumed (the partial sum
    // depends on it) when the partial leaves
    if (tid == 0) st_async_peer(&peer_part, &xbar, mine, rank ^ 1u);
    // the other CTA's partial (thread 0 polls, bounded)
    const bool got = __syncthreads_and(tid == 0 ? mbar_wait(&xbar, 0) : true) != 0;
    if (got) {
        mbar_try_wait(&xbar, 0);
    } else if (tid == 0) {
        if (p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
        mbar_wait_drain(&xbar, 0);  // its write must land before this CTA's memory is released
    }
    const float theirs = got ? peer_part : 0.f;

    // shift the conv state: CTA 0 writes the q channels, CTA 1 the k
    // channels, each its own v channels
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int cl = tid + j * kFusedThreads;
        if (cl < NL && (cl >= 2 * DK || cl / DK == (int)rank)) {
            const int c = cl < 2 * DK ? cl : cl + vbase;
            cs[c] = c1[j];
            cs[NC + c] = c2[j];
            cs[2 * NC + c] = cx[j];
        }
    }

    // rank 0's half first on both CTAs: the same bits
    const float p0 = rank == 0 ? mine : theirs, p1 = rank == 0 ? theirs : mine;
    const float inv = rsqrtf(__fadd_rn(__fmul_rn(__fadd_rn(p0, p1), 1.0f / DV), p.eps_o));

    if (l < R) {
        // lane l of the group writes its row rr = l (R <= 8 lanes)
        float ol = o[0];
#pragma unroll
        for (int rr = 1; rr < R; ++rr) ol = l == rr ? o[rr] : ol;
        const float y = __fmul_rn(__fmul_rn(__fmul_rn(ol, inv), nw), sigmoid_f(zraw));
        Elem<T>::store1(orow + orow_l, y);
    }
}

template <int DK, typename T>
static cudaError_t launch_fused_t(const DecodeFusedParams &p, cudaStream_t st) {
    const int64_t grid = 2 * (int64_t)p.batch * p.H;  // a CTA pair per (sequence, head)
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    switch (p.dv) {
        case 128: decode_fused_kernel<DK, T, 4><<<(unsigned)grid, kFusedThreads, 0, st>>>(p); break;
        case 64: decode_fused_kernel<DK, T, 2><<<(unsigned)grid, kFusedThreads, 0, st>>>(p); break;
        case 32: decode_fused_kernel<DK, T, 1><<<(unsigned)grid, kFusedThreads, 0, st>>>(p); break;
        default: return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_fused(const DecodeFusedParams &p, int dk, int dtype, cudaStream_t st) {
    if (dtype == KDA_DT_BF16) {
        if (dk == 128) return launch_fused_t<128, __nv_bfloat16>(p, st);
        if (dk == 64) return launch_fused_t<64, __nv_bfloat16>(p, st);
        return launch_fused_t<32, __nv_bfloat16>(p, st);
    }
    if (dk == 128) return launch_fused_t<128, float>(p, st);
    if (dk == 64) return launch_fused_t<64, float>(p, st);
    return launch_fused_t<32, float>(p, st);
}

}  // namespace kda
