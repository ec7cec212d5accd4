// ReplaySSM verify for the benchmarked shape (bf16 inputs, dk = dv = 128,
// draft windows of up to 8 tokens), with the state product on tcgen05.
//
// "2.8x faster Kimi K3 inference on CANN", section 04 "ReplaySSM": verify
// keeps only the per-token update records and the outputs of every draft
// token; it never writes the pool.
//
// The window is evaluated in chunk form over the committed state S0 (the
// algebra is written out in kda_window.cuh), in two launches:
//
//   window_kernel  one 64-thread CTA per (sequence, head), one draft token
//                  per 8-lane group.  Writes the records (the key and beta
//                  with the decode kernel's routine, so they replay bit for
//                  bit) and a scratch record: the B tile [K~; Q~] already in
//                  the 128-byte-swizzled K-major image the MMA reads, beta,
//                  p_jj, and the rows K^_m = k^_m / E_m.
//   state_kernel   one 128-thread CTA per (sequence, head), three per SM.
//                  Copies S0 (TMA, four 32-channel boxes) and the scratch
//                  record (one bulk copy), forms the window products
//                  a_jm = K~_j . K^_m and p_jm = Q~_j . K^_m while the state
//                  lands, runs D[i][j] = S0[i] . K~_j, D[i][8 + j] = S0[i] . Q~_j
//                  as one M = 128, N = 16, K = 128 kind::tf32 product into
//                  TMEM, and the per-row triangular recurrence.
//
// Only the state kernel holds a 64 KB tile, and only while its copy is in
// flight and its product runs, so three of them share an SM and keep enough
// state bytes in flight for HBM; the latency-bound token work runs in the
// small window CTAs.  The scratch record (about 12.6 KB per (sequence, head))
// stays in L2: the state is streamed with an evict-first policy, and each
// record's lines are discarded once read, so they are never written back.
// The state kernel is a programmatic dependent launch: its state copy is
// issued before it waits for the window kernel.
//
// The factored products need 1 / E_m: a window whose decay product falls
// below 1e-30 in some channel takes the running products instead (the window
// kernel forms a_jm and p_jm itself and flags the record).
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include "kda.h"
#include "kda_bulk.cuh"
#include "kda_check.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"
#include "kda_window.cuh"

namespace kda {
namespace verify_tc {

constexpr int DK = 128;
constexpr int kDraft = 8;
constexpr uint32_t kTmemCols = 32;
constexpr uint32_t kStateBytes = 128 * DK * 4;
constexpr uint32_t kTileBytes = 4 * 16 * 128;  // [K~ rows 0..7; Q~ rows 8..15], four channel atoms
constexpr float kTinyDecay = 1e-30f;            // below this, 1 / E_m is not taken
// scratch record per (sequence, head): [B tile | A | P | beta | flag | K^ rows],
// padded to whole 128-byte lines; the first kCopyBytes go to shared memory
// in one bulk copy
constexpr uint32_t kOffA = kTileBytes, kOffP = kOffA + kDraft * kDraft * 4, kOffBeta = kOffP + kDraft * kDraft * 4;
constexpr uint32_t kOffFlag = kOffBeta + kDraft * 4, kCopyBytes = kOffFlag + 16, kOffKhat = kCopyBytes;
constexpr uint32_t kRecBytes = (kOffKhat + kDraft * DK * 4 + 127) / 128 * 128;
static_assert(kCopyBytes % 16 == 0 && kRecBytes % 16 == 0, "bulk copy granularity");
constexpr int kWinThreads = 64;  // one (sequence, head) per CTA, one token per 8-lane group
constexpr int kStateThreads = 128;  // one thread per state row

struct WinSmem {
    float kh[kDraft][DK];
    float qh[kDraft][DK];
    float al[kDraft][DK];
};

struct StateSmem {
    unsigned char st[4][128 * 128];  // S0: 4 channel atoms of [128 rows][128 B], 128B-swizzled
    unsigned char kq[4][16 * 128];   // the scratch record lands from here on
    float A[kDraft][kDraft];
    float P[kDraft][kDraft];
    float beta[kDraft];
    int flag[4];
    uint64_t rbar;  // record landed
    uint64_t sbar;  // state landed
    uint64_t mbar;  // product done
    uint32_t tmem_base;
};
static_assert(offsetof(StateSmem, A) - offsetof(StateSmem, kq) == kOffA, "record layout");
static_assert(offsetof(StateSmem, flag) - offsetof(StateSmem, kq) == kOffFlag, "record layout");
static_assert(offsetof(StateSmem, rbar) - offsetof(StateSmem, kq) >= kCopyBytes, "record layout");
constexpr size_t kStateSmemBytes = sizeof(StateSmem) + 1024;  // + alignment of the swizzled tiles

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_3d_ef(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar,
                                               uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_ef(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// Drops one 128-byte line from L2 without writing it back (its contents
// become undefined).
__device__ __forceinline__ void discard_l2(const void *p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// This lane's entries as streaming stores (records are not read again here).
template <int N>
__device__ __forceinline__ void store_lane_vec_cs(float *p, int l, const LaneVec<N> &x) {
#pragma unroll
    for (int j = 0; j < N / 32; ++j)
        __stcs(reinterpret_cast<float4 *>(p + 4 * l + 32 * j),
               make_float4(x.v[2 * j].x, x.v[2 * j].y, x.v[2 * j + 1].x, x.v[2 * j + 1].y));
}

// Row `row` of the 16-row swizzled B tile: this lane's four float4 slots
// (channels 4l + 32a .. 4l + 32a + 3 sit in channel atom a, 16-byte chunk
// l ^ (row & 7)).
__device__ __forceinline__ void store_b_row(unsigned char *tile, int row, int l, const LaneVec<DK> &x) {
#pragma unroll
    for (int a = 0; a < DK / 32; ++a)
        *reinterpret_cast<float4 *>(tile + a * 16 * 128 + row * 128 + ((l ^ (row & 7)) << 4)) =
            make_float4(x.v[2 * a].x, x.v[2 * a].y, x.v[2 * a + 1].x, x.v[2 * a + 1].y);
}

template <typename T>
__global__ void __launch_bounds__(kWinThreads) window_kernel(const VerifyParams p, unsigned char *ws) {
    __shared__ __align__(16) WinSmem sm;
    const int tid = threadIdx.x;
    const int64_t sh = blockIdx.x;  // (sequence, head)
    const int h = (int)(sh % p.H), n = (int)(sh / p.H);
    const int grp = tid >> 3, l = tid & 7;  // this group's draft token, lane in the group
    const int D = p.D;
    // the state kernel may start now: it waits for this grid's completion
    // before it reads any scratch record
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // checked build: this (sequence, head)'s scratch record and its window's
    // token-heads
    const int64_t items = (int64_t)p.batch * p.H;
    if (!in_bounds(sh * kRecBytes, kRecBytes, items * kRecBytes, p.err_flag) ||
        !in_bounds((int64_t)n * D * p.H + h, (int64_t)(D - 1) * p.H + 1, items * D, p.err_flag))
        return;
    unsigned char *rec = ws + sh * kRecBytes;
    float *Aw = reinterpret_cast<float *>(rec + kOffA);
    float *Pw = reinterpret_cast<float *>(rec + kOffP);
    float *Bw = reinterpret_cast<float *>(rec + kOffBeta);
    float *Kw = reinterpret_cast<float *>(rec + kOffKhat);

    // value records: bit copies of the D rows
    {
        constexpr int E = 16 / sizeof(T);
        const int per_row = p.dv / E;
        uint4 x[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = tid + kWinThreads * u;
            if (idx < D * per_row) {
                const int j = idx / per_row, c = (idx - j * per_row) * E;
                x[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const T *>(p.v) +
                                                             (((int64_t)n * D + j) * p.H + h) * p.dv + c));
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = tid + kWinThreads * u;
            if (idx < D * per_row && p.rec_v) {
                const int j = idx / per_row, c = (idx - j * per_row) * E;
                __stcs(reinterpret_cast<uint4 *>(static_cast<T *>(p.rec_v) + (((int64_t)n * D + j) * p.H + h) * p.dv + c),
                       x[u]);
            }
        }
    }
    // token grp's key, query, gate and beta: every load is issued before any
    // is used
    const int j = grp;
    const bool act = j < D;
    const int64_t tk = ((int64_t)n * D + (act ? j : 0)) * p.H + h;
    uint2 kr[DK / 32], qr[DK / 32];
    float4 gr[DK / 32];
    {
        const T *kp = static_cast<const T *>(p.k) + tk * DK + 4 * l;
        const T *qp = static_cast<const T *>(p.q) + tk * DK + 4 * l;
        const float *gp = p.g + tk * DK + 4 * l;
#pragma unroll
        for (int s = 0; s < DK / 32; ++s) {
            kr[s] = __ldg(reinterpret_cast<const uint2 *>(kp + 32 * s));
            qr[s] = __ldg(reinterpret_cast<const uint2 *>(qp + 32 * s));
            gr[s] = __ldg(reinterpret_cast<const float4 *>(gp + 32 * s));
        }
    }
    const T br = static_cast<const T *>(p.b)[tk];
    // bf16 pairs widened exactly as Elem<bf16>::load4 does
    auto widen = [](const uint2 (&raw)[DK / 32], LaneVec<DK> &x) {
#pragma unroll
        for (int s = 0; s < DK / 32; ++s)
            split4(make_float4(__uint_as_float(raw[s].x << 16), __uint_as_float(raw[s].x & 0xffff0000u),
                               __uint_as_float(raw[s].y << 16), __uint_as_float(raw[s].y & 0xffff0000u)),
                   x.v[2 * s], x.v[2 * s + 1]);
    };
    // k^ and beta with the decode routine's arithmetic (records), q^, and
    // alpha = exp(g) (the gate record is the raw g)
    {
        LaneVec<DK> x;
        widen(kr, x);
        l2norm_lane<DK>(x, p.eps);
        if (act) {
            store_lane_vec<DK>(&sm.kh[j][0], l, x);
            store_lane_vec_cs<DK>(p.rec_k_hat + tk * DK, l, x);
            if (l == 0) {
                const float bt = sigmoid_f(Elem<T>::to_f(br));
                Bw[j] = bt;
                if (p.rec_beta) __stcs(p.rec_beta + tk, bt);
            }
        }
        widen(qr, x);
        l2norm_lane<DK>(x, p.eps);
        if (act) store_lane_vec<DK>(&sm.qh[j][0], l, x);
#pragma unroll
        for (int s = 0; s < DK / 32; ++s) split4(gr[s], x.v[2 * s], x.v[2 * s + 1]);
        if (act) {
            store_lane_vec_cs<DK>(p.rec_g + tk * DK, l, x);
            exp_lane<DK>(x);
            store_lane_vec<DK>(&sm.al[j][0], l, x);
        }
    }
    __syncthreads();
    // E_j = prod_{l<=j} alpha_l in token order; K~_j, Q~_j, p_jj and
    // K^_j = k^_j / E_j
    bool tiny = false;
    {
        const int jj = act ? j : 0;
        LaneVec<DK> w, kj, qj, a;
        set_ones<DK>(w);
        for (int li = 0; li < D; ++li)  // warp-uniform trip count
            if (li <= jj) {
                load_lane_vec_smem<DK>(&sm.al[li][0], l, a);
                mul_lane<DK>(w, a);
            }
        load_lane_vec_smem<DK>(&sm.kh[jj][0], l, kj);
        load_lane_vec_smem<DK>(&sm.qh[jj][0], l, qj);
        const float pjj = group_sum(lane_dot<DK>(kj, qj));
        LaneVec<DK> kb;
#pragma unroll
        for (int i = 0; i < DK / 16; ++i) {
            kb.v[i] = make_float2(__fdiv_rn(kj.v[i].x, w.v[i].x), __fdiv_rn(kj.v[i].y, w.v[i].y));
            tiny |= act && (w.v[i].x < kTinyDecay || w.v[i].y < kTinyDecay);
        }
        mul_lane<DK>(kj, w);
        mul_lane<DK>(qj, w);
        if (act) {
            store_b_row(rec, j, l, kj);
            store_b_row(rec, kDraft + j, l, qj);
            store_lane_vec<DK>(Kw + j * DK, l, kb);
            if (l == 0) Pw[j * kDraft + j] = pjj;
        }
    }
    // a decay product at the bottom of the fp32 range (or below it): the
    // window products are formed here with running products instead
    const bool slow = __syncthreads_or(tiny) != 0;
    if (slow) {
        const int npairs = D * (D - 1) / 2;
        constexpr int groups = kWinThreads / 8;
        auto none = [](float *, float *, int, int, const LaneVec<DK> &, const LaneVec<DK> &) {};
        for (int base = 0; base < npairs; base += groups) {
            if (base + (tid >> 5) * kGroupsPerWarp >= npairs) break;  // warp-uniform
            window_pair<DK>(D + base + j, base + j < npairs, D, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0],
                            nullptr, nullptr, Aw, Pw, kDraft, none);
        }
    }
    if (tid == 0) *reinterpret_cast<int *>(rec + kOffFlag) = slow ? 1 : 0;
}

template <typename T>
__global__ void __launch_bounds__(kStateThreads, 3) state_kernel(const VerifyParams p,
                                                               const __grid_constant__ CUtensorMap smap,
                                                               const unsigned char *ws) {
    extern __shared__ unsigned char smem_raw[];
    StateSmem &sm = *reinterpret_cast<StateSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int sh = blockIdx.x;
    const int h = sh % p.H, n = sh / p.H;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int D = p.D;
    // checked build: the scratch record and the window's token-heads
    const int64_t items = (int64_t)p.batch * p.H;
    if (!in_bounds((int64_t)sh * kRecBytes, kRecBytes, items * kRecBytes, p.err_flag) ||
        !in_bounds((int64_t)n * D * p.H + h, (int64_t)(D - 1) * p.H + 1, items * D, p.err_flag))
        return;

    const int slot = __ldg(p.slot_ids + n);
    const bool valid = slot >= 0 && (int64_t)slot < p.num_slots;
    if (slot >= 0 && !valid && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);

    const int grp = (tid & 31) >> 3, l = tid & 7, gid = warp * kGroupsPerWarp + grp;
    const unsigned char *rec = ws + (size_t)sh * kRecBytes;
    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid == 0) {
        mbar_init(&sm.rbar, 1);
        mbar_init(&sm.sbar, 1);
        mbar_init(&sm.mbar, 1);
        fence_barrier_init();
        if (valid) {
            const uint64_t pol = evict_first_policy();
            mbar_arrive_expect_tx(&sm.sbar, kStateBytes);
            const int z = slot * p.H + h;
#pragma unroll
            for (int a = 0; a < 4; ++a) tma_load_3d_ef(sm.st[a], &smap, 32 * a, 0, z, &sm.sbar, pol);
        }
    }
    // S0 does not depend on the window kernel, its scratch record does: this
    // waits for that grid to complete (at once without a programmatic launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0 && valid) {
        mbar_arrive_expect_tx(&sm.rbar, kCopyBytes);
        bulk_g2s_ef(&sm.kq[0][0], rec, kCopyBytes, &sm.rbar, evict_first_policy());
    }
    // pair tasks (m < j) of this group, two rounds of 16: K^_m rows now
    constexpr int kGroups = kStateThreads / 8;
    const int npairs = D * (D - 1) / 2;
    int pm[2], pj[2];
    LaneVec<DK> kb[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        int t = r * kGroups + gid, m = 0;
        const bool act = t < npairs;
        if (act)
            while (t >= D - 1 - m) {  // pairs (m, m+1 .. D-1) come in runs of D - 1 - m
                t -= D - 1 - m;
                ++m;
            }
        pm[r] = act ? m : -1;
        pj[r] = act ? m + 1 + t : 0;
        if (act && valid) {
            const float *src = reinterpret_cast<const float *>(rec + kOffKhat) + m * DK + 4 * l;
#pragma unroll
            for (int s2 = 0; s2 < DK / 32; ++s2)
                split4(__ldg(reinterpret_cast<const float4 *>(src + 32 * s2)), kb[r].v[2 * s2], kb[r].v[2 * s2 + 1]);
        } else {
            set_ones<DK>(kb[r]);
        }
    }
    // this thread's state row: its value entries
    float vr[kDraft];
    {
        const T *vb = static_cast<const T *>(p.v) + ((int64_t)n * D * p.H + h) * p.dv + tid;
#pragma unroll
        for (int j = 0; j < kDraft; ++j) vr[j] = j < D ? Elem<T>::load1(vb + (int64_t)j * p.H * p.dv) : 0.f;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem_base;

    bool ok = true;
    bool issued = false;
    float o[kDraft], uu[kDraft];
#pragma unroll
    for (int j = 0; j < kDraft; ++j) o[j] = uu[j] = 0.f;
    if (valid) {
        ok = __syncthreads_and(mbar_wait(&sm.rbar, 0)) != 0;
        if (ok && sm.flag[0] == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r * kGroups + warp * kGroupsPerWarp >= npairs) break;  // warp-uniform
                const int j = pm[r] >= 0 ? pj[r] : 0;
                LaneVec<DK> kt, qt;
#pragma unroll
                for (int s2 = 0; s2 < DK / 32; ++s2) {
                    const int off = s2 * 16 * 128 + ((l ^ (j & 7)) << 4);
                    split4(*reinterpret_cast<const float4 *>(&sm.kq[0][0] + off + j * 128), kt.v[2 * s2],
                           kt.v[2 * s2 + 1]);
                    split4(*reinterpret_cast<const float4 *>(&sm.kq[0][0] + off + (kDraft + j) * 128), qt.v[2 * s2],
                           qt.v[2 * s2 + 1]);
                }
                const float av = group_sum(lane_dot<DK>(kt, kb[r]));
                const float pv = group_sum(lane_dot<DK>(qt, kb[r]));
                if (pm[r] >= 0 && l == 0) {
                    sm.A[j][pm[r]] = av;
                    sm.P[j][pm[r]] = pv;
                }
            }
        }
        if (ok) ok = __syncthreads_and(mbar_wait(&sm.sbar, 0)) != 0;
        // every read of the scratch record is complete: drop its lines from L2
        // without writing them back
        if (ok && warp == 1)
            for (int i = tid & 31; i < (int)(kRecBytes / 128); i += 32) discard_l2(rec + 128 * i);
        if (ok) {
            if (tid == 0) {
                constexpr uint32_t id = tc::idesc_tf32(128, 16);
                const uint32_t a0 = tc::smem_u32(sm.st), b0 = tc::smem_u32(sm.kq);
#pragma unroll
                for (int ks = 0; ks < DK / 8; ++ks)
                    tc::mma_tf32_ss(tm, tc::desc_tf32_kstep(a0, 128, ks), tc::desc_tf32_kstep(b0, 16, ks), id,
                                    ks > 0);
                tc::commit(&sm.mbar);
            }
            issued = true;
            ok = __syncthreads_and(mbar_wait(&sm.mbar, 0)) != 0;
            tc::fence_after_sync();
        }
        if (ok) {
            float d[16];
            tc::ld16(tc::lane_addr(tm, warp, 0), d);
            tc::wait_ld();
            float u[kDraft];
#pragma unroll
            for (int j = 0; j < kDraft; ++j) {
                u[j] = 0.f;
                if (j < D) {
                    float r = d[j];
#pragma unroll
                    for (int m = 0; m < j; ++m) r = __fmaf_rn(sm.A[j][m], u[m], r);
                    u[j] = __fmul_rn(sm.beta[j], __fsub_rn(vr[j], r));
                    float c = d[kDraft + j];
#pragma unroll
                    for (int m = 0; m <= j; ++m) c = __fmaf_rn(sm.P[j][m], u[m], c);
                    o[j] = __fmul_rn(p.scale, c);
                    uu[j] = u[j];
                }
            }
        } else {
            if (tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            // bounded second chances: no copy or product may still be running
            mbar_wait_drain(&sm.rbar, 0);
            mbar_wait_drain(&sm.sbar, 0);
            if (issued) mbar_wait_drain(&sm.mbar, 0);
        }
    }
    {
        T *ob = static_cast<T *>(p.out) + ((int64_t)n * D * p.H + h) * p.dv + tid;
#pragma unroll
        for (int j = 0; j < kDraft; ++j)
            if (j < D) Elem<T>::store1(ob + (int64_t)j * p.H * p.dv, (valid && ok) ? o[j] : 0.f);
        // u records (zero for a skipped entry)
        if (p.rec_u) {
            float *ub = p.rec_u + ((int64_t)n * D * p.H + h) * p.dv + tid;
#pragma unroll
            for (int j = 0; j < kDraft; ++j)
                if (j < D) __stcs(ub + (int64_t)j * p.H * p.dv, (valid && ok) ? uu[j] : 0.f);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, kTmemCols);
}



}  // namespace verify_tc

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

size_t verify_workspace_bytes(int H, int dk, int dv, int dtype, int64_t batch, int D) {
    if (dtype != KDA_DT_BF16 || dk != verify_tc::DK || dv != 128 || D < 1 || D > verify_tc::kDraft || batch <= 0 ||
        H <= 0)
        return 0;
    return (size_t)batch * (size_t)H * verify_tc::kRecBytes;
}

bool verify_tc_supported(const VerifyParams &p, int dk, int dtype) {
    return verify_workspace_bytes(p.H, dk, p.dv, dtype, p.batch, p.D) > 0 && p.workspace != nullptr &&
           p.num_slots > 0 && p.num_slots * (int64_t)p.H <= 0x7fffffffLL &&
           (int64_t)p.batch * p.H <= 0x7fffffffLL && tensor_map_encode_fn() != nullptr;
}

cudaError_t launch_verify_tc(const VerifyParams &p, cudaStream_t st) {
    using namespace verify_tc;
    const int64_t items = (int64_t)p.batch * p.H;
    unsigned char *ws = static_cast<unsigned char *>(p.workspace);
    CUtensorMap map;
    const cuuint64_t dims[3] = {(cuuint64_t)DK, 128, (cuuint64_t)p.num_slots * (cuuint64_t)p.H};
    const cuuint64_t strides[2] = {(cuuint64_t)DK * 4, (cuuint64_t)128 * DK * 4};
    const cuuint32_t box[3] = {32, 128, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = tensor_map_encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(p.pool), dims,
                                   strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const size_t smem_bytes = kStateSmemBytes;
    auto kern = state_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    window_kernel<__nv_bfloat16><<<(unsigned)items, kWinThreads, 0, st>>>(p, ws);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the state copies start while the window
    // kernel finishes; the state kernel waits for it before reading the records
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)items);
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const VerifyParams pp = p;
    const unsigned char *wsc = ws;
    return cudaLaunchKernelEx(&cfg, kern, pp, map, wsc);
}

}  // namespace kda
