// Tensor-core chunked prefill (tcgen05 + TMEM), dk = dv = 128, bf16 inputs.
//
// "Ascend day-0 support for Kimi K3", section "KDA Prefill and Decode dual
// path": the prefill takes 64-token chunks and organises Q/K normalisation,
// gate accumulation and the chunk KDA as batched computation.  The chunk
// form (WY/UT; gamma = in-chunk cumulative gate per key channel):
//
//   A = strict-lower( beta_r sum_c k^_r k^_j e^{gamma_r - gamma_j} ),
//   P = lower( sum_c q^_r k^_j e^{gamma_r - gamma_j} ),  T = (I + A)^-1
//   W^T = (beta K~)^T T^T,  U'^T = (beta V)^T T^T                (WY factors)
//   U^T = U'^T - S W^T,  O^T = scale (S Q~^T + U^T P^T),
//   S <- S diag(e^{gamma_C}) + U^T K^                            (chunk step)
//
// The chunk step splits into what the state does not touch and one product
// of the state (G = W^T K^, Q' = Q~ - P W):
//
//   D = U'^T K^ - S G,  O^T = scale (S Q'^T + U'^T P^T),
//   S <- S diag(e^{gamma_C}) + D
//
// Two kernels on tcgen05 (fp32 accumulate), pipelined in segments of the
// chunks (plan_segments):
//
// prep_tc_kernel  one CTA per (chunk, head), the chunks of a segment of all
//   sequences in parallel.  Computes everything that does not depend on the
//   state (A/P and the WY factors on kind::tf32, G^T and P W on kind::f16)
//   and writes, per (chunk, head), an operand image that the chain copies
//   into shared memory with one bulk copy: [-G^T; Q'] (192 x 128 keys),
//   U'^T (128 x 64 tokens) and [K^^T; P] (192 x 64 tokens) as K-major
//   128B-swizzled fp16 tiles, then e^{gamma_C} (128 fp32).
// chain_kernel  one CTA per (sequence, head) walks the chunks in order with
//   the fp32 state in registers and its fp16 copy S16 in tensor memory
//   (value row i = TMEM lane i), the A operand of the one state product:
//     ACC = U'^T [K^^T; P]^T + S16 [-G^T; Q']^T = [D | O^T]     (N = 192)
//   on kind::f16.  The first product is issued for the next chunk while the
//   state of this one is updated; the next chunks' images are in flight, and
//   a chunk's outputs leave while the next chunk's product runs.
//
// Operand precision of the chain: fp16 has the same 10-bit mantissa as tf32
// and rounds to nearest; the operands (normalised keys and queries times
// decays <= 1, the WY factors, U and the state) stay far inside its range
// for the recurrence's inputs.  A value beyond +-65504 sets KDA_DEVERR_RANGE
// (that sequence's results are then not valid).
//
// Decay factors in the A/P product: with ref = gamma at token 31 of the chunk,
// K+ = k^ e^{gamma-ref}, Q+ = q^ e^{gamma-ref}, K- = k^ e^{ref-gamma}, so that
// [K+; Q+] K-^T carries e^{gamma_r - gamma_j}.  A chunk whose gamma spans more
// than 80 (natural units) around ref on some channel would overflow these
// factors; that chunk computes A and P with one exp per (r, j, c) instead.
#include <cuda_fp16.h>
#include <stddef.h>
#include <stdint.h>

#include <climits>
#include <cmath>

#include "kda.h"
#include "kda_bulk.cuh"
#include "kda_check.cuh"
#include "kda_internal.h"
#include "kda_rowmath.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace prefill_tc {

constexpr int C = 64;   // chunk length
constexpr int D = 128;  // dk = dv
constexpr float kSpanLimit = 80.f;
constexpr float kLog2e = 1.4426950408889634f;  // log2(e)

// Operand image of one (chunk, head) in the workspace (bytes).
// Every tile is fp16, K-major and 128B-swizzled, in the layout the chain's
// products read it; row counts are those of the stacked tiles.
constexpr uint32_t IMG_BQ = 0;                         // [-G^T; Q']: 128 key rows + 64 token rows, K = 128 keys
constexpr uint32_t IMG_UPT = IMG_BQ + 192 * 128 * 2;   // U'^T: 128 value rows, K = 64 tokens
constexpr uint32_t IMG_KP = IMG_UPT + 128 * 64 * 2;    // [K^^T; P]: 128 key rows + 64 token rows, K = 64 tokens
constexpr uint32_t IMG_EGC = IMG_KP + 192 * 64 * 2;    // e^{gamma_C}, 128 fp32
constexpr uint32_t IMG_TILES = IMG_EGC;                // the tiles, copied to the chain as one block
constexpr uint32_t IMG_BYTES = IMG_EGC + 1024;         // 89 KiB
constexpr float kHalfMax = 65504.f;                    // largest finite fp16

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t plan_bytes(int32_t num_seqs) {
    return round_up(sizeof(int32_t) * ((size_t)num_seqs + 2), 1024);
}
__host__ __device__ inline int64_t max_chunks(int32_t num_seqs, int64_t total_tokens) {
    return (total_tokens + C - 1) / C + num_seqs;
}

// fp16 element (row, k) of a K-major 128B-swizzled tile
__device__ __forceinline__ void st_h(unsigned char *tile, int rows, int row, int k, float x) {
    *reinterpret_cast<__half *>(tile + tc::sw128_off16(row, k, rows)) = __float2half_rn(x);
}

// four consecutive floats of a 16-byte aligned shared-memory row
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// two fp16 values in one 32-bit word: a in the low half, b in the high half
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// pack_h2 that also folds |a|, |b| (as fp16) into a running maximum: the
// maximum is infinite once a value overflowed fp16 (NaNs are ignored)
__device__ __forceinline__ uint32_t pack_h2_track(float a, float b, __half2 &hmax) {
    const __half2 h = __floats2half2_rn(a, b);
    hmax = __hmax2(hmax, __habs2(h));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 2^x with the special function unit's approximate base-2 exponential
// (results below the normal range flush to zero); e^y = 2^{y log2(e)}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait on an MMA-completion barrier; the result is made uniform across
// the CTA and a timeout is recorded in the error flag.  `phase` advances only
// when the wait succeeded, so after a timeout it still names the pending
// phase, which is the one a drain must wait for.
// Thread 0 alone polls; the other threads wait in the CTA barrier, where
// they spend no issue slots.
__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase, int32_t *err_flag) {
    const bool mine = threadIdx.x == 0 ? mbar_wait(bar, phase & 1) : true;
    const bool ok = __syncthreads_and(mine) != 0;
    if (ok) phase ^= 1;
    if (!ok && threadIdx.x == 0 && err_flag) atomicOr(err_flag, KDA_DEVERR_TIMEOUT);
    tc::fence_after_sync();
    return ok;
}

// Sequence s owning global chunk index c (plan[s] <= c < plan[s+1]).
__device__ inline int find_seq(const int32_t *plan, int n, int32_t c) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (plan[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ================================================================== prep

// One CTA of 8 warps per (chunk, head), two CTAs per SM.  TMEM lane l of a
// warp's quarter is either a token row (row phases: lanes 0..63 the chunk's
// keys, 64..127 its queries) or a key channel / value row (channel phases);
// warps w and w + 4 serve the same lanes and take one half of the columns
// (row phases) or of the tokens (channel phases).
//
// The chunk's k, q and g arrive by TMA as K-major 128B-swizzled boxes (the
// layout of an MMA operand tile, so both row and column reads are free of
// bank conflicts); v follows into q's buffer once q has been used.  Steps:
//   0. (fused prefill) ShortConv of k and q in place in their boxes
//   1. L2Norm sums of squares per token row
//   2. gamma = running sum of g per channel, in place (four token quarters
//      at once, each then adding the sums of the quarters before it); ref =
//      gamma_31, gamma_C and the span check; norms and beta
//   3. row phase: [K+; Q+] into TMEM (the A operand of the A/P product),
//      K- into a shared tile (its B operand), Q~ rows of the image
//   4. channel phase, while G = [K+; Q+] K-^T runs: beta K~^T into TMEM (the
//      A operand of W^T), K^^T rows of the image
//   5. A' and P from G; P rows of the image
//   6. T = (I + A)^-1 by doubling
//   7. beta V^T into TMEM; W^T = (beta K~)^T T^T, U'^T = (beta V)^T T^T
//   8. W^T into a shared tile, U'^T rows of the image (one bulk store)
//   9. G^T = K^^T W and P W (kind::f16, [K^^T; P] read back from the
//      image); [-G^T; Q'] rows of the image (one bulk store)
// Independent products are issued from two threads (0 and 32).
// TMEM columns: [K+; Q+] 0..127 (then beta V^T 0..63 and W^T 64..127),
// G 128..191 (then U'^T), beta K~^T 192..255; step 9's G^T 0..127 and
// P W 128..255.
constexpr uint32_t PT_A = 0, PT_BV = 0, PT_WT = 64, PT_G = 128, PT_UPT = 128, PT_BK = 192;
constexpr uint32_t PT_COLS = 256;
constexpr int kPrepThreads = 256;

// Scratch of the UT inverse, laid over the k staging and the K- tile once the
// A/P product and the channel phase have read them.
struct InvScratch {
    float As[C][C + 4];  // rows 16-byte aligned; a quarter warp's rows hit distinct banks
    float Ts[C][C + 4];  // the same: its rows leave as float4 reads, a quarter warp's free of conflicts
};

struct PrepSmem {
    union {
        struct {
            unsigned char kst[C * D * 2];  // k: two 64-channel boxes, bf16, 128B-swizzled
            unsigned char km[C * D * 4];   // K- (B of the A/P product): 64 rows x K 128, tf32
        } a;
        InvScratch inv;
    } u1;
    unsigned char qv[C * D * 2];           // q, then v (the same box layout as k)
    union {
        unsigned char gam[C * D * 4];      // g, then gamma in place: four 32-channel fp32 boxes
        unsigned char t[C * C * 4];        // T (B of the WY products) once gamma is no longer read
    } u2;
    float invk[C], invq[C], beta[C];
    float nrm[2][2 * C];  // sums of squares over each channel half: rows k_0..k_63, q_0..q_63
    float ref[D];         // gamma at token 31
    float gC[D];          // gamma at the chunk's last token
    float eref[D];        // e^{ref}
    float nrl[D];         // -ref log2(e)
    union {
        float xs[32][33];  // partial products of the UT inverse
        struct {           // the gamma scan's token quarters, per channel:
            float tot[4][D];  // sums
            float mn[3][D];   // extremes of the running sums of quarters 1..3
            float mx[3][D];
        } gq;
    } u3;
    float vhist[3][D];    // fused: the three value inputs before the chunk
    uint64_t bar_in, bar_v, bar_mma, bar_q, bar_kp;
    uint32_t tmem_base;
};
constexpr size_t kPrepSmem = sizeof(PrepSmem) + 1024;
static_assert(sizeof(InvScratch) <= C * D * 6, "inverse scratch must fit the k staging and the K- tile");
static_assert(offsetof(InvScratch, Ts) % 16 == 0, "float4 rows of T");
static_assert(offsetof(PrepSmem, qv) % 1024 == 0 && offsetof(PrepSmem, u2) % 1024 == 0, "TMA boxes");
static_assert(offsetof(PrepSmem, invk) % 16 == 0 && offsetof(PrepSmem, beta) % 16 == 0, "vector loads");
static_assert(offsetof(PrepSmem, u3) % 8 == 0 && offsetof(PrepSmem, gC) % 8 == 0, "paired gamma statistics");

// The staged k and q boxes hold the bf16 inputs; the fused prefill
// overwrites them with the convolved values as fp16 (10-bit mantissa, so the
// rounding stays below the later fp16 operands').  A 32-bit word of a box
// holds two consecutive channels.
template <bool F16>
__device__ __forceinline__ float2 box_pair(uint32_t w) {
    if constexpr (F16) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
}

template <bool F16>
__device__ __forceinline__ float box_elem(const unsigned char *box, int r, int c) {
    const unsigned char *e = box + tc::sw128_off16(r, c, C);
    if constexpr (F16) {
        return __half2float(*reinterpret_cast<const __half *>(e));
    } else {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(e));
    }
}

// staged bf16 element (row r, channel c) and fp32 element of a 64-row tile
__device__ __forceinline__ float st_bf16(const unsigned char *box, int r, int c) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(box + tc::sw128_off16(r, c, C)));
}
__device__ __forceinline__ float &st_f32(unsigned char *tile, int r, int c) {
    return *reinterpret_cast<float *>(tile + tc::sw128_off(r, c, C));
}

// ---- fused ShortConv (the MegaKDA-style prefill)

constexpr int kConvChannels = 3 * D;  // q | k | v channels of a head

// sigmoid(z), the output gate, with the fast exponential and division (a
// few ulp)
__device__ __forceinline__ float sigmoid_gate(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// The three raw inputs before token t0 of conv channel ch (q | k | v order)
// of head h, oldest first: from the sequence itself after its first chunk,
// else from the slot's conv state (init_from_pool) or zero.
template <typename T>
__device__ __forceinline__ void conv_history(const PrefillParams &p, bool first, int slot, int h, int t0, int ch,
                                             float (&hist)[3]) {
    if (!first) {
        const T *src = ch < D ? static_cast<const T *>(p.q) : ch < 2 * D ? static_cast<const T *>(p.k)
                                                                       : static_cast<const T *>(p.v);
        const int c = ch % D;
#pragma unroll
        for (int j = 0; j < 3; ++j) hist[j] = Elem<T>::load1(src + ((int64_t)(t0 - 3 + j) * p.H + h) * D + c);
    } else if (p.init_from_pool) {
        const T *cs = static_cast<const T *>(p.conv_state) + ((int64_t)slot * p.H + h) * (3 * kConvChannels);
#pragma unroll
        for (int j = 0; j < 3; ++j) hist[j] = Elem<T>::load1(cs + j * kConvChannels + ch);
    } else {
        hist[0] = hist[1] = hist[2] = 0.f;
    }
}

// 1/x with the special function unit's approximate reciprocal
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu of two values: a / (1 + e^{-a}), e^{-a} = 2^{-a log2(e)}, on the
// approximate exponential and reciprocal (a few ulp; the convolved k and q
// are rounded to fp16 right after, v enters beta V^T in fp32)
__device__ __forceinline__ float2 silu2(float2 a) {
    const float2 t = __fmul2_rn(a, make_float2(-kLog2e, -kLog2e));
    const float2 d = __fadd2_rn(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
    return __fmul2_rn(a, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// silu(w . (x_{t-3}, x_{t-2}, x_{t-1}, x_t)) at two consecutive tokens t
// (inputs x0..x3) and t + 1 (x1..x4), in the fused decode's order of taps
__device__ __forceinline__ float2 conv_tap2(float4 w, float x0, float x1, float x2, float x3, float x4) {
    float2 acc = __fmul2_rn(make_float2(w.x, w.x), make_float2(x0, x1));
    acc = __ffma2_rn(make_float2(w.y, w.y), make_float2(x1, x2), acc);
    acc = __ffma2_rn(make_float2(w.z, w.z), make_float2(x2, x3), acc);
    acc = __ffma2_rn(make_float2(w.w, w.w), make_float2(x3, x4), acc);
    return silu2(acc);
}

template <typename T, bool FUSED>
__global__ void __launch_bounds__(kPrepThreads, 2) prep_tc_kernel(const PrefillParams p,
                                                                   const __grid_constant__ CUtensorMap kmap,
                                                                   const __grid_constant__ CUtensorMap qmap,
                                                                   const __grid_constant__ CUtensorMap vmap,
                                                                   const __grid_constant__ CUtensorMap gmap,
                                                                   const int seg_lo, const int seg_len,
                                                                   const int pdl_wait) {
    extern __shared__ unsigned char smem_raw[];
    PrepSmem &sm =
        *reinterpret_cast<PrepSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t *plan = static_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    // A segment launched behind the previous segment's chain (pdl_wait) may
    // run beside it; one CTA waits for that chain to complete before it
    // exits, so the next chain, an ordinary launch behind this grid, starts
    // from the state the previous one wrote.
    const bool waiter = pdl_wait && blockIdx.x == 0 && blockIdx.y == 0;
    auto leave = [&]() {
        if (waiter) asm volatile("griddepcontrol.wait;" ::: "memory");
    };
    if (plan[n + 1] == 0) return leave();
    // the chunk: seg_len > 0 maps CTA x to local chunk seg_lo + x % seg_len
    // of sequence x / seg_len; seg_len = 0 maps it to global chunk x, taken
    // only from local chunk seg_lo on
    auto map_chunk = [&](int x, int &sq, int32_t &ch) {
        if (seg_len > 0) {
            sq = x / seg_len;
            if (sq >= n) return false;
            const int32_t local = seg_lo + (int32_t)(x % seg_len);
            if (local >= plan[sq + 1] - plan[sq]) return false;
            ch = plan[sq] + local;
        } else {
            ch = x;
            if (ch >= plan[n]) return false;
            sq = find_seq(plan, n, ch);
            if (ch - plan[sq] < seg_lo) return false;
        }
        return true;
    };
    int32_t chunk;
    int s;
    if (!map_chunk((int)blockIdx.x, s, chunk)) return leave();
    const int h = blockIdx.y, H = p.H;
    const int slot = p.slot_ids[s];
    if (slot < 0 || (int64_t)slot >= p.num_slots) return leave();  // the chain writes zeros
    const int t0 = p.cu_seqlens[s] + (chunk - plan[s]) * C;
    const int L = p.cu_seqlens[s + 1] - t0 < C ? p.cu_seqlens[s + 1] - t0 : C;
    // checked build: the chunk's tokens, its operand image and the slot's
    // conv state
    if (!in_bounds(t0, L, p.total_tokens, p.err_flag) ||
        !in_bounds((int64_t)(plan_bytes(n) + ((size_t)chunk * H + h) * IMG_BYTES), IMG_BYTES,
                   (int64_t)p.workspace_bytes, p.err_flag) ||
        (FUSED && !in_bounds(((int64_t)slot * H + h) * 3 * kConvChannels, 3 * kConvChannels,
                             p.num_slots * H * (int64_t)(3 * kConvChannels), p.err_flag)))
        return leave();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lr = ((warp & 3) << 5) | lane;  // TMEM lane
    const int hf = warp >> 2;                 // half of the columns or tokens
    unsigned char *__restrict__ img = static_cast<unsigned char *>(p.workspace) + plan_bytes(n) +
                                      ((size_t)chunk * H + h) * (size_t)IMG_BYTES;
    // fused: the conv histories are requested first, so that they arrive
    // with the staged inputs (k and q per thread; v's through shared memory)
    float khist[3];
    if constexpr (FUSED) {
        conv_history<T>(p, chunk == plan[s], slot, h, t0, (tid >= 128 ? 0 : D) + (tid & 127), khist);
        if (tid < D) {
            float vh[3];
            conv_history<T>(p, chunk == plan[s], slot, h, t0, 2 * D + tid, vh);
#pragma unroll
            for (int j = 0; j < 3; ++j) sm.vhist[j][tid] = vh[j];
        }
    }
    unsigned char *kst = sm.u1.a.kst, *km = sm.u1.a.km, *qv = sm.qv, *gam = sm.u2.gam;

    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, PT_COLS);
    if (tid == 0) {
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_v, 1);
        mbar_init(&sm.bar_q, 1);
        mbar_init(&sm.bar_kp, 1);
        mbar_init(&sm.bar_mma, 2);  // threads 0 and 32 each commit their products
        fence_barrier_init();
        mbar_arrive_expect_tx(&sm.bar_in, 2 * (C * D * 2) + C * D * 4);  // k, q (bf16) and g (fp32)
        tma_load_2d(kst, &kmap, h * D, t0, &sm.bar_in);
        tma_load_2d(kst + C * 128, &kmap, h * D + 64, t0, &sm.bar_in);
        tma_load_2d(qv, &qmap, h * D, t0, &sm.bar_in);
        tma_load_2d(qv + C * 128, &qmap, h * D + 64, t0, &sm.bar_in);
#pragma unroll
        for (int i = 0; i < 4; ++i) tma_load_2d(gam + i * C * 128, &gmap, h * D + 32 * i, t0, &sm.bar_in);
    }
    const T *__restrict__ bb = static_cast<const T *>(p.b);
    // b of token tid - 128, for the thread that forms that token's beta
    const float bval = (tid >= 2 * C && tid - 2 * C < L) ? Elem<T>::load1(bb + (int64_t)(t0 + tid - 2 * C) * H + h)
                                                         : 0.f;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem_base;
    uint32_t phase = 0;
    // outstanding asynchronous work, for the drain after a timeout
    bool in_pend = true, v_pend = false, mma_pend = false, q_pend = false, kp_pend = false;
    bool ok = __syncthreads_and(tid == 0 ? mbar_wait(&sm.bar_in, 0) : true) != 0;
    if (ok) {
        in_pend = false;
        mbar_try_wait(&sm.bar_in, 0);
    } else if (tid == 0 && p.err_flag) {
        atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
    }
    __half2 hmax = __float2half2_rn(0.f);  // largest |entry| of the chain's fp16 operands written here
    bool bulk_out = false;  // thread 0: bulk stores of staged image tiles issued
    bool unsafe = false;
    auto issue_v = [&]() {  // thread 0, once q has been read
        mbar_arrive_expect_tx(&sm.bar_v, C * D * 2);
        tma_load_2d(qv, &vmap, h * D, t0, &sm.bar_v);
        tma_load_2d(qv + C * 128, &vmap, h * D + 64, t0, &sm.bar_v);
    };

    if (FUSED && ok) {
        // ---- 0. ShortConv of k (threads 0..127: channel tid) and q (128..255),
        // in place in the staged boxes as fp16, tokens in descending order so
        // that every step still reads raw (bf16) inputs
        const int ch = tid & 127;
        const bool isq = tid >= 128;
        const int cch = (isq ? 0 : D) + ch;  // conv channel (q | k | v)
        unsigned char *box = (isq ? qv : kst) + (ch >> 6) * C * 128;
        const int cc = ch & 63;
        const float4 w = __ldg(reinterpret_cast<const float4 *>(p.conv_w) + (int64_t)h * kConvChannels + cch);
        const float(&hist)[3] = khist;
        // row r of the channel sits at r * 128 + ((u ^ (r & 7)) << 4) + e in
        // its box; the unrolled 16-row blocks make r & 7 a constant
        const int u = cc >> 3, e = (cc & 7) << 1;
        auto at = [&](int r) { return box + r * 128 + ((u ^ (r & 7)) << 4) + e; };
        auto x_at = [&](int r) {
            return r >= 0 ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(at(r))) : hist[3 + r];
        };
        // blocks of 16 rows from the top: the block's 16 inputs and the three
        // below it are loaded first (those rows are still raw: only rows
        // above have been overwritten), then its 16 outputs are stored
#pragma unroll 1
        for (int blk = (L - 1) >> 4; blk >= 0; --blk) {
            float x[19];  // x[i] = input of row 16 blk - 3 + i
#pragma unroll
            for (int i = 0; i < 19; ++i) {
                const int r = 16 * blk - 3 + i;
                x[i] = r < L ? x_at(r) : 0.f;
            }
            // rows r and r + 1 at once; a row past the chunk is neither
            // stored nor range-checked (an overflow shows as infinity in hmax)
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const int r = 16 * blk + j;
                if (r < L) {
                    const float2 y = conv_tap2(w, x[j], x[j + 1], x[j + 2], x[j + 3], x[j + 4]);
                    const __half2 h2 = __floats2half2_rn(y.x, r + 1 < L ? y.y : 0.f);
                    hmax = __hmax2(hmax, __habs2(h2));
                    *reinterpret_cast<__half *>(at(r)) = __low2half(h2);
                    if (r + 1 < L) *reinterpret_cast<__half *>(at(r + 1)) = __high2half(h2);
                }
            }
        }
        __syncthreads();
    }
    if (ok) {
        // ---- 1. L2Norm sums of squares (thread = row of k (0..63) or q, one
        // 64-channel half; the 16-byte units of a row are read in its swizzled
        // order, so a warp's rows hit distinct banks)
        {
            const int row = tid & 127, ch = tid >> 7;
            const int r = row & 63;
            const unsigned char *box = (row < 64 ? kst : qv) + ch * C * 128;
            float2 ss = make_float2(0.f, 0.f);
            if (r < L) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(box + r * 128 + ((u ^ (r & 7)) << 4));
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 ab = box_pair<FUSED>(w4[e]);
                        ss = __ffma2_rn(ab, ab, ss);
                    }
                }
            }
            sm.nrm[ch][row] = ss.x + ss.y;
        }
        // ---- 2. gamma, in place (thread = channel pair cp, channels 2 cp and
        // 2 cp + 1, and token quarter qq, tokens 16 qq .. + 15): each
        // quarter's running sums from zero on paired adds, then, once the
        // quarters' sums are known, the sum of the quarters before it added;
        // rows past the chunk's end repeat gamma_C.  The quarter-0 threads
        // finish each channel: ref = gamma_31, gamma_C, the span check.
        {
            const int cp = tid & 63, qq = tid >> 6, c2 = 2 * cp;
            float2 part[16];
            float2 acc = make_float2(0.f, 0.f), mn = acc, mx = acc, gcl = acc;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * qq + i;
                if (r < L) acc = __fadd2_rn(acc, *reinterpret_cast<const float2 *>(gam + tc::sw128_off(r, c2, C)));
                part[i] = acc;
                if (r == L - 1) gcl = acc;
                mn = i == 0 ? acc : make_float2(fminf(mn.x, acc.x), fminf(mn.y, acc.y));
                mx = i == 0 ? acc : make_float2(fmaxf(mx.x, acc.x), fmaxf(mx.y, acc.y));
            }
            *reinterpret_cast<float2 *>(&sm.u3.gq.tot[qq][c2]) = acc;
            if (qq > 0) {
                *reinterpret_cast<float2 *>(&sm.u3.gq.mn[qq - 1][c2]) = mn;
                *reinterpret_cast<float2 *>(&sm.u3.gq.mx[qq - 1][c2]) = mx;
            }
            if (((L - 1) >> 4) == qq) *reinterpret_cast<float2 *>(&sm.gC[c2]) = gcl;  // the quarter's own sum
            __syncthreads();
            float2 off[4];
            off[0] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 1; j < 4; ++j)
                off[j] = __fadd2_rn(off[j - 1], *reinterpret_cast<const float2 *>(&sm.u3.gq.tot[j - 1][c2]));
            auto off_of = [&](int j) { return j == 0 ? off[0] : j == 1 ? off[1] : j == 2 ? off[2] : off[3]; };
            const float2 o = off_of(qq);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<float2 *>(gam + tc::sw128_off(16 * qq + i, c2, C)) = __fadd2_rn(part[i], o);
            if (qq == 0) {
                const float2 ref = off[2];  // gamma_31
                float2 gmin = mn, gmax = mx;
#pragma unroll
                for (int j = 1; j < 4; ++j) {
                    const float2 a = __fadd2_rn(*reinterpret_cast<const float2 *>(&sm.u3.gq.mn[j - 1][c2]), off[j]);
                    const float2 b = __fadd2_rn(*reinterpret_cast<const float2 *>(&sm.u3.gq.mx[j - 1][c2]), off[j]);
                    gmin = make_float2(fminf(gmin.x, a.x), fminf(gmin.y, a.y));
                    gmax = make_float2(fmaxf(gmax.x, b.x), fmaxf(gmax.y, b.y));
                }
                const float2 gCv = __fadd2_rn(*reinterpret_cast<const float2 *>(&sm.gC[c2]), off_of((L - 1) >> 4));
                *reinterpret_cast<float2 *>(&sm.gC[c2]) = gCv;
                *reinterpret_cast<float2 *>(&sm.ref[c2]) = ref;
                unsafe = fmaxf(gmax.x - ref.x, ref.x - gmin.x) > kSpanLimit ||
                         fmaxf(gmax.y - ref.y, ref.y - gmin.y) > kSpanLimit;
                *reinterpret_cast<float2 *>(img + IMG_EGC + 4 * c2) = make_float2(expf(gCv.x), expf(gCv.y));
                *reinterpret_cast<float2 *>(&sm.eref[c2]) = make_float2(expf(ref.x), expf(ref.y));
                *reinterpret_cast<float2 *>(&sm.nrl[c2]) = make_float2(-ref.x * kLog2e, -ref.y * kLog2e);
            } else if (tid >= 2 * C) {
                // (threads 128..255 = k row, then q row) the norms and beta
                const int t = tid - 2 * C, r = t & (C - 1);
                const float inv = (r < L) ? rsqrtf(sm.nrm[0][t] + sm.nrm[1][t] + p.eps) : 0.f;
                if (t >= C) {
                    sm.invq[r] = inv;
                } else {
                    sm.invk[r] = inv;
                    sm.beta[r] = (r < L) ? sigmoid_f(bval) : 0.f;
                }
            }
        }
        unsafe = __syncthreads_or(unsafe) != 0;

        // ---- 3. row phase (thread = token row lr of k (lr < 64) or of q,
        // channels 64 hf .. 64 hf + 63, eight at a time)
        {
            const int tok = lr & (C - 1);
            const bool isq = lr >= C;
            const float inv = isq ? sm.invq[tok] : sm.invk[tok];
            const unsigned char *box = (isq ? qv : kst) + hf * C * 128;
#pragma unroll 1
            for (int u = 0; u < 8; ++u) {
                const int c0 = 64 * hf + 8 * u;
                const uint4 raw = *reinterpret_cast<const uint4 *>(box + tok * 128 + ((u ^ (tok & 7)) << 4));
                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
                float2 x2[4], g2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) x2[e] = __fmul2_rn(box_pair<FUSED>(w4[e]), make_float2(inv, inv));
                {
                    const float4 g0 = *reinterpret_cast<const float4 *>(gam + tc::sw128_off(tok, c0, C));
                    const float4 g1 = *reinterpret_cast<const float4 *>(gam + tc::sw128_off(tok, c0 + 4, C));
                    g2[0] = make_float2(g0.x, g0.y);
                    g2[1] = make_float2(g0.z, g0.w);
                    g2[2] = make_float2(g1.x, g1.y);
                    g2[3] = make_float2(g1.z, g1.w);
                }
                float2 qt2[4];
                if (!unsafe) {
                    // t = (gamma - ref) log2(e): e^{gamma - ref} = 2^t and
                    // e^{ref - gamma} = 2^-t
                    const float4 n0 = *reinterpret_cast<const float4 *>(&sm.nrl[c0]);
                    const float4 n1 = *reinterpret_cast<const float4 *>(&sm.nrl[c0 + 4]);
                    const float2 nr2[4] = {make_float2(n0.x, n0.y), make_float2(n0.z, n0.w), make_float2(n1.x, n1.y),
                                           make_float2(n1.z, n1.w)};
                    float2 t2[4], plus2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        t2[e] = __ffma2_rn(g2[e], make_float2(kLog2e, kLog2e), nr2[e]);
                        plus2[e] = __fmul2_rn(x2[e], make_float2(ex2_approx(t2[e].x), ex2_approx(t2[e].y)));
                    }
                    tc::st8(tc::lane_addr(tm, warp, PT_A + c0), *reinterpret_cast<const float(*)[8]>(&plus2[0]));
                    if (!isq) {  // (warp-uniform) K- = k^ e^{ref - gamma}
                        float2 mi2[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            mi2[e] = __fmul2_rn(x2[e], make_float2(ex2_approx(-t2[e].x), ex2_approx(-t2[e].y)));
                        *reinterpret_cast<float4 *>(km + tc::sw128_off(tok, c0, C)) =
                            make_float4(mi2[0].x, mi2[0].y, mi2[1].x, mi2[1].y);
                        *reinterpret_cast<float4 *>(km + tc::sw128_off(tok, c0 + 4, C)) =
                            make_float4(mi2[2].x, mi2[2].y, mi2[3].x, mi2[3].y);
                    } else {  // Q~ = q^ e^{gamma} = Q+ e^{ref}
                        const float4 e0 = *reinterpret_cast<const float4 *>(&sm.eref[c0]);
                        const float4 e1 = *reinterpret_cast<const float4 *>(&sm.eref[c0 + 4]);
                        qt2[0] = __fmul2_rn(plus2[0], make_float2(e0.x, e0.y));
                        qt2[1] = __fmul2_rn(plus2[1], make_float2(e0.z, e0.w));
                        qt2[2] = __fmul2_rn(plus2[2], make_float2(e1.x, e1.y));
                        qt2[3] = __fmul2_rn(plus2[3], make_float2(e1.z, e1.w));
                    }
                } else if (isq) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        qt2[e] = make_float2(x2[e].x * expf(g2[e].x), x2[e].y * expf(g2[e].y));
                }
                if (isq)  // Q~: row 128 + tok of [-G^T; Q'] until Q' replaces it
                    *reinterpret_cast<uint4 *>(img + IMG_BQ + tc::sw128_off16(128 + tok, c0, 192)) =
                        make_uint4(pack_h2(qt2[0].x, qt2[0].y), pack_h2(qt2[1].x, qt2[1].y),
                                   pack_h2(qt2[2].x, qt2[2].y), pack_h2(qt2[3].x, qt2[3].y));
            }
            // the Q~ rows come back by bulk copy in step 9
            fence_proxy_async_global();
        }
        tc::wait_st();
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (!unsafe) {
            if (tid == 0 || tid == 32) {
                // G = [K+; Q+] K-^T: M = 128, N = 64 tokens j, K = 128
                // (kind::tf32); threads 0 and 32 issue one 32-token half each
                constexpr uint32_t id = tc::idesc_tf32(128, 32);
                const int jh = tid >> 5;
                const uint32_t b0 = tc::smem_u32(km) + jh * 32 * 128;
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_tf32_ts(tm + PT_G + 32 * jh, tm + PT_A + 8 * ks, tc::desc_tf32_kstep(b0, 64, ks), id,
                                    ks > 0);
                tc::commit(&sm.bar_mma);
                if (tid == 0) issue_v();  // q has been read: v takes its buffer
            }
            mma_pend = v_pend = true;
        }

        // ---- 4. channel phase (thread = channel lr, tokens 32 hf .. + 31):
        // beta K~^T into TMEM, K^^T row lr of the image
        {
            // K^ = k^ e^{gamma_C - gamma} = K- e^{gamma_C - ref} on the split
            // path (K- is zero past the chunk's end); directly otherwise
            const float gCv = sm.gC[lr];
            const float egcref = unsafe ? 0.f : expf(gCv - sm.ref[lr]);
            float bk[32];
            uint32_t kw[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                // tokens r and r + 1 as pairs: beta k^ e^{gamma} = beta k^ 2^{gamma log2(e)}
                const int r = 32 * hf + i;
                const float2 ik = *reinterpret_cast<const float2 *>(&sm.invk[r]);
                const float2 bt = *reinterpret_cast<const float2 *>(&sm.beta[r]);
                const float2 kx =
                    __fmul2_rn(make_float2(box_elem<FUSED>(kst, r, lr), box_elem<FUSED>(kst, r + 1, lr)), ik);
                const float2 g = make_float2(st_f32(gam, r, lr), st_f32(gam, r + 1, lr));
                const float2 t = __fmul2_rn(g, make_float2(kLog2e, kLog2e));
                const float2 b2 = __fmul2_rn(__fmul2_rn(bt, kx), make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                bk[i] = b2.x;
                bk[i + 1] = b2.y;
                float2 kh;
                if (!unsafe)
                    kh = __fmul2_rn(make_float2(st_f32(km, r, lr), st_f32(km, r + 1, lr)), make_float2(egcref, egcref));
                else
                    kh = make_float2(r < L ? kx.x * expf(gCv - g.x) : 0.f, r + 1 < L ? kx.y * expf(gCv - g.y) : 0.f);
                kw[i >> 1] = pack_h2(kh.x, kh.y);
            }
            tc::st16(tc::lane_addr(tm, warp, PT_BK + 32 * hf), *reinterpret_cast<float(*)[16]>(&bk[0]));
            tc::st16(tc::lane_addr(tm, warp, PT_BK + 32 * hf + 16), *reinterpret_cast<float(*)[16]>(&bk[16]));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4 *>(img + IMG_KP + tc::sw128_off16(lr, 32 * hf + 8 * j, 192)) =
                    make_uint4(kw[4 * j], kw[4 * j + 1], kw[4 * j + 2], kw[4 * j + 3]);
        }

        // ---- 5. A' and P
        if (!unsafe) {
            ok = wait_mma(&sm.bar_mma, phase, p.err_flag);
            if (ok) {
                mma_pend = false;
                // G rows (TMEM lanes): 0..63 are A', 64..127 are P; columns
                // (tokens j) 32 hf .. + 31
                float g32[32];
                tc::ld16(tc::lane_addr(tm, warp, PT_G + 32 * hf), *reinterpret_cast<float(*)[16]>(&g32[0]));
                tc::ld16(tc::lane_addr(tm, warp, PT_G + 32 * hf + 16), *reinterpret_cast<float(*)[16]>(&g32[16]));
                tc::wait_ld();
                if (lr < C) {
                    const int r = lr;
                    const float br = sm.beta[r];
#pragma unroll
                    for (int j4 = 0; j4 < 32; j4 += 4) {
                        float a4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 32 * hf + j4 + e;
                            a4[e] = (j < r) ? br * g32[j4 + e] : 0.f;
                        }
                        *reinterpret_cast<float4 *>(&sm.u1.inv.As[r][32 * hf + j4]) =
                            make_float4(a4[0], a4[1], a4[2], a4[3]);
                    }
                } else {
                    const int r = lr - C;
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 32 * hf + 8 * j8 + 2 * e;
                            w[e] = pack_h2(j <= r ? g32[8 * j8 + 2 * e] : 0.f, j + 1 <= r ? g32[8 * j8 + 2 * e + 1] : 0.f);
                        }
                        *reinterpret_cast<uint4 *>(img + IMG_KP + tc::sw128_off16(128 + r, 32 * hf + 8 * j8, 192)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        } else {
            // exact path: one exp per (r, j, c); A goes to registers first
            // because its scratch overlays the k staging
            float areg[C * C / kPrepThreads];
#pragma unroll 1
            for (int it = 0; it < C * C / kPrepThreads; ++it) {
                const int idx = tid + it * kPrepThreads;
                const int r = idx / C, j = idx % C;
                float a = 0.f, pp = 0.f;
                if (j <= r) {
                    for (int cc = 0; cc < D; ++cc) {
                        const float gr = st_f32(gam, r, cc), gj = st_f32(gam, j, cc);
                        const float m = box_elem<FUSED>(kst, j, cc) * sm.invk[j] * expf(gr - gj);
                        a = fmaf(box_elem<FUSED>(kst, r, cc) * sm.invk[r], m, a);
                        pp = fmaf(box_elem<FUSED>(qv, r, cc) * sm.invq[r], m, pp);
                    }
                }
                areg[it] = (j < r) ? sm.beta[r] * a : 0.f;
                st_h(img + IMG_KP, 192, 128 + r, j, (j <= r) ? pp : 0.f);
            }
            __syncthreads();
#pragma unroll
            for (int it = 0; it < C * C / kPrepThreads; ++it) {
                const int idx = tid + it * kPrepThreads;
                sm.u1.inv.As[idx / C][idx % C] = areg[it];
            }
            if (tid == 0) issue_v();
            v_pend = true;
        }
        // the image rows of K^^T and P are read back by a bulk copy later
        fence_proxy_async_global();
        __syncthreads();
    }

    if (ok) {
        // ---- 6. T = (I + A)^-1 (unit lower triangular) by doubling: the four
        // 16 x 16 diagonal blocks by forward substitution (one column per
        // thread, in registers); then the lower-left 16 x 16 block of each
        // 32-row block as -T22 (A21 T11); then the lower-left 32 x 32 block of
        // the whole matrix the same way
        float(*As)[C + 4] = sm.u1.inv.As;
        float(*Ts)[C + 4] = sm.u1.inv.Ts;
        if (tid < C) {
            const int I = tid >> 4, jj = tid & 15, o = 16 * I;
            float col[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc2 = (r == jj) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m)
                    if (m >= jj) acc2 = fmaf(-As[o + r][o + m], col[m], acc2);
                col[r] = (r >= jj) ? acc2 : 0.f;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Ts[o + r][o + jj] = col[r];
        } else {
            for (int idx = tid - C; idx < C * C; idx += kPrepThreads - C) {
                const int r = idx / C, j = idx % C;
                if ((j >> 4) > (r >> 4)) Ts[r][j] = 0.f;
            }
        }
        __syncthreads();
        // The block products keep two outputs (level 1) or a 2 x 2 block of
        // outputs (level 2) per thread, so that each operand load serves two
        // products, which run as one paired fp32 fused multiply-add; the row
        // operands (rows of A or T, 16-byte aligned) are read four at a time.
        // The upper triangles of the diagonal blocks and the upper right
        // blocks hold zeros, so the sums run over whole blocks.
        {
            // level 1: X1 = A21 T11 per 32-row block ob (rows 2 rp, 2 rp + 1,
            // column j of the 16 x 16 block), then T21 = -T22 X1
            const int ob = tid >> 7, o = 32 * ob, rp = (tid >> 4) & 7, j = tid & 15;
            const int r0 = 2 * rp;
            float2 x01 = make_float2(0.f, 0.f);  // rows r0, r0 + 1
#pragma unroll
            for (int k4 = 0; k4 < 16; k4 += 4) {
                const float4 a0 = ld4(&As[o + 16 + r0][o + k4]), a1 = ld4(&As[o + 17 + r0][o + k4]);
                const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float t = Ts[o + k4 + e][o + j];
                    x01 = __ffma2_rn(make_float2(av0[e], av1[e]), make_float2(t, t), x01);
                }
            }
            sm.u3.xs[16 * ob + r0][j] = x01.x;
            sm.u3.xs[16 * ob + r0 + 1][j] = x01.y;
            __syncthreads();
            float2 y01 = make_float2(0.f, 0.f);
#pragma unroll
            for (int m4 = 0; m4 < 16; m4 += 4) {
                const float4 a0 = ld4(&Ts[o + 16 + r0][o + 16 + m4]), a1 = ld4(&Ts[o + 17 + r0][o + 16 + m4]);
                const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = sm.u3.xs[16 * ob + m4 + e][j];
                    y01 = __ffma2_rn(make_float2(av0[e], av1[e]), make_float2(x, x), y01);
                }
            }
            Ts[o + 16 + r0][o + j] = -y01.x;
            Ts[o + 17 + r0][o + j] = -y01.y;
        }
        __syncthreads();
        {
            // level 2: X2 = A21 T11 over the 32 x 32 blocks (rows 2 rp,
            // 2 rp + 1; columns cp, cp + 16), then T21 = -T22 X2
            const int rp = tid >> 4, cp = tid & 15;
            const int r0 = 2 * rp;
            // row r0 (x0) and r0 + 1 (x1), columns (cp, cp + 16) as pairs
            float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k4 = 0; k4 < 32; k4 += 4) {
                const float4 a0 = ld4(&As[32 + r0][k4]), a1 = ld4(&As[33 + r0][k4]);
                const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 t = make_float2(Ts[k4 + e][cp], Ts[k4 + e][cp + 16]);
                    x0 = __ffma2_rn(make_float2(av0[e], av0[e]), t, x0);
                    x1 = __ffma2_rn(make_float2(av1[e], av1[e]), t, x1);
                }
            }
            sm.u3.xs[r0][cp] = x0.x;
            sm.u3.xs[r0][cp + 16] = x0.y;
            sm.u3.xs[r0 + 1][cp] = x1.x;
            sm.u3.xs[r0 + 1][cp + 16] = x1.y;
            __syncthreads();
            float2 y0 = make_float2(0.f, 0.f), y1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int m4 = 0; m4 < 32; m4 += 4) {
                const float4 a0 = ld4(&Ts[32 + r0][32 + m4]), a1 = ld4(&Ts[33 + r0][32 + m4]);
                const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = make_float2(sm.u3.xs[m4 + e][cp], sm.u3.xs[m4 + e][cp + 16]);
                    y0 = __ffma2_rn(make_float2(av0[e], av0[e]), x, y0);
                    y1 = __ffma2_rn(make_float2(av1[e], av1[e]), x, y1);
                }
            }
            Ts[32 + r0][cp] = -y0.x;
            Ts[32 + r0][cp + 16] = -y0.y;
            Ts[33 + r0][cp] = -y1.x;
            Ts[33 + r0][cp + 16] = -y1.y;
        }
        __syncthreads();
        // T into its swizzled tile (over gamma, which nothing reads any more)
        for (int idx = tid; idx < C * C / 4; idx += kPrepThreads) {
            const int r = idx / (C / 4), j = (idx % (C / 4)) * 4;
            *reinterpret_cast<float4 *>(sm.u2.t + tc::sw128_off(r, j, 64)) = ld4(&Ts[r][j]);
        }
        // ---- 7. beta V^T into TMEM (thread = value row lr, tokens 32 hf ..)
        ok = __syncthreads_and(tid == 0 ? mbar_wait(&sm.bar_v, 0) : true) != 0;
        if (ok && tid == 0) {
            // [K^^T; P] (this CTA's image rows) back into u1 behind the
            // coming W^T tile, and a second copy of P behind them, for the
            // products of step 9; the inverse's scratch there has been read
            unsigned char *kp = reinterpret_cast<unsigned char *>(&sm.u1) + 128 * 64 * 2;
            mbar_arrive_expect_tx(&sm.bar_kp, 256 * 64 * 2);
            bulk_g2s(kp, img + IMG_KP, 192 * 64 * 2, &sm.bar_kp);
            bulk_g2s(kp + 192 * 128, img + IMG_KP + 128 * 128, 64 * 64 * 2, &sm.bar_kp);
        }
        kp_pend = ok;
        if (ok) {
            v_pend = false;
            mbar_try_wait(&sm.bar_v, 0);
            float bv[32];
            if constexpr (!FUSED) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int r = 32 * hf + i;
                    const float4 b4 = *reinterpret_cast<const float4 *>(&sm.beta[r]);
                    const float2 lo = __fmul2_rn(make_float2(b4.x, b4.y),
                                                 make_float2(st_bf16(qv, r, lr), st_bf16(qv, r + 1, lr)));
                    const float2 hi = __fmul2_rn(make_float2(b4.z, b4.w),
                                                 make_float2(st_bf16(qv, r + 2, lr), st_bf16(qv, r + 3, lr)));
                    bv[i] = r < L ? lo.x : 0.f;
                    bv[i + 1] = r + 1 < L ? lo.y : 0.f;
                    bv[i + 2] = r + 2 < L ? hi.x : 0.f;
                    bv[i + 3] = r + 3 < L ? hi.y : 0.f;
                }
            } else {
                // ShortConv of value channel lr on the fly (fp32), the three
                // inputs before token 32 hf from the box or the history
                const float4 w =
                    __ldg(reinterpret_cast<const float4 *>(p.conv_w) + (int64_t)h * kConvChannels + 2 * D + lr);
                float hist[3];
                if (hf == 0) {
#pragma unroll
                    for (int j = 0; j < 3; ++j) hist[j] = sm.vhist[j][lr];
                } else {
#pragma unroll
                    for (int j = 0; j < 3; ++j) hist[j] = st_bf16(qv, 29 + j, lr);
                }
                float x0 = hist[0], x1 = hist[1], x2 = hist[2];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const int r = 32 * hf + i;
                    const float x3 = st_bf16(qv, r, lr), x4 = st_bf16(qv, r + 1, lr);
                    const float2 y = __fmul2_rn(*reinterpret_cast<const float2 *>(&sm.beta[r]),
                                                conv_tap2(w, x0, x1, x2, x3, x4));
                    bv[i] = r < L ? y.x : 0.f;
                    bv[i + 1] = r + 1 < L ? y.y : 0.f;
                    x0 = x2;
                    x1 = x3;
                    x2 = x4;
                }
            }
            tc::st16(tc::lane_addr(tm, warp, PT_BV + 32 * hf), *reinterpret_cast<float(*)[16]>(&bv[0]));
            tc::st16(tc::lane_addr(tm, warp, PT_BV + 32 * hf + 16), *reinterpret_cast<float(*)[16]>(&bv[16]));
            tc::wait_st();
        } else if (tid == 0 && p.err_flag) {
            atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    if (ok) {
        // ---- W^T = (beta K~)^T T^T (thread 0) and U'^T = (beta V)^T T^T
        // (thread 32)
        if (tid == 0 || tid == 32) {
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
            const uint32_t b0 = tc::smem_u32(sm.u2.t);
            const uint32_t d = tid == 0 ? PT_WT : PT_UPT, a = tid == 0 ? PT_BK : PT_BV;
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ts(tm + d, tm + a + 8 * ks, tc::desc_tf32_kstep(b0, 64, ks), id, ks > 0);
            tc::commit(&sm.bar_mma);
        }
        mma_pend = true;
        ok = wait_mma(&sm.bar_mma, phase, p.err_flag);
        if (ok) {
            mma_pend = false;
            // ---- 8. lane lr, tokens 32 hf .. + 31: row lr of W^T into a
            // shared tile (over the inverse's scratch; the B operand of the
            // two products of step 9) and row lr of U'^T into a shared copy
            // of its image tile (over T, which the finished products have
            // read), stored by one bulk copy
            unsigned char *wt = reinterpret_cast<unsigned char *>(&sm.u1);
            unsigned char *ut = sm.u2.t;
#pragma unroll
            for (int r0 = 0; r0 < 32; r0 += 16) {
                float w16[16], u16[16];
                tc::ld16(tc::lane_addr(tm, warp, PT_WT + 32 * hf + r0), w16);
                tc::ld16(tc::lane_addr(tm, warp, PT_UPT + 32 * hf + r0), u16);
                tc::wait_ld();
#pragma unroll
                for (int q8 = 0; q8 < 16; q8 += 8) {
                    uint32_t pw[4], pu[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = w16[q8 + 2 * e], a1 = w16[q8 + 2 * e + 1];
                        const float b0 = u16[q8 + 2 * e], b1 = u16[q8 + 2 * e + 1];
                        pw[e] = pack_h2_track(a0, a1, hmax);
                        pu[e] = pack_h2_track(b0, b1, hmax);
                    }
                    const int t = 32 * hf + r0 + q8;
                    *reinterpret_cast<uint4 *>(wt + tc::sw128_off16(lr, t, 128)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    *reinterpret_cast<uint4 *>(ut + tc::sw128_off16(lr, t, 128)) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
                }
            }
        }
    }
    if (ok) {
        // ---- 9. the state-independent products of the chain step:
        // G^T = K^^T W (M = 128 key rows, N = 128 keys) and P W (M = 128:
        // P's 64 rows twice; N = 128 keys), kind::f16, K = 64 tokens.
        // [K^^T; P] came back from the image (this CTA's own writes) into
        // the shared memory behind the W^T tile by a bulk copy issued in
        // step 7, and a second copy of P behind it, so that TMEM lanes
        // 64..127 hold P W again and every warp takes part in Q'.
        unsigned char *wt = reinterpret_cast<unsigned char *>(&sm.u1);
        unsigned char *kp = wt + 128 * 64 * 2;
        static_assert(128 * 64 * 2 + 2 * 128 * 64 * 2 <= sizeof(sm.u1), "W^T and the [K^^T; P] A tiles fit u1");
        static_assert(192 * 128 * 2 <= sizeof(sm.u1) && 128 * 64 * 2 <= sizeof(sm.u2.t), "staged image tiles fit");
        fence_proxy_async_smem();  // the W^T and U'^T tiles, for the products and the bulk store
        tc::fence_before_sync();   // step 8's TMEM reads, before the products overwrite those columns
        __syncthreads();
        // the Q~ rows of the [-G^T; Q'] tile (one 8 KB run per 64-key
        // column block) into the upper half of u2, for the Q' epilogue
        unsigned char *qs = sm.u2.gam + 128 * 64 * 2;
        static_assert(2 * 128 * 64 * 2 <= sizeof(sm.u2), "U'^T and Q~ fit u2");
        if (tid == 0) {
            bulk_s2g(img + IMG_UPT, sm.u2.t, 128 * 64 * 2);
            bulk_commit();
            bulk_out = true;
            mbar_arrive_expect_tx(&sm.bar_q, 2 * C * 128);
            bulk_g2s(qs, img + IMG_BQ + 128 * 128, C * 128, &sm.bar_q);
            bulk_g2s(qs + C * 128, img + IMG_BQ + 192 * 128 + 128 * 128, C * 128, &sm.bar_q);
        }
        q_pend = true;
        ok = __syncthreads_and(tid == 0 ? mbar_wait(&sm.bar_kp, 0) : true) != 0;
        if (ok) {
            kp_pend = false;
            mbar_try_wait(&sm.bar_kp, 0);
        } else if (tid == 0 && p.err_flag) {
            atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
        }
        tc::fence_after_sync();
        if (ok && (tid == 0 || tid == 32)) {
            // G^T (thread 0, columns 0..127) and P W (thread 32, 128..255)
            constexpr uint32_t id = tc::idesc_f16(128, 128);
            const uint32_t a0 = tc::smem_u32(tid == 0 ? kp : kp + 128 * 128), bw = tc::smem_u32(wt);
            const uint32_t d = tid == 0 ? 0u : 128u;
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                tc::mma_f16_ss(tm + d, tc::desc_tf32_kstep(a0, 128, ks), tc::desc_tf32_kstep(bw, 128, ks), id, ks > 0);
            tc::commit(&sm.bar_mma);
        }
        mma_pend = ok;
        if (ok) ok = wait_mma(&sm.bar_mma, phase, p.err_flag);
        if (ok) {
            mma_pend = false;
            // [-G^T; Q'] goes to a shared copy of its image tile over u1 (the
            // products that read W^T and [K^^T; P] there are done), then out
            // by one bulk copy.
            unsigned char *bq = reinterpret_cast<unsigned char *>(&sm.u1);
            // -G^T row lr (key channel lr), keys 64 hf .. + 63
#pragma unroll
            for (int j0 = 0; j0 < 64; j0 += 16) {
                float g16[16];
                tc::ld16(tc::lane_addr(tm, warp, 64 * hf + j0), g16);
                tc::wait_ld();
#pragma unroll
                for (int q8 = 0; q8 < 16; q8 += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = g16[q8 + 2 * e], a1 = g16[q8 + 2 * e + 1];
                        w[e] = pack_h2_track(-a0, -a1, hmax);
                    }
                    *reinterpret_cast<uint4 *>(bq + tc::sw128_off16(lr, 64 * hf + j0 + q8, 192)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            // Q' = Q~ - P W: row 128 + rq of the tile; lanes 0..63 take keys
            // 0..31 of column block hf, lanes 64..127 (the second copy of
            // P W) keys 32..63 (Q~ from its staged copy: row rq of the 64-row
            // run of column block hf)
            ok = __syncthreads_and(tid == 0 ? mbar_wait(&sm.bar_q, 0) : true) != 0;
            if (ok) {
                q_pend = false;
                mbar_try_wait(&sm.bar_q, 0);
            } else if (tid == 0 && p.err_flag) {
                atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            }
            if (ok) {
                const int rq = lr & (C - 1), c32 = 32 * (lr >> 6);
#pragma unroll
                for (int j0 = c32; j0 < c32 + 32; j0 += 16) {
                    float pw16[16];
                    tc::ld16(tc::lane_addr(tm, warp, 128 + 64 * hf + j0), pw16);
                    tc::wait_ld();
#pragma unroll
                    for (int q8 = 0; q8 < 16; q8 += 8) {
                        const int u = (j0 + q8) >> 3;
                        const uint4 qt = *reinterpret_cast<const uint4 *>(qs + hf * C * 128 + rq * 128 +
                                                                          ((u ^ (rq & 7)) << 4));
                        const uint32_t qw[4] = {qt.x, qt.y, qt.z, qt.w};
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 qf = __half22float2(*reinterpret_cast<const __half2 *>(&qw[e]));
                            const float a0 = qf.x - pw16[q8 + 2 * e], a1 = qf.y - pw16[q8 + 2 * e + 1];
                            w[e] = pack_h2_track(a0, a1, hmax);
                        }
                        *reinterpret_cast<uint4 *>(bq + tc::sw128_off16(128 + rq, 64 * hf + j0 + q8, 192)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (ok && tid == 0) {
                bulk_s2g(img + IMG_BQ, bq, 192 * 128 * 2);
                bulk_commit();
            }
        }
    }
    // the staged tiles have been read out of shared memory before the CTA ends
    // (their global writes complete with the kernel)
    if (tid == 0 && bulk_out) bulk_wait_read_all();
    if (!ok && tid == 0) {
        // let every copy and product still in flight finish before the CTA
        // releases its memory
        if (in_pend) mbar_wait_drain(&sm.bar_in, 0);
        if (v_pend) mbar_wait_drain(&sm.bar_v, 0);
        if (q_pend) mbar_wait_drain(&sm.bar_q, 0);
        if (kp_pend) mbar_wait_drain(&sm.bar_kp, 0);
        if (mma_pend) mbar_wait_drain(&sm.bar_mma, phase & 1);
    }
    const bool big = !(__low2float(hmax) <= kHalfMax) || !(__high2float(hmax) <= kHalfMax);
    if (__syncthreads_or(big) && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_RANGE);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, PT_COLS);
    leave();
}

// ================================================================== chain

// One CTA per (sequence, head): 16 data warps and one issuing warp.  Value
// row i of the state is TMEM lane i; the data warps w, w + 4, w + 8, w + 12
// serve the same 32 lanes and take one quarter of the columns each.  The fp32
// state lives in the data warps' registers (thread (i, quarter q) holds
// S[i][32 q .. 32 q + 31]); its fp16 copy S16 in TMEM is the A operand of the
// one product that needs it.  With G = W^T K^ and Q' = Q~ - P W formed by
// the prep kernel, chunk c is (accumulator ACC = [D | O^T], 192 columns)
//   ACC  = U'^T [K^^T; P]^T            kind::f16, N = 192, K = 64 tokens
//   ACC += S16 [-G^T; Q']^T            kind::f16, N = 192, K = 128 keys
//   S = S diag(e^{gamma_C}) + D, S16 = fp16(S)     data warps
//   outputs = scale * O^T                          data warps
// The first product does not depend on the state: it is issued for chunk
// c + 1 while the data warps update the state of chunk c, so the serial path
// is only S16 -> the second product -> the state update -> S16.  The issuing
// warp (one thread) waits on the "S16 ready" barrier and on "accumulator
// free" barriers that the data warps arrive on, issues the products and the
// bulk copies of the operand images (two buffers; the chunk after next
// prefetched into L2; e^{gamma_C} into a ring of four with barriers of its
// own, so that an image buffer can be refilled as soon as its products are
// done and only the issuing thread ever waits on an image barrier).  The data warps observe
// the products' completion barriers themselves, one lane per warp polling,
// so no CTA-wide barrier sits in the chunk loop.  A full chunk's outputs
// leave through a shared tile and one TMA tensor store.
constexpr int kDataWarps = 16;
constexpr int kDataThreads = 32 * kDataWarps;
constexpr int kChainThreads = kDataThreads + 32;  // + the issuing warp
constexpr uint32_t CT_ACC = 0;      // accumulators [D (128) | O^T (64)] at columns 0 and 256
constexpr uint32_t CT_ACC_STRIDE = 256;
constexpr uint32_t CT_S16 = 448;    // fp16 state, two per column: 64 columns
constexpr uint32_t CT_COLS = 512;
constexpr uint32_t kAccN = 192;
static_assert(IMG_TILES % 1024 == 0, "image buffers stay 1024-aligned");

struct ChainSmem {
    unsigned char img[2][IMG_TILES];  // a chunk's operand tiles, as laid out in the workspace
    unsigned char ot[2][C * D * 2];   // a full chunk's outputs [64 tokens][128 value rows], for the TMA store
    float egc[4][D];                  // e^{gamma_C} of chunk c in egc[c & 3]
    uint64_t full[2];                 // chunk images landed
    uint64_t egc_full[4];             // e^{gamma_C} of chunk c landed in egc[c & 3]
    uint64_t acc_done[2];             // both products of the chunk using this accumulator done
    uint64_t acc_free[2];             // the data warps have read this accumulator (one arrival per data warp)
    uint64_t s16_ready;               // S16 written (one arrival per data warp)
    uint64_t tile_full;               // an output tile written (one arrival per data warp)
    uint64_t tile_free[2];            // an output tile's tensor store has read it (thread 0)
    uint32_t tmem_base;
};
constexpr size_t kChainSmem = sizeof(ChainSmem) + 1024;

// One lane of the warp polls `bar` (bounded); on success every lane observes
// the completed phase itself.  Warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    bool okw = true;
    if ((threadIdx.x & 31) == 0) okw = mbar_wait(bar, parity);
    okw = __shfl_sync(0xffffffffu, okw ? 1 : 0, 0) != 0;
    if (okw) mbar_try_wait(bar, parity);
    tc::fence_after_sync();
    return okw;
}

// The data warp's hand-off: its TMEM accesses are complete and ordered
// before lane 0's arrival.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

template <typename T, bool FUSED>
__global__ void __launch_bounds__(kChainThreads, 1) chain_kernel(const PrefillParams p,
                                                                  const __grid_constant__ CUtensorMap omap,
                                                                  const int seg_lo, const int seg_hi) {
    // the next segment's prep kernel may start beside this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ unsigned char smem_raw[];
    ChainSmem &sm =
        *reinterpret_cast<ChainSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t *plan = static_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    if (plan[n + 1] == 0) return;
    const int s = blockIdx.x, h = blockIdx.y, H = p.H;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t cs = p.cu_seqlens[s], ce = p.cu_seqlens[s + 1];
    const int slot = p.slot_ids[s];
    T *out = static_cast<T *>(p.out);
    const int64_t tok_stride = (int64_t)H * D, hoff = (int64_t)h * D;
    // this launch walks the sequence's local chunks [c_lo, c_hi); a later
    // segment starts from the state the previous one wrote to the pool
    const int nchunks_all = plan[s + 1] - plan[s];
    const int c_lo = seg_lo, c_hi = seg_hi < nchunks_all ? seg_hi : nchunks_all;
    if (seg_lo > 0 && c_lo >= c_hi) return;
    const int nchunks = c_hi > c_lo ? c_hi - c_lo : 0;  // chunks of this launch; loop index i is c_lo + i
    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        const int64_t t_end = seg_hi < nchunks_all ? (int64_t)cs + (int64_t)c_hi * C : (int64_t)ce;
        for (int64_t t = cs + (int64_t)c_lo * C + (tid >> 7); t < t_end; t += kChainThreads / D)
            Elem<T>::store1(out + t * tok_stride + hoff + (tid & 127), 0.f);
        if (slot >= 0 && seg_lo == 0 && h == 0 && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    const unsigned char *ws = static_cast<const unsigned char *>(p.workspace) + plan_bytes(n);
    auto image = [&](int ci) { return ws + ((size_t)(plan[s] + c_lo + ci) * H + h) * (size_t)IMG_BYTES; };
    // checked build: this launch's operand images (its last one ends highest),
    // the sequence's tokens, the slot's state and conv state
    if ((nchunks > 0 && !in_bounds((int64_t)(plan_bytes(n) + ((size_t)(plan[s] + c_lo + nchunks - 1) * H + h) *
                                                             (size_t)IMG_BYTES),
                                   IMG_BYTES, (int64_t)p.workspace_bytes, p.err_flag)) ||
        !in_bounds(cs, (int64_t)ce - cs, p.total_tokens, p.err_flag) ||
        !in_bounds(((int64_t)slot * H + h) * D * D, D * D, p.num_slots * H * (int64_t)(D * D), p.err_flag) ||
        (FUSED && !in_bounds(((int64_t)slot * H + h) * 3 * kConvChannels, 3 * kConvChannels,
                             p.num_slots * H * (int64_t)(3 * kConvChannels), p.err_flag)))
        return;

    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, CT_COLS);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.full[b], 1);
            mbar_init(&sm.acc_done[b], 1);
            mbar_init(&sm.acc_free[b], kDataWarps);
            mbar_init(&sm.tile_free[b], 1);
        }
        for (int r = 0; r < 4; ++r) mbar_init(&sm.egc_full[r], 1);
        mbar_init(&sm.s16_ready, kDataWarps);
        mbar_init(&sm.tile_full, kDataWarps);
        fence_barrier_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem_base;
    bool ok = true;
    float *Sg = nullptr;
    float S[32];

    if (warp == kDataWarps) {
        // ================= issuing warp (lane 0)
        if ((tid & 31) == 0) {
            int last_issue[2] = {-1, -1}, last_egc[4] = {-1, -1, -1, -1};
            int ndone[2] = {0, 0};  // commits on acc_done[b]
            int open_b = -1;        // an accumulator with products issued after its last commit
            auto issue = [&](int ci) {
                const int b = ci & 1;
                mbar_arrive_expect_tx(&sm.full[b], IMG_TILES);
                bulk_g2s(sm.img[b], image(ci), IMG_TILES, &sm.full[b]);
                mbar_arrive_expect_tx(&sm.egc_full[ci & 3], D * 4);
                bulk_g2s(sm.egc[ci & 3], image(ci) + IMG_EGC, D * 4, &sm.egc_full[ci & 3]);
                last_issue[b] = ci;
                last_egc[ci & 3] = ci;
                if (ci + 2 < nchunks) bulk_prefetch_l2(image(ci + 2), IMG_BYTES);
            };
            constexpr uint32_t id = tc::idesc_f16(128, kAccN);
            // ACC[b] = U'^T [K^^T; P]^T (chunk ci's image in buffer b = ci & 1)
            auto mma_u = [&](int ci) {
                const int b = ci & 1;
                const uint32_t a0 = tc::smem_u32(sm.img[b] + IMG_UPT), b0 = tc::smem_u32(sm.img[b] + IMG_KP);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    tc::mma_f16_ss(tm + CT_ACC + b * CT_ACC_STRIDE, tc::desc_tf32_kstep(a0, 128, ks),
                                   tc::desc_tf32_kstep(b0, 192, ks), id, ks > 0);
                open_b = b;
            };
            // ACC[b] += S16 [-G^T; Q']^T, then the commit that releases both
            auto mma_s = [&](int ci) {
                const int b = ci & 1;
                const uint32_t b0 = tc::smem_u32(sm.img[b] + IMG_BQ);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_f16_ts(tm + CT_ACC + b * CT_ACC_STRIDE, tm + CT_S16 + 8 * ks,
                                   tc::desc_tf32_kstep(b0, 192, ks), id, 1);
                tc::commit(&sm.acc_done[b]);
                ++ndone[b];
                open_b = -1;
            };
            if (nchunks > 0) issue(0);
            if (nchunks > 1) issue(1);
            if (nchunks > 0) {
                ok = mbar_wait(&sm.full[0], 0);
                if (ok) {
                    tc::fence_after_sync();
                    mma_u(0);
                    ok = mbar_wait(&sm.s16_ready, 0);
                }
            }
            for (int c = 0; c < nchunks && ok; ++c) {
                const int b = c & 1;
                // ---- the serial product of chunk c (S16 of chunk c is ready)
                tc::fence_after_sync();
                mma_s(c);
                // ---- the state-independent product of chunk c + 1: its image
                // has landed and the data warps have read chunk c - 1's
                // accumulator, which it reuses
                if (c + 1 < nchunks) {
                    ok = mbar_wait(&sm.full[b ^ 1], ((c + 1) >> 1) & 1) &&
                         (c == 0 || mbar_wait(&sm.acc_free[b ^ 1], ((c - 1) >> 1) & 1));
                    if (!ok) break;
                    tc::fence_after_sync();
                    mma_u(c + 1);
                }
                // ---- chunk c's products have read image buffer b: refill it
                if (c + 2 < nchunks) {
                    ok = mbar_wait(&sm.acc_done[b], (c >> 1) & 1);
                    if (!ok) break;
                    issue(c + 2);
                }
                if (c + 1 < nchunks) ok = mbar_wait(&sm.s16_ready, (c + 1) & 1);
            }
            if (!ok && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            // no product or copy may still be writing when the CTA releases its
            // memory: products issued after the last commit get one of their
            // own, then the last commit of each barrier and the last copy into
            // each buffer are waited for (a phase already complete passes at once)
            if (open_b >= 0) {
                tc::commit(&sm.acc_done[open_b]);
                ++ndone[open_b];
            }
            for (int b = 0; b < 2; ++b) {
                if (ndone[b] > 0) mbar_wait_drain(&sm.acc_done[b], (ndone[b] - 1) & 1);
                if (last_issue[b] >= 0) mbar_wait_drain(&sm.full[b], (last_issue[b] >> 1) & 1);
            }
            for (int r = 0; r < 4; ++r)
                if (last_egc[r] >= 0) mbar_wait_drain(&sm.egc_full[r], (last_egc[r] >> 2) & 1);
        }
    } else {
        // ================= data warps
        const int lr = ((warp & 3) << 5) | (tid & 31);  // value row = TMEM lane
        const int cq = warp >> 2;                        // quarter of the columns this thread takes
        auto taddr = [&](uint32_t col) { return tc::lane_addr(tm, warp, (int)col); };
        __half2 s16max = __float2half2_rn(0.f);  // running max of |S16|: inf or NaN once S16 overflowed
        Sg = p.pool + ((int64_t)slot * H + h) * (int64_t)D * D + (int64_t)lr * D + cq * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 v4 = (p.init_from_pool || seg_lo > 0) ? *reinterpret_cast<const float4 *>(Sg + e)
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
            S[e] = v4.x; S[e + 1] = v4.y; S[e + 2] = v4.z; S[e + 3] = v4.w;
        }
        auto store_s16 = [&](uint32_t (&w)[16]) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const __half2 h2 = __floats2half2_rn(S[2 * e], S[2 * e + 1]);
                w[e] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            tc::st16u(taddr(CT_S16 + cq * 16), w);
        };
        // the range check of S16, once it has been handed over
        auto track_s16 = [&](const uint32_t (&w)[16]) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
                s16max = __hmax2_nan(s16max, __habs2(*reinterpret_cast<const __half2 *>(&w[e])));
        };
        // outputs of chunk cj (tokens cq * 16 .. + 15 of value row lr), read
        // from its accumulator (complete: acc_done was observed): a full
        // chunk through its tile and one tensor store, a partial one straight
        // to global memory.  Tile hand-offs go through mbarriers (bounded
        // waits): the data warps arrive on tile_full once their part is
        // written, thread 0 then issues the store and, once the previous
        // store has read its tile, arrives on that tile's tile_free.
        constexpr bool fused = FUSED;
        auto output = [&](int cj) {
            const int64_t tj = (int64_t)cs + (int64_t)(c_lo + cj) * C;
            const int Lj = (int)((int64_t)ce - tj < C ? (int64_t)ce - tj : C);
            float o[16];
            tc::ld16(taddr(CT_ACC + (cj & 1) * CT_ACC_STRIDE + 128 + cq * 16), o);
            tc::wait_ld();
            warp_arrive(&sm.acc_free[cj & 1]);  // the accumulator has been read
#pragma unroll
            for (int r = 0; r < 16; ++r) o[r] = p.scale * o[r];
            if (Lj == C) {
                const int t = cj & 1, use = cj >> 1;  // the tile and its use count
                if (use > 0 && !warp_wait(&sm.tile_free[t], (use - 1) & 1)) return false;
                T *tile = reinterpret_cast<T *>(sm.ot[t]) + (cq * 16) * D + lr;
#pragma unroll
                for (int r = 0; r < 16; ++r) Elem<T>::store1(tile + r * D, o[r]);
                fence_proxy_async_smem();
                __syncwarp();
                if ((tid & 31) == 0) mbar_arrive(&sm.tile_full);
                if (warp == 0) {
                    bool stored = true;
                    if (tid == 0) {
                        stored = mbar_wait(&sm.tile_full, cj & 1);
                        if (stored) {
                            tma_store_2d(&omap, h * D, (int)tj, sm.ot[t]);
                            bulk_commit();
                            if (cj > 0) {
                                bulk_wait_read_le1();
                                mbar_arrive(&sm.tile_free[t ^ 1]);
                            }
                        }
                    }
                    if (__shfl_sync(0xffffffffu, stored ? 1 : 0, 0) == 0) return false;  // warp-uniform
                }
            } else {
                T *dst = out + (tj + cq * 16) * tok_stride + hoff + lr;
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    if (cq * 16 + r < Lj) Elem<T>::store1(dst + (int64_t)r * tok_stride, o[r]);
            }
            return true;
        };
        {
            uint32_t w[16];
            store_s16(w);
            warp_arrive(&sm.s16_ready);
            track_s16(w);
        }
        // snapshot requests of this sequence (the same for every thread)
        int snap_ptr = 0, snap_hi = 0;
        bool snap_bad = false;
        if (p.num_snaps > 0) {
            snap_range(p, s, snap_ptr, snap_hi);
            // requests up to this segment's first chunk were an earlier launch's
            if (seg_lo > 0)
                while (snap_ptr < snap_hi && (int64_t)p.snap_tokens[snap_ptr] <= (int64_t)c_lo * C) ++snap_ptr;
        }
        auto store_snapshot = [&](int sl) {
            float *dst = p.pool + ((int64_t)sl * H + h) * (int64_t)D * D + (int64_t)lr * D + cq * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(dst + e) = make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
        };
        for (int c = 0; c < nchunks && ok; ++c) {
            const int b = c & 1;
            // ---- S = S diag(e^{gamma_C}) + D, and its fp16 copy (each warp
            // observes the barrier of chunk c's e^{gamma_C} before reading it;
            // its slot is refilled only after every data warp has handed
            // over S16 of chunk c + 1)
            ok = warp_wait(&sm.acc_done[b], (c >> 1) & 1) && warp_wait(&sm.egc_full[c & 3], (c >> 2) & 1);
            if (!ok) break;
            uint32_t w[16];
            {
                float d[32];
                tc::ld32(taddr(CT_ACC + b * CT_ACC_STRIDE + cq * 32), d);
                const float4 *e4 = reinterpret_cast<const float4 *>(sm.egc[c & 3]) + cq * 8;
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 g4 = e4[j];
                    const float2 lo = __ffma2_rn(make_float2(S[4 * j], S[4 * j + 1]), make_float2(g4.x, g4.y),
                                                 make_float2(d[4 * j], d[4 * j + 1]));
                    const float2 hi = __ffma2_rn(make_float2(S[4 * j + 2], S[4 * j + 3]), make_float2(g4.z, g4.w),
                                                 make_float2(d[4 * j + 2], d[4 * j + 3]));
                    S[4 * j] = lo.x; S[4 * j + 1] = lo.y; S[4 * j + 2] = hi.x; S[4 * j + 3] = hi.y;
                }
                store_s16(w);
            }
            warp_arrive(&sm.s16_ready);
            track_s16(w);
            // ---- chunk c's outputs, off the serial path
            ok = output(c);
            if (!ok) break;
            // the state after c + 1 chunks, where a snapshot asks for it
            if (snap_ptr < snap_hi)
                snap_ptr = snap_due(p, snap_ptr, snap_hi, min((int64_t)(c_lo + c + 1) * C, (int64_t)ce - cs), C,
                                    snap_bad, store_snapshot);
        }
        // requests past the sequence's last whole chunk can never be met
        if (ok && snap_ptr < snap_hi && c_hi == nchunks_all) snap_bad = true;
        if (fused && c_hi == nchunks_all) {
            // the slot's conv state: the last three raw inputs of the
            // sequence, preceded by its old history (or zeros) when the
            // sequence is shorter; the prep kernel read the old one before
            // this launch (the first chunk's segment runs first)
            const int Ls = ce - cs;
            T *cst = static_cast<T *>(p.conv_state) + ((int64_t)slot * H + h) * (3 * kConvChannels);
            for (int ch = tid; ch < kConvChannels; ch += kDataThreads) {
                const T *src = ch < D ? static_cast<const T *>(p.q) : ch < 2 * D ? static_cast<const T *>(p.k)
                                                                               : static_cast<const T *>(p.v);
                const int c = ch % D;
                T old[3], nv[3];
#pragma unroll
                for (int j = 0; j < 3; ++j) old[j] = p.init_from_pool ? cst[j * kConvChannels + ch] : T(0.f);
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int pos = Ls - 3 + j;
                    nv[j] = pos >= 0 ? src[((int64_t)cs + pos) * tok_stride + hoff + c] : old[3 + pos];
                }
#pragma unroll
                for (int j = 0; j < 3; ++j) cst[j * kConvChannels + ch] = nv[j];
            }
        }
        if (snap_bad && h == 0 && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SNAPSHOT);
        if (tid == 0) bulk_wait_all();  // every tensor store complete before shared memory goes
        const bool bad = !(__low2float(s16max) <= kHalfMax) || !(__high2float(s16max) <= kHalfMax);
        if (bad && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_RANGE);
        if (!ok && (tid & 31) == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
    }
    // the final state, only when every warp finished its loop
    const bool all_ok = __syncthreads_and(ok) != 0;
    if (all_ok && warp < kDataWarps) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(Sg + e) = make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, CT_COLS);
}

// The fused prefill's output side: out = o / sqrt(mean(o^2) + eps_o) * norm_w
// * sigmoid(z) per (token, head), in place over the chain's outputs.  One
// warp per (token, head), four values per lane; the sum of squares is a
// butterfly over the warp (the same bits on every lane).  Padding sequences'
// zero outputs stay zero.
constexpr int kGateWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kGateWarps * 32) norm_gate_kernel(const PrefillParams p) {
    const int64_t row = (int64_t)blockIdx.x * kGateWarps + (threadIdx.x >> 5);  // token x head
    if (row >= p.total_tokens * p.H) return;
    const int lane = threadIdx.x & 31;
    T *o = static_cast<T *>(p.out) + row * D + 4 * lane;
    const T *z = static_cast<const T *>(p.z) + row * D + 4 * lane;
    static_assert(sizeof(T) == 2, "four 16-bit values per 8-byte access");
    const uint2 ov = *reinterpret_cast<const uint2 *>(o), zv = *reinterpret_cast<const uint2 *>(z);
    const T *oe = reinterpret_cast<const T *>(&ov), *ze = reinterpret_cast<const T *>(&zv);
    float x[4], zz[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[e] = Elem<T>::to_f(oe[e]);
        zz[e] = Elem<T>::to_f(ze[e]);
    }
    const float4 w = __ldg(reinterpret_cast<const float4 *>(p.norm_w) + lane);
    float ss = __fmaf_rn(x[3], x[3], __fmaf_rn(x[2], x[2], __fmaf_rn(x[1], x[1], __fmul_rn(x[0], x[0]))));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, m));
    const float inv = rsqrtf(__fadd_rn(__fmul_rn(ss, 1.0f / D), p.eps_o));
    const float wv[4] = {w.x, w.y, w.z, w.w};
    T y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = T(__fmul_rn(__fmul_rn(__fmul_rn(x[e], inv), wv[e]), sigmoid_gate(zz[e])));
    *reinterpret_cast<uint2 *>(o) = *reinterpret_cast<const uint2 *>(y);
}

}  // namespace prefill_tc

#ifndef KDA_PREFILL_TC
#define KDA_PREFILL_TC 1
#endif

bool prefill_tc_supported(int dk, int dv, int dtype) {
    return KDA_PREFILL_TC && dtype == KDA_DT_BF16 && dk == 128 && dv == 128 && tensor_map_encode_fn() != nullptr;
}

size_t prefill_tc_workspace_bytes(int H, int32_t num_seqs, int64_t total_tokens) {
    using namespace prefill_tc;
    return plan_bytes(num_seqs) + (size_t)max_chunks(num_seqs, total_tokens) * (size_t)H * IMG_BYTES;
}

// Segments of a pipelined prefill (see launch_tc).  Segment k + 1's prep
// runs on the SMs that segment k's chains leave free and should take about
// as long as those chains, so segment lengths form a geometric series of
// ratio rho = (a chain step) / (a chunk's prep for every chain on the free
// SMs).  A prep CTA lives about 12 chain steps at two CTAs per SM, so
// rho = kSegRatioScale x free SMs / chains (0.6 at 32 chains; below 1 the
// segments shrink, above it they grow).  Segments hold at least
// max(16, chunks / 50) chunks and 256 prep CTAs.  Measured at 32 heads,
// against equal segments: 8192 tokens 65 / 39 / 24 chunks, 438.7 us against
// 444.6 us; 102 400 tokens six segments from 671 chunks down to 52, 4.22 ms
// against 4.44 ms (the minimum of 16 chunks there: 4.27 ms).
constexpr double kSegRatioScale = 0.16;
constexpr int kMaxSegments = 64;

// Local chunk indices where segments start (lo[0] = 0); returns the segment
// count (1: no pipelining).  chains = sequences x heads; per_seq = mean
// chunks per sequence.
static int plan_segments(int64_t chains, int sms, int64_t per_seq, int (&lo)[kMaxSegments + 1]) {
    lo[0] = 0;
    if (chains <= 0 || chains >= sms || per_seq < 2) return 1;
    const double rho = kSegRatioScale * (double)(sms - chains) / (double)chains;
    const double P = (double)per_seq;
    double m = per_seq / 50 > 16 ? (double)(per_seq / 50) : 16.0;
    if ((double)((256 + chains - 1) / chains) > m) m = (double)((256 + chains - 1) / chains);
    auto first = [&](int k) {  // first length of k segments summing to P
        return std::fabs(rho - 1.0) < 1e-9 ? P / k : P * (1.0 - rho) / (1.0 - std::pow(rho, k));
    };
    int K = 1;
    for (int k = 2; k <= kMaxSegments; ++k) {
        const double n0 = first(k), nl = n0 * std::pow(rho, k - 1);
        if ((n0 < nl ? n0 : nl) >= m) K = k; else break;
    }
    const double n0 = first(K);
    double acc = 0.0;
    for (int k = 1; k < K; ++k) {
        acc += n0 * std::pow(rho, k - 1);
        lo[k] = (int)(acc + 0.5);
    }
    return K;
}

template <bool FUSED>
static cudaError_t launch_tc(const PrefillParams &p, cudaStream_t st) {
    using namespace prefill_tc;
    cudaError_t e = cudaFuncSetAttribute(prep_tc_kernel<__nv_bfloat16, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chain_kernel<__nv_bfloat16, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kChainSmem);
    if (e != cudaSuccess) return e;
    const int64_t mc = max_chunks(p.num_seqs, p.total_tokens);
    // the token inputs as [total_tokens][H * 128] tensors, boxes of 64
    // tokens x 64 channels (bf16) or 32 channels (g, fp32), 128B-swizzled
    CUtensorMap kmap, qmap, vmap, gmap;
    const bool any = mc > 0 && p.total_tokens > 0;
    if (any) {
        const cuuint64_t dims[2] = {(cuuint64_t)p.H * D, (cuuint64_t)p.total_tokens};
        const cuuint64_t sb[1] = {(cuuint64_t)p.H * D * 2}, sf[1] = {(cuuint64_t)p.H * D * 4};
        const cuuint32_t boxb[2] = {64, (cuuint32_t)C}, boxf[2] = {32, (cuuint32_t)C};
        const cuuint32_t elem[2] = {1, 1};
        const void *srcs[3] = {p.k, p.q, p.v};
        CUtensorMap *maps[3] = {&kmap, &qmap, &vmap};
        for (int i = 0; i < 3; ++i)
            if (tensor_map_encode_fn()(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(srcs[i]), dims,
                                       sb, boxb, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        if (tensor_map_encode_fn()(&gmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p.g), dims, sf, boxf,
                                   elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // the output tensor as [total_tokens][H * 128] bf16, boxes of 64 tokens x
    // one head's 128 values (the chain's full-chunk tensor stores)
    CUtensorMap omap;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.H * D, (cuuint64_t)(p.total_tokens > 0 ? p.total_tokens : 1)};
        const cuuint64_t strides[1] = {(cuuint64_t)p.H * D * 2};
        const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)C};
        const cuuint32_t elem[2] = {1, 1};
        const CUresult r = tensor_map_encode_fn()(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, dims, strides,
                                                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // Pipelining: when few (sequence, head) chains would walk many chunks
    // each, the chunks are cut into segments (plan_segments).  Segment k's
    // prep runs beside segment k - 1's chain (programmatic dependent launch:
    // the chain lets it start at once; one of its CTAs waits for that chain
    // before the grid ends), and segment k's chain, an ordinary launch,
    // follows its prep and so the previous chain.  The last segment takes
    // every remaining chunk.  Only the last chain is exposed.
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        sms = 1;
    int lo_k[kMaxSegments + 1];
    const int64_t per_seq = p.num_seqs > 0 ? (p.total_tokens + C - 1) / C / p.num_seqs : 0;
    const int nseg = any && p.num_seqs > 0 ? plan_segments((int64_t)p.num_seqs * p.H, sms, per_seq, lo_k) : 1;
    lo_k[0] = 0;
    const dim3 cgrid((unsigned)p.num_seqs, (unsigned)p.H);
    for (int k = 0; k < nseg; ++k) {
        const bool last = k == nseg - 1;
        const int lo = lo_k[k];
        const int len = last ? 0 : lo_k[k + 1] - lo_k[k];
        if (any) {
            const int seg_len = last ? 0 : len;
            const int64_t gx = last ? mc : (int64_t)p.num_seqs * len;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)gx, (unsigned)p.H);
            cfg.blockDim = dim3(kPrepThreads);
            cfg.dynamicSmemBytes = kPrepSmem;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = k > 0 ? 1 : 0;
            const PrefillParams pp = p;
            e = cudaLaunchKernelEx(&cfg, prep_tc_kernel<__nv_bfloat16, FUSED>, pp, kmap, qmap, vmap, gmap, lo, seg_len,
                                   k > 0 ? 1 : 0);
            if (e != cudaSuccess) return e;
        }
        chain_kernel<__nv_bfloat16, FUSED><<<cgrid, kChainThreads, kChainSmem, st>>>(p, omap, lo,
                                                                             last ? INT_MAX : lo + len);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (FUSED && p.total_tokens > 0) {
        const int64_t rows = p.total_tokens * p.H;
        norm_gate_kernel<__nv_bfloat16>
            <<<(unsigned)((rows + kGateWarps - 1) / kGateWarps), kGateWarps * 32, 0, st>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t st) {
    return p.conv_w != nullptr ? launch_tc<true>(p, st) : launch_tc<false>(p, st);
}

}  // namespace kda
