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
// Two kernels, both on tcgen05 (kind::tf32, fp32 accumulate):
//
// prep_tc_kernel  one CTA per (chunk, head), all chunks of all sequences in
//   parallel over the whole GPU.  Computes everything that does not depend on
//   the state and writes, per (chunk, head), an operand image that the chain
//   kernel copies into shared memory with one bulk copy:
//     [W; Q~] (128 x 128), P (64 x 64), K^^T (128 x 64) as K-major 128B-swizzled
//     tf32 tiles, e^{gamma_C} (128) and U' (64 x 128, plain fp32).
// chain_tc_kernel  one CTA per (sequence, head, block of 32 value rows) walks
//   the chunks in order; rows of the state are independent, so four CTAs
//   share a head.  The rows sit on the N side of the products and the state
//   block is a swizzled tile in shared memory (the B operand).  The operand
//   images of the next chunk are in flight (bulk copies) while a chunk computes.
//
// Decay factors in the A/P product: with ref = gamma at token 31 of the chunk,
// K+ = k^ e^{gamma-ref}, Q+ = q^ e^{gamma-ref}, K- = k^ e^{ref-gamma}, so that
// [K+; Q+] K-^T carries e^{gamma_r - gamma_j}.  A chunk whose gamma spans more
// than 80 (natural units) around ref on some channel would overflow these
// factors; that chunk computes A and P with one exp per (r, j, c) instead.
#include <stdint.h>

#include "kda.h"
#include "kda_bulk.cuh"
#include "kda_internal.h"
#include "kda_rowmath.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace prefill_tc {

constexpr int C = 64;   // chunk length
constexpr int D = 128;  // dk = dv
constexpr int kThreads = 256;  // chain CTA
constexpr float kSpanLimit = 80.f;

// Operand image of one (chunk, head) in the workspace (bytes).
constexpr uint32_t IMG_BW = 0;                         // [W; Q~]  128 rows x K 128
constexpr uint32_t IMG_P = IMG_BW + 128 * 128 * 4;     // P        64 rows x K 64
constexpr uint32_t IMG_KT = IMG_P + 64 * 64 * 4;       // K^^T     128 rows x K 64
constexpr uint32_t IMG_TILES = IMG_KT + 128 * 64 * 4;  // = 112 KiB, one bulk copy
constexpr uint32_t IMG_EGC = IMG_TILES;                // e^{gamma_C}, 128 fp32
constexpr uint32_t IMG_UP = IMG_EGC + 1024;            // U' plain [64 tokens][128 value rows] fp32
constexpr uint32_t IMG_BYTES = IMG_UP + 64 * 128 * 4;

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t plan_bytes(int32_t num_seqs) {
    return round_up(sizeof(int32_t) * ((size_t)num_seqs + 2), 1024);
}
__host__ __device__ inline int64_t max_chunks(int32_t num_seqs, int64_t total_tokens) {
    return (total_tokens + C - 1) / C + num_seqs;
}

__device__ __forceinline__ void st_sw(unsigned char *tile, int rows, int row, int k, float x) {
    *reinterpret_cast<float *>(tile + tc::sw128_off(row, k, rows)) = x;
}

__device__ __forceinline__ void sync_for_mma() {
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Bounded wait on an MMA-completion barrier; the result is made uniform across
// the CTA and a timeout is recorded in the error flag.  `phase` advances only
// when the wait succeeded, so after a timeout it still names the pending
// phase, which is the one a drain must wait for.
__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase, int32_t *err_flag) {
    const bool mine = mbar_wait(bar, phase & 1);
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

// TMEM columns of the prep kernel (256 per CTA, so two CTAs share an SM):
// W^T is written over G once G has been read.
constexpr int PT_BKT = 0, PT_BVT = 64, PT_G = 128, PT_WT = 128, PT_UPT = 192;
constexpr uint32_t PT_COLS = 256;

// 8 warps: thread (warp w, lane) owns key channel c = 32 (w & 3) + lane, which
// is also its TMEM lane and its row of the value-side tiles, for the token
// half 32 (w >> 2) .. 32 (w >> 2) + 31.
constexpr int kPrepThreads = 256;

// Scratch of the UT inverse, laid over the [K+; Q+] tile once the A/P
// product that reads it has completed.
struct InvScratch {
    float As[C][C + 1];
    float Ts[C][C + 1];
};

struct PrepSmem {
    union {
        unsigned char bufKQ[128 * 128 * 4];  // [K+; Q+]  (A of the A/P product)
        InvScratch inv;
    };
    union {
        unsigned char bufKM[64 * 128 * 4];   // K-        (B of the A/P product)
        unsigned char bufT[64 * 64 * 4];     // T         (B of the WY products)
    };
    float invk[C], invq[C], beta[C];
    float nrm[2][2 * C];  // sums of squares over each channel half: rows k_0..k_63, q_0..q_63
    float ref[D];         // gamma at token 31
    float gC[D];          // gamma at the chunk's last token
    float egcref[D];      // e^{gamma_C - ref}
    float xs[32][33];     // partial products of the UT inverse
    uint64_t bar;
    uint32_t tmem_base;
};
constexpr size_t kPrepSmem = sizeof(PrepSmem) + 1024;
static_assert(sizeof(InvScratch) <= 128 * 128 * 4, "inverse scratch must fit the [K+; Q+] tile");

template <typename T>
__global__ void __launch_bounds__(kPrepThreads, 2) prep_tc_kernel(const PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    PrepSmem &sm =
        *reinterpret_cast<PrepSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t *plan = static_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    if (plan[n + 1] == 0) return;
    const int32_t chunk = blockIdx.x;
    if (chunk >= plan[n]) return;
    const int h = blockIdx.y, H = p.H;
    const int s = find_seq(plan, n, chunk);
    const int slot = p.slot_ids[s];
    if (slot < 0 || (int64_t)slot >= p.num_slots) return;  // the chain writes zeros
    const int64_t t0 = (int64_t)p.cu_seqlens[s] + (int64_t)(chunk - plan[s]) * C;
    const int L = (int)((int64_t)p.cu_seqlens[s + 1] - t0 < C ? (int64_t)p.cu_seqlens[s + 1] - t0 : C);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = ((warp & 3) << 5) | lane;  // key channel = TMEM lane
    const int rb = 32 * (warp >> 2);          // first token of this thread's half
    const T *__restrict__ q = static_cast<const T *>(p.q);
    const T *__restrict__ k = static_cast<const T *>(p.k);
    const T *__restrict__ v = static_cast<const T *>(p.v);
    const T *__restrict__ bb = static_cast<const T *>(p.b);
    const float *__restrict__ gptr = p.g;
    const int64_t tok_stride = (int64_t)H * D, hoff = (int64_t)h * D;
    unsigned char *__restrict__ img = static_cast<unsigned char *>(p.workspace) + plan_bytes(n) +
                                      ((size_t)chunk * H + h) * (size_t)IMG_BYTES;

    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, PT_COLS);
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_barrier_init();
    }

    // this channel's gates over its token half, in flight during the norms
    float gh[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) gh[r] = (rb + r < L) ? __ldg(gptr + (t0 + rb + r) * tok_stride + hoff + c) : 0.f;

    // ---- 1a. sums of squares: thread = (row of k or q, half of the channels);
    // the loop is unrolled so that the row is in flight at once
    {
        const int row = tid & (2 * C - 1), ch = tid >> 7;
        const int r = row & (C - 1);
        float ss = 0.f;
        if (r < L) {
            const T *src = (row >= C ? q : k) + (t0 + r) * tok_stride + hoff + 64 * ch;
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                const float4 x = Elem<T>::load4(src + j);
                ss = fmaf(x.x, x.x, ss);
                ss = fmaf(x.y, x.y, ss);
                ss = fmaf(x.z, x.z, ss);
                ss = fmaf(x.w, x.w, ss);
            }
        }
        sm.nrm[ch][row] = ss;
    }
    // ---- 1b. gamma (thread = key channel c): the first half's running sum
    // ends at ref = gamma_31; the second half continues it from there.  Rows
    // past the chunk's end repeat gamma_C.
    float acc = 0.f, gmin = 0.f, gmax = 0.f, gC = 0.f;
    if (rb == 0) {
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            acc += gh[r];
            if (r == L - 1) gC = acc;
            gmin = r == 0 ? acc : fminf(gmin, acc);
            gmax = r == 0 ? acc : fmaxf(gmax, acc);
        }
        sm.ref[c] = acc;
        if (L <= 32) sm.gC[c] = gC;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid < 2 * C) {
        const int r = tid & (C - 1);
        const float inv = (r < L) ? rsqrtf(sm.nrm[0][tid] + sm.nrm[1][tid] + p.eps) : 0.f;
        if (tid >= C) {
            sm.invq[r] = inv;
        } else {
            sm.invk[r] = inv;
            sm.beta[r] = (r < L) ? sigmoid_f(Elem<T>::load1(bb + (t0 + r) * H + h)) : 0.f;
        }
    }
    const float ref = sm.ref[c];
    if (rb == 32) {
        acc = ref;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            acc += gh[r];
            if (32 + r == L - 1) gC = acc;
            gmin = r == 0 ? acc : fminf(gmin, acc);
            gmax = r == 0 ? acc : fmaxf(gmax, acc);
        }
        if (L > 32) sm.gC[c] = gC;
    }
    const float span = fmaxf(gmax - ref, ref - gmin);
    const bool unsafe = __syncthreads_or(span > kSpanLimit) != 0;
    gC = sm.gC[c];
    if (rb == 0) {
        reinterpret_cast<float *>(img + IMG_EGC)[c] = expf(gC);
        sm.egcref[c] = expf(gC - ref);
    }
    const uint32_t tm = sm.tmem_base;
    uint32_t phase = 0;

    // ---- 2. this thread's 32 tokens, 8 at a time; the next block's loads are
    // in flight while the current block computes
    {
        const float eref = expf(ref);
        acc = rb == 0 ? 0.f : ref;
        float kb[8], qb[8], vb[8], gb[8];
        auto load_block = [&](int r0, float (&kk)[8], float (&qq)[8], float (&vv)[8], float (&gg)[8]) {
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const bool ok_r = rb + r0 + rr < L;
                const int64_t off = (t0 + rb + r0 + rr) * tok_stride + hoff + c;
                kk[rr] = ok_r ? Elem<T>::load1(k + off) : 0.f;
                qq[rr] = ok_r ? Elem<T>::load1(q + off) : 0.f;
                vv[rr] = ok_r ? Elem<T>::load1(v + off) : 0.f;
                gg[rr] = ok_r ? __ldg(gptr + off) : 0.f;
            }
        };
        load_block(0, kb, qb, vb, gb);
        // swizzled stores of channel c in rows rb + r0 + rr: the row's low
        // three bits are rr (rb and r0 are multiples of 8), so the 16-byte
        // chunk is (c's chunk) ^ rr and only the block's first row varies
        const uint32_t cpart = (uint32_t)((c & 3) << 2), cx4 = (uint32_t)(((c & 31) >> 2) << 4);
        unsigned char *const kq0 = sm.bufKQ + (c >> 5) * 128 * 128 + cpart;
        unsigned char *const km0 = sm.bufKM + (c >> 5) * 64 * 128 + cpart;
        unsigned char *const bw0 = img + IMG_BW + (c >> 5) * 128 * 128 + cpart + 64 * 128;
#pragma unroll 1
        for (int r0 = 0; r0 < 32; r0 += 8) {
            float nk[8], nq[8], nv[8], ng[8];
            if (r0 + 8 < 32) load_block(r0 + 8, nk, nq, nv, ng);
            float bkt[8], bvt[8];
            const int rowb = (rb + r0) * 128;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = rb + r0 + rr;
                const bool valid = r < L;
                const uint32_t sw = (cx4 ^ (uint32_t)(rr << 4)) + rr * 128;
                acc += gb[rr];
                const float gam = acc;
                const float kx = kb[rr] * sm.invk[r];
                const float qx = qb[rr] * sm.invq[r];
                float ktil, qtil;
                if (!unsafe) {
                    const float E = __expf(gam - ref);
                    const float Ei = __expf(ref - gam);
                    const float kp = kx * E, qp = qx * E;
                    *reinterpret_cast<float *>(kq0 + rowb + sw) = kp;
                    *reinterpret_cast<float *>(kq0 + rowb + 64 * 128 + sw) = qp;
                    *reinterpret_cast<float *>(km0 + rowb + sw) = kx * Ei;
                    ktil = kp * eref;
                    qtil = qp * eref;
                } else {
                    // plain [64][128] copies of k^, q^ and gamma for the exact path
                    reinterpret_cast<float *>(sm.bufKQ)[r * D + c] = kx;
                    reinterpret_cast<float *>(sm.bufKQ)[C * D + r * D + c] = qx;
                    reinterpret_cast<float *>(sm.bufKM)[r * D + c] = gam;
                    const float eg = expf(gam);
                    ktil = kx * eg;
                    qtil = qx * eg;
                    st_sw(img + IMG_KT, 128, c, r, valid ? kx * expf(gC - gam) : 0.f);
                }
                *reinterpret_cast<float *>(bw0 + rowb + sw) = qtil;  // Q~ rows of [W; Q~]
                bkt[rr] = sm.beta[r] * ktil;
                bvt[rr] = sm.beta[r] * vb[rr];
            }
            tc::st8(tc::lane_addr(tm, warp, PT_BKT + rb + r0), bkt);
            tc::st8(tc::lane_addr(tm, warp, PT_BVT + rb + r0), bvt);
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                kb[rr] = nk[rr];
                qb[rr] = nq[rr];
                vb[rr] = nv[rr];
                gb[rr] = ng[rr];
            }
        }
    }
    tc::wait_st();
    sync_for_mma();

    bool ok = true;
    // ---- 3. A and P
    if (!unsafe) {
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
            const uint32_t a0 = tc::smem_u32(sm.bufKQ), b0 = tc::smem_u32(sm.bufKM);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_tf32_ss(tm + PT_G, tc::desc_tf32_kstep(a0, 128, ks), tc::desc_tf32_kstep(b0, 64, ks), id,
                                ks > 0);
            tc::commit(&sm.bar);
        }
        ok = wait_mma(&sm.bar, phase, p.err_flag);
        if (ok) {
            // the K^^T image tile, transposed out of K- (K^ = K- e^{gamma_C - ref})
            // now that its product has completed: warp w writes rows
            // 16 w .. 16 w + 15 of both 32-token halves, one token per lane, so
            // every store is one 128-byte line
#pragma unroll 4
            for (int it = 0; it < 32; ++it) {
                const int cc = 16 * warp + (it >> 1);
                const int r = 32 * (it & 1) + lane;
                const float km = *reinterpret_cast<const float *>(sm.bufKM + tc::sw128_off(r, cc, 64));
                st_sw(img + IMG_KT, 128, cc, r, r < L ? km * sm.egcref[cc] : 0.f);
            }
            // G rows (TMEM lanes): 0..63 are A', 64..127 are P; warp w takes
            // columns 32 (w >> 2) .. 32 (w >> 2) + 31
            const int grow = c, r = grow & (C - 1), j0 = rb;
            float g16[16];
#pragma unroll
            for (int jb = 0; jb < 32; jb += 16) {
                tc::ld16(tc::lane_addr(tm, warp, PT_G + j0 + jb), g16);
                tc::wait_ld();
                if (grow < C) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jb + jj;
                        sm.inv.As[r][j] = (j < r) ? sm.beta[r] * g16[jj] : 0.f;
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4) {
                        const int j = j0 + jb + jj;
                        *reinterpret_cast<float4 *>(img + IMG_P + tc::sw128_off(r, j, 64)) =
                            make_float4(j <= r ? g16[jj] : 0.f, j + 1 <= r ? g16[jj + 1] : 0.f,
                                        j + 2 <= r ? g16[jj + 2] : 0.f, j + 3 <= r ? g16[jj + 3] : 0.f);
                    }
                }
            }
        }
    } else {
        // exact path; A goes to registers first because its scratch overlays k^
        const float *kh = reinterpret_cast<const float *>(sm.bufKQ);
        const float *qh = kh + C * D;
        const float *gm = reinterpret_cast<const float *>(sm.bufKM);
        float areg[C * C / kPrepThreads];
#pragma unroll 1
        for (int it = 0; it < C * C / kPrepThreads; ++it) {
            const int idx = tid + it * kPrepThreads;
            const int r = idx / C, j = idx % C;
            float a = 0.f, pp = 0.f;
            if (j <= r) {
                for (int cc = 0; cc < D; ++cc) {
                    const float m = kh[j * D + cc] * expf(gm[r * D + cc] - gm[j * D + cc]);
                    a = fmaf(kh[r * D + cc], m, a);
                    pp = fmaf(qh[r * D + cc], m, pp);
                }
            }
            areg[it] = (j < r) ? sm.beta[r] * a : 0.f;
            *reinterpret_cast<float *>(img + IMG_P + tc::sw128_off(r, j, 64)) = (j <= r) ? pp : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < C * C / kPrepThreads; ++it) {
            const int idx = tid + it * kPrepThreads;
            sm.inv.As[idx / C][idx % C] = areg[it];
        }
    }
    __syncthreads();

    if (ok) {
        // ---- 4. T = (I + A)^-1 (unit lower triangular) by doubling: the four
        // 16 x 16 diagonal blocks by forward substitution (one column per
        // thread, in registers); then the lower-left 16 x 16 block of each
        // 32-row block as -T22 (A21 T11); then the lower-left 32 x 32 block of
        // the whole matrix the same way.
        float(*As)[C + 1] = sm.inv.As;
        float(*Ts)[C + 1] = sm.inv.Ts;
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
            // zero the blocks above the diagonal
            for (int idx = tid - C; idx < C * C; idx += kPrepThreads - C) {
                const int r = idx / C, j = idx % C;
                if ((j >> 4) > (r >> 4)) Ts[r][j] = 0.f;
            }
        }
        __syncthreads();
        // level 1: both 32-row blocks at once (o = 0, 32)
        for (int idx = tid; idx < 2 * 256; idx += kPrepThreads) {
            const int o = 32 * (idx >> 8), r = (idx >> 4) & 15, j = idx & 15;
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                x0 = fmaf(As[o + 16 + r][o + k], Ts[o + k][o + j], x0);
                x1 = fmaf(As[o + 16 + r][o + k + 1], Ts[o + k + 1][o + j], x1);
            }
            sm.xs[(idx >> 8) * 16 + r][j] = x0 + x1;
        }
        __syncthreads();
        for (int idx = tid; idx < 2 * 256; idx += kPrepThreads) {
            const int o = 32 * (idx >> 8), r = (idx >> 4) & 15, j = idx & 15;
            float t = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m <= r) t = fmaf(Ts[o + 16 + r][o + 16 + m], sm.xs[(idx >> 8) * 16 + m][j], t);
            Ts[o + 16 + r][o + j] = -t;
        }
        __syncthreads();
        // level 2: the 32 x 32 blocks
        for (int idx = tid; idx < 32 * 32; idx += kPrepThreads) {
            const int r = idx >> 5, j = idx & 31;
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                x0 = fmaf(As[32 + r][k], Ts[k][j], x0);
                x1 = fmaf(As[32 + r][k + 1], Ts[k + 1][j], x1);
            }
            sm.xs[r][j] = x0 + x1;
        }
        __syncthreads();
        for (int idx = tid; idx < 32 * 32; idx += kPrepThreads) {
            const int r = idx >> 5, j = idx & 31;
            float t0 = 0.f, t1 = 0.f;
#pragma unroll
            for (int m = 0; m < 32; m += 2) {
                if (m <= r) t0 = fmaf(Ts[32 + r][32 + m], sm.xs[m][j], t0);
                if (m + 1 <= r) t1 = fmaf(Ts[32 + r][32 + m + 1], sm.xs[m + 1][j], t1);
            }
            Ts[32 + r][j] = -(t0 + t1);
        }
        __syncthreads();
        for (int idx = tid; idx < C * C / 4; idx += kPrepThreads) {
            const int r = idx / (C / 4), j = (idx % (C / 4)) * 4;
            *reinterpret_cast<float4 *>(sm.bufT + tc::sw128_off(r, j, 64)) =
                make_float4(sm.inv.Ts[r][j], sm.inv.Ts[r][j + 1], sm.inv.Ts[r][j + 2], sm.inv.Ts[r][j + 3]);
        }
        sync_for_mma();

        // ---- 5. W^T = (beta K~)^T T^T and U'^T = (beta V)^T T^T
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
            const uint32_t b0 = tc::smem_u32(sm.bufT);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const uint64_t bd = tc::desc_tf32_kstep(b0, 64, ks);
                tc::mma_tf32_ts(tm + PT_WT, tm + PT_BKT + 8 * ks, bd, id, ks > 0);
                tc::mma_tf32_ts(tm + PT_UPT, tm + PT_BVT + 8 * ks, bd, id, ks > 0);
            }
            tc::commit(&sm.bar);
        }
        ok = wait_mma(&sm.bar, phase, p.err_flag);
        if (ok) {
            // lane c: W[r][c] and U'[r][c] for this thread's token half (a warp's
            // stores of one token row are one 128-byte line)
            float w16[16];
            float *up = reinterpret_cast<float *>(img + IMG_UP);
#pragma unroll
            for (int r0 = 0; r0 < 32; r0 += 16) {
                tc::ld16(tc::lane_addr(tm, warp, PT_WT + rb + r0), w16);
                tc::wait_ld();
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) st_sw(img + IMG_BW, 128, rb + r0 + rr, c, w16[rr]);
                tc::ld16(tc::lane_addr(tm, warp, PT_UPT + rb + r0), w16);
                tc::wait_ld();
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) up[(rb + r0 + rr) * D + c] = w16[rr];
            }
        }
    }
    if (!ok) mbar_wait_drain(&sm.bar, phase & 1);  // the product whose wait gave up
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, PT_COLS);
}

// ================================================================== chain

// One CTA per (sequence, head, block of NR value rows).  With the rows on the
// N side, a chunk step is
//   D1 = [W; Q~] Sb^T            M = 128 (token rows of W, then of Q~), N = NR, K = 128
//   U = U' - D1[0:64]            token r = TMEM lane r, into the swizzled U tile
//   D3 = K^^T U                  M = 128 channels, N = NR, K = 64 tokens
//   D1[64:128] += P U            A = P placed in rows 64..127 of a 128-row tile
//   Sb <- Sb diag(e^{gamma_C}) + D3^T,   O = scale D1[64:128]
// (the A operands come from the chunk's operand image; Sb and U are K-major
// 128-byte-swizzled tiles in shared memory).  Only D1 -> U -> D3 -> Sb is on
// the serial path: P U has its own completion barrier and D1 alternates
// between two TMEM regions, so a chunk's output is written while the next
// chunk's first product runs.  The thread phases run on 8 warps: warps w and
// w + 4 read the same TMEM lanes and take one half of the NR columns each
// (256 threads measured 807 us per 8192-token prefill, 128 threads 842 us,
// 512 threads 830 us).
constexpr int NR = 32;
constexpr int kRowBlocks = D / NR;
constexpr uint32_t CT_D1 = 0, CT_D3 = 2 * NR;  // D1 ping-pongs between columns 0 and NR
constexpr uint32_t CT_COLS = 128;
constexpr uint32_t kPKBytes = 2 * 8192 + 128 * 64 * 4 + D * 4;  // P, K^^T, e^{gamma_C}

struct ChainSmem {
    unsigned char bw[2][128 * 128 * 4];  // [W; Q~], double-buffered
    unsigned char p128[2][128 * 128];    // 2 token atoms of a 128-row tile; P in rows 64..127
    unsigned char kt[2][128 * 128];      // K^^T: 2 token atoms of 128 channel rows
    unsigned char sb[4][NR * 128];       // state block: 4 channel atoms of NR rows
    unsigned char ub[2][NR * 128];       // U block: 2 token atoms of NR rows
    float egc[2][D];
    uint64_t full_bw[2];
    uint64_t full_pk;
    uint64_t mma1, mma2, mma3;  // [W; Q~] Sb^T, P U, K^^T U done
    uint32_t tmem_base;
};
constexpr size_t kChainSmem = sizeof(ChainSmem) + 1024;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) chain_tc_kernel(const PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    ChainSmem &sm =
        *reinterpret_cast<ChainSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t *plan = static_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    if (plan[n + 1] == 0) return;
    const int s = blockIdx.x, h = blockIdx.y, i0 = blockIdx.z * NR, H = p.H;
    const int tid = threadIdx.x, warp = tid >> 5;
    // TMEM lane of this thread (warps w and w + 4 share lanes 32 (w & 3) ..),
    // and the half of the block's NR value rows (columns) it takes
    const int lr = ((warp & 3) << 5) | (tid & 31), hf = warp >> 2;
    constexpr int NH = NR / 2;
    const int32_t cs = p.cu_seqlens[s], ce = p.cu_seqlens[s + 1];
    const int slot = p.slot_ids[s];
    T *out = static_cast<T *>(p.out);
    const int64_t tok_stride = (int64_t)H * D, hoff = (int64_t)h * D + i0;
    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        for (int64_t t = cs; t < ce; ++t)
            if (tid < NR) Elem<T>::store1(out + t * tok_stride + hoff + tid, 0.f);
        if (slot >= 0 && h == 0 && blockIdx.z == 0 && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    const int nchunks = plan[s + 1] - plan[s];
    const unsigned char *ws = static_cast<const unsigned char *>(p.workspace) + plan_bytes(n);
    auto image = [&](int ci) {
        return ws + ((size_t)(plan[s] + ci) * H + h) * (size_t)IMG_BYTES;
    };
    auto issue_bw = [&](int ci, int b) {
        mbar_arrive_expect_tx(&sm.full_bw[b], 128 * 128 * 4);
        bulk_g2s(sm.bw[b], image(ci) + IMG_BW, 128 * 128 * 4, &sm.full_bw[b]);
    };
    auto issue_pk = [&](int ci) {
        mbar_arrive_expect_tx(&sm.full_pk, kPKBytes);
        bulk_g2s(sm.p128[0] + 8192, image(ci) + IMG_P, 8192, &sm.full_pk);
        bulk_g2s(sm.p128[1] + 8192, image(ci) + IMG_P + 8192, 8192, &sm.full_pk);
        bulk_g2s(sm.kt, image(ci) + IMG_KT, 128 * 64 * 4, &sm.full_pk);
        bulk_g2s(sm.egc[ci & 1], image(ci) + IMG_EGC, D * 4, &sm.full_pk);
    };

    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, CT_COLS);
    if (tid == 0) {
        mbar_init(&sm.full_bw[0], 1);
        mbar_init(&sm.full_bw[1], 1);
        mbar_init(&sm.full_pk, 1);
        mbar_init(&sm.mma1, 1);
        mbar_init(&sm.mma2, 1);
        mbar_init(&sm.mma3, 1);
        fence_barrier_init();
        if (nchunks > 0) {
            issue_bw(0, 0);
            issue_pk(0);
        }
    }
    // rows 0..63 of the P tile only feed discarded accumulator lanes; zeroed
    // once so that they hold finite values
    for (int idx = tid; idx < 2 * 8192 / 16; idx += kThreads)
        *reinterpret_cast<uint4 *>(sm.p128[idx >> 9] + (idx & 511) * 16) = make_uint4(0, 0, 0, 0);
    // initial state block (rows i0 .. i0 + NR) into the swizzled tile
    float *Sg = p.pool + ((int64_t)slot * H + h) * (int64_t)D * D + (int64_t)i0 * D;
    for (int idx = tid; idx < NR * (D / 4); idx += kThreads) {
        const int i = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
        const float4 x = p.init_from_pool ? *reinterpret_cast<const float4 *>(Sg + (int64_t)i * D + c4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(&sm.sb[0][0] + tc::sw128_off(i, c4, NR)) = x;
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem_base;

    uint32_t ph1 = 0, ph2 = 0, ph3 = 0;
    // products committed and not yet observed complete (uniform across the CTA)
    bool pend1 = false, pend2 = false, pend3 = false;
    bool ok = true;
    int last_bw0 = nchunks > 0 ? 0 : -1, last_bw1 = -1, last_pk = nchunks > 0 ? 0 : -1;
    // this token thread's U' values for the block (threads 0..63), the next
    // chunk's in flight while the current one computes
    float upc[NH], upn[NH];
    auto load_up = [&](int ci, float (&dst)[NH]) {
        const float4 *src =
            reinterpret_cast<const float4 *>(image(ci) + IMG_UP) + ((size_t)lr * D + i0 + hf * NH) / 4;
#pragma unroll
        for (int j = 0; j < NH / 4; ++j) {
            const float4 x = __ldg(src + j);
            dst[4 * j] = x.x; dst[4 * j + 1] = x.y; dst[4 * j + 2] = x.z; dst[4 * j + 3] = x.w;
        }
    };
    // O = scale D1[64:128] of chunk cj from the D1 region at column col
    // (token threads 64..127; warp-uniform)
    auto write_output = [&](int cj, uint32_t col) {
        const int64_t tj = (int64_t)cs + (int64_t)cj * C;
        const int Lj = (int)((int64_t)ce - tj < C ? (int64_t)ce - tj : C);
        float o[NH];
        tc::ld16(tc::lane_addr(tm, warp, col + hf * NH), o);
        tc::wait_ld();
        if (lr - C < Lj) {
            T *dst = out + (tj + lr - C) * tok_stride + hoff + hf * NH;
            constexpr int V = 16 / sizeof(T);  // elements per 16-byte store
#pragma unroll
            for (int v0 = 0; v0 < NH; v0 += V) {
                alignas(16) T pack[V];
#pragma unroll
                for (int e2 = 0; e2 < V; ++e2) Elem<T>::store1(&pack[e2], p.scale * o[v0 + e2]);
                *reinterpret_cast<uint4 *>(dst + v0) = *reinterpret_cast<const uint4 *>(pack);
            }
        }
    };
    if (lr < C && nchunks > 0) load_up(0, upc);

    for (int ci = 0; ci < nchunks; ++ci) {
        const int b = ci & 1;
        const uint32_t d1 = CT_D1 + b * NR;
        const bool landed = mbar_wait(&sm.full_bw[b], (ci >> 1) & 1);
        if (__syncthreads_and(landed) == 0) {
            if (tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            ok = false;
            break;
        }
        tc::fence_after_sync();
        // ---- D1 = [W; Q~] Sb^T
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, NR);
            const uint32_t a0 = tc::smem_u32(sm.bw[b]), b0 = tc::smem_u32(sm.sb);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_tf32_ss(tm + d1, tc::desc_tf32_kstep(a0, 128, ks), tc::desc_tf32_kstep(b0, NR, ks), id,
                                ks > 0);
            tc::commit(&sm.mma1);
            // the other [W; Q~] buffer's last product (chunk ci - 1) has completed
            if (ci + 1 < nchunks) {
                issue_bw(ci + 1, b ^ 1);
                if (b) last_bw0 = ci + 1; else last_bw1 = ci + 1;
                // the next chunk's P, K^^T and e^{gamma_C} towards L2 ahead of their copy
                bulk_prefetch_l2(image(ci + 1) + IMG_P, IMG_EGC + D * 4 - IMG_P);
            }
        }
        // the previous chunk's output goes out while this chunk's first product runs
        if (ci > 0 && lr >= C) write_output(ci - 1, CT_D1 + (b ^ 1) * NR);
        if (lr < C && ci + 1 < nchunks) load_up(ci + 1, upn);
        pend1 = true;
        ok = wait_mma(&sm.mma1, ph1, p.err_flag);
        if (!ok) break;
        pend1 = false;
        // ---- U = U' - W Sb^T (thread = token r = TMEM lane r)
        if (lr < C) {
            float d[NH];
            tc::ld16(tc::lane_addr(tm, warp, d1 + hf * NH), d);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < NH; ++i) st_sw(&sm.ub[0][0], NR, hf * NH + i, lr, upc[i] - d[i]);
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---- D3 = K^^T U (serial path), then D1[64:128] += P U
        const bool pk = mbar_wait(&sm.full_pk, ci & 1);
        if (__syncthreads_and(pk) == 0) {
            if (tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            ok = false;
            break;
        }
        tc::fence_after_sync();
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, NR);
            const uint32_t ap = tc::smem_u32(sm.p128), ak = tc::smem_u32(sm.kt), b0 = tc::smem_u32(sm.ub);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ss(tm + CT_D3, tc::desc_tf32_kstep(ak, 128, ks), tc::desc_tf32_kstep(b0, NR, ks), id,
                                ks > 0);
            tc::commit(&sm.mma3);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ss(tm + d1, tc::desc_tf32_kstep(ap, 128, ks), tc::desc_tf32_kstep(b0, NR, ks), id, 1);
            tc::commit(&sm.mma2);
        }
        pend2 = pend3 = true;
        ok = wait_mma(&sm.mma3, ph3, p.err_flag);
        if (!ok) break;
        pend3 = false;
        // ---- Sb <- Sb diag(e^{gamma_C}) + D3^T (thread = channel c = TMEM lane c)
        {
            float d[NH];
            tc::ld16(tc::lane_addr(tm, warp, CT_D3 + hf * NH), d);
            tc::wait_ld();
            const float e = sm.egc[b][lr];
#pragma unroll
            for (int i = 0; i < NH; ++i) {
                float *sp = reinterpret_cast<float *>(&sm.sb[0][0] + tc::sw128_off(hf * NH + i, lr, NR));
                *sp = fmaf(*sp, e, d[i]);
            }
        }
        if (lr < C) {
#pragma unroll
            for (int j = 0; j < NH; ++j) upc[j] = upn[j];
        }
        // P U is done (it ran during the update): P and K^^T are free, and the
        // other e^{gamma_C} slot was last read by chunk ci - 1
        ok = wait_mma(&sm.mma2, ph2, p.err_flag);
        if (!ok) break;
        pend2 = false;
        if (tid == 0 && ci + 1 < nchunks) {
            issue_pk(ci + 1);
            last_pk = ci + 1;
        }
        fence_proxy_async_smem();  // Sb writes before the next product; e^{gamma_C} reads before its refill
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    if (ok && nchunks > 0 && lr >= C) write_output(nchunks - 1, CT_D1 + ((nchunks - 1) & 1) * NR);

    if (ok) {
        for (int idx = tid; idx < NR * (D / 4); idx += kThreads) {
            const int i = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
            *reinterpret_cast<float4 *>(Sg + (int64_t)i * D + c4) =
                *reinterpret_cast<const float4 *>(&sm.sb[0][0] + tc::sw128_off(i, c4, NR));
        }
    } else if (tid == 0) {
        // bounded waits so that no product or bulk copy is still writing when
        // the CTA releases its memory: each product still outstanding on its
        // pending phase, and the last copy issued into each buffer (a copy
        // already observed complete passes its phase at once)
        if (pend1) mbar_wait_drain(&sm.mma1, ph1 & 1);
        if (pend2) mbar_wait_drain(&sm.mma2, ph2 & 1);
        if (pend3) mbar_wait_drain(&sm.mma3, ph3 & 1);
        if (last_bw0 >= 0) mbar_wait_drain(&sm.full_bw[0], (last_bw0 >> 1) & 1);
        if (last_bw1 >= 0) mbar_wait_drain(&sm.full_bw[1], (last_bw1 >> 1) & 1);
        if (last_pk >= 0) mbar_wait_drain(&sm.full_pk, last_pk & 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, CT_COLS);
}

}  // namespace prefill_tc

#ifndef KDA_PREFILL_TC
#define KDA_PREFILL_TC 1
#endif

bool prefill_tc_supported(int dk, int dv, int dtype) {
    return KDA_PREFILL_TC && dtype == KDA_DT_BF16 && dk == 128 && dv == 128;
}

size_t prefill_tc_workspace_bytes(int H, int32_t num_seqs, int64_t total_tokens) {
    using namespace prefill_tc;
    return plan_bytes(num_seqs) + (size_t)max_chunks(num_seqs, total_tokens) * (size_t)H * IMG_BYTES;
}

cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t st) {
    using namespace prefill_tc;
    cudaError_t e = cudaFuncSetAttribute(prep_tc_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chain_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kChainSmem);
    if (e != cudaSuccess) return e;
    const int64_t mc = max_chunks(p.num_seqs, p.total_tokens);
    if (mc > 0) {
        prep_tc_kernel<__nv_bfloat16><<<dim3((unsigned)mc, (unsigned)p.H), kPrepThreads, kPrepSmem, st>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    chain_tc_kernel<__nv_bfloat16>
        <<<dim3((unsigned)p.num_seqs, (unsigned)p.H, (unsigned)kRowBlocks), kThreads, kChainSmem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
