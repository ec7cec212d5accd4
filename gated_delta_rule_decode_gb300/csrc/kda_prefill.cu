// Chunked KDA prefill in WY/UT form (64-token chunks).
//
// "Ascend day-0 support for Kimi K3", section "KDA Prefill and Decode dual
// path": the prefill takes 64-token chunks and organises Q/K normalisation,
// gate accumulation and the chunk KDA as batched computation.  The chunk form
// used here follows from unrolling the token recurrence inside a chunk
// (gamma = in-chunk cumulative gate, per key channel):
//
//   A[r,j] = beta_r sum_c k^_r[c] k^_j[c] e^{gamma_r[c]-gamma_j[c]}   (j < r)
//   P[r,j] =        sum_c q^_r[c] k^_j[c] e^{gamma_r[c]-gamma_j[c]}   (j <= r)
//   T = (I + A)^-1,  W = T diag(beta) K~,  U' = T diag(beta) V
//   with K~_r = k^_r e^{gamma_r},  Q~_r = q^_r e^{gamma_r},
//        K^_j = k^_j e^{gamma_C - gamma_j}
//   per chunk, in sequence order, with S the state entering the chunk:
//   U = U' - W S^T;  O = scale (Q~ S^T + P U);  S <- S diag(e^{gamma_C}) + U^T K^
//
// Two kernels:
//   chunk_prep_kernel  (one CTA per chunk x head, all chunks in parallel):
//       normalisation, gate cumsum, A and P, the UT inverse T, and the WY
//       factors W and U'; writes W, U', Q~, K^, P and e^{gamma_C} to the
//       workspace.
//   chunk_chain_kernel (one CTA per sequence x head x block of value rows):
//       walks the chunks of its sequence in order carrying its rows of S
//       (value rows of the state are independent), writes the outputs and
//       finally the state to the sequence's slot.
//
// Overflow safety of the decay factors: the exponent difference
// gamma_r - gamma_j is split at a reference point ref_I = gamma at the first
// token of the 16-row block I that holds r:  e^{gamma_r - ref_I} <= 1 and,
// for j before block I, e^{ref_I - gamma_j} <= 1 (gamma is non-increasing
// for g <= 0); only inside the diagonal 16x16 block does a factor exceed 1,
// by at most the decay over 15 tokens.
#include <stdint.h>

#include "kda.h"
#include "kda_check.cuh"
#include "kda_internal.h"
#include "kda_rowmath.cuh"

namespace kda {
namespace prefill {

constexpr int C = 64;          // chunk length
constexpr int kPrepThreads = 256;
constexpr int kChainThreads = 256;
constexpr int kChainRows = 32;  // value rows per chain CTA

// ---------------------------------------------------------------- workspace

struct WsLayout {
    size_t plan_bytes;   // int32 chunk offsets [num_seqs + 1] + status word
    size_t chunk_bytes;  // per (chunk, head)
    size_t off_w, off_u, off_q, off_k, off_p, off_e;
    int64_t max_chunks;
};

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int dk, int dv, int32_t num_seqs, int64_t total_tokens) {
    WsLayout L;
    L.plan_bytes = round_up(sizeof(int32_t) * ((size_t)num_seqs + 2), 256);
    size_t o = 0;
    L.off_w = o; o += (size_t)C * dk * 4;
    L.off_u = o; o += (size_t)C * dv * 4;
    L.off_q = o; o += (size_t)C * dk * 4;
    L.off_k = o; o += (size_t)C * dk * 4;
    L.off_p = o; o += (size_t)C * C * 4;
    L.off_e = o; o += (size_t)dk * 4;
    L.chunk_bytes = round_up(o, 256);
    L.max_chunks = (total_tokens + C - 1) / C + num_seqs;
    return L;
}

// ---------------------------------------------------------------- plan

// Validates cu_seqlens and writes the per-sequence chunk offsets.
// plan[s] = number of chunks before sequence s; plan[n+1] = 1 when valid.
__global__ void plan_kernel(const int32_t *cu, int32_t n, int64_t total_tokens, int32_t *plan,
                            int32_t *err_flag) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    bool ok = (cu[0] == 0);
    int32_t acc = 0;
    for (int s = 0; s < n; ++s) {
        plan[s] = acc;
        const int32_t a = cu[s], b = cu[s + 1];
        if (b < a || (int64_t)b > total_tokens) ok = false;
        if (ok) acc += (b - a + C - 1) / C;
    }
    plan[n] = acc;
    plan[n + 1] = ok ? 1 : 0;
    if (!ok && err_flag) atomicOr(err_flag, KDA_DEVERR_SEQLENS);
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

template <typename T>
__device__ inline float ld1(const T *p) { return Elem<T>::load1(p); }

// ---------------------------------------------------------------- chunk prep

template <int DK, int DV, typename T>
struct PrepSmem {
    float kh[C][DK + 1];   // normalised key (rows >= len are zero)
    float qh[C][DK + 1];   // normalised query; later beta_j k^_j e^{gamma_j}
    float gam[C][DK + 1];  // in-chunk cumulative gate
    float km[C][DK + 1];   // column-side factors of the current row block
    float kp[16][DK + 1];  // row-side factors of the current row block
    float qp[16][DK + 1];
    float A[C][C + 1];
    float P[C][C + 1];     // stored to the workspace, then reused for T
    float vb[C][DV + 1];   // beta_j v_j
    float beta[C];
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kPrepThreads) chunk_prep_kernel(const PrefillParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<PrepSmem<DK, DV, T> *>(smem_raw);
    const WsLayout L = ws_layout(DK, DV, p.num_seqs, p.total_tokens);
    const int32_t *plan = reinterpret_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    if (plan[n + 1] == 0) return;
    const int32_t chunk = blockIdx.x;
    if (chunk >= plan[n]) return;
    const int h = blockIdx.y;
    const int H = p.H;
    const int s = find_seq(plan, n, chunk);
    const int slot = p.slot_ids[s];
    if (slot < 0 || (int64_t)slot >= p.num_slots) return;  // nothing to prepare
    const int64_t t0 = (int64_t)p.cu_seqlens[s] + (int64_t)(chunk - plan[s]) * C;
    const int len = (int)((int64_t)p.cu_seqlens[s + 1] - t0 < C ? (int64_t)p.cu_seqlens[s + 1] - t0 : C);
    // checked build: the chunk's tokens and its workspace block
    if (!in_bounds(t0, len, p.total_tokens, p.err_flag) ||
        !in_bounds((int64_t)(L.plan_bytes + ((size_t)chunk * H + h) * L.chunk_bytes), (int64_t)L.chunk_bytes,
                   (int64_t)p.workspace_bytes, p.err_flag))
        return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *bb = static_cast<const T *>(p.b);

    // 1. Q/K L2Norm (one warp per token row), beta
    for (int r = warp; r < C; r += kPrepThreads / 32) {
        if (r < len) {
            const int64_t base = ((t0 + r) * H + h) * DK;
            float kx[DK / 32], qx[DK / 32];
            float ks = 0.f, qs = 0.f;
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) {
                kx[e] = ld1(k + base + lane + 32 * e);
                qx[e] = ld1(q + base + lane + 32 * e);
                ks = fmaf(kx[e], kx[e], ks);
                qs = fmaf(qx[e], qx[e], qs);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ks += __shfl_xor_sync(0xffffffffu, ks, o);
                qs += __shfl_xor_sync(0xffffffffu, qs, o);
            }
            const float ki = rsqrtf(ks + p.eps), qi = rsqrtf(qs + p.eps);
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) {
                sm.kh[r][lane + 32 * e] = kx[e] * ki;
                sm.qh[r][lane + 32 * e] = qx[e] * qi;
            }
            if (lane == 0) sm.beta[r] = sigmoid_f(ld1(bb + (t0 + r) * H + h));
        } else {
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) {
                sm.kh[r][lane + 32 * e] = 0.f;
                sm.qh[r][lane + 32 * e] = 0.f;
            }
            if (lane == 0) sm.beta[r] = 0.f;
        }
    }
    // 2. gate accumulation: gamma_r = sum_{j<=r} g_j, one thread per channel
    for (int c = tid; c < DK; c += kPrepThreads) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            if (r < len) acc += p.g[((t0 + r) * H + h) * DK + c];
            sm.gam[r][c] = acc;  // rows past the end repeat the last value
        }
    }
    __syncthreads();

    // 3. A and P, one 16-row block I at a time with reference gamma[16 I]
    for (int I = 0; I < C / 16; ++I) {
        const int ncol = 16 * (I + 1);
        const int o = 16 * I;
        for (int idx = tid; idx < ncol * DK; idx += kPrepThreads) {
            const int j = idx / DK, c = idx % DK;
            sm.km[j][c] = sm.kh[j][c] * expf(sm.gam[o][c] - sm.gam[j][c]);
        }
        for (int idx = tid; idx < 16 * DK; idx += kPrepThreads) {
            const int r = idx / DK, c = idx % DK;
            const float f = expf(sm.gam[o + r][c] - sm.gam[o][c]);
            sm.kp[r][c] = sm.kh[o + r][c] * f;
            sm.qp[r][c] = sm.qh[o + r][c] * f;
        }
        __syncthreads();
        // rows r in block I, columns j < ncol: 16 x ncol entries of A and P
        for (int idx = tid; idx < 16 * ncol; idx += kPrepThreads) {
            const int rl = idx / ncol, j = idx % ncol, r = o + rl;
            float a = 0.f, pp = 0.f;
            if (j <= r) {
#pragma unroll 8
                for (int c = 0; c < DK; ++c) {
                    a = fmaf(sm.kp[rl][c], sm.km[j][c], a);
                    pp = fmaf(sm.qp[rl][c], sm.km[j][c], pp);
                }
            }
            sm.A[r][j] = (j < r) ? sm.beta[r] * a : 0.f;
            sm.P[r][j] = (j <= r) ? pp : 0.f;
        }
        __syncthreads();
    }
    // upper parts are zero
    for (int idx = tid; idx < C * C; idx += kPrepThreads) {
        const int r = idx / C, j = idx % C;
        if (j > r) { sm.A[r][j] = 0.f; sm.P[r][j] = 0.f; }
    }
    __syncthreads();

    // P is final: store it, then reuse its buffer for T.
    unsigned char *blk = static_cast<unsigned char *>(p.workspace) + L.plan_bytes +
                         ((size_t)chunk * H + h) * L.chunk_bytes;
    float *Pg = reinterpret_cast<float *>(blk + L.off_p);
    for (int idx = tid; idx < C * C; idx += kPrepThreads) Pg[idx] = sm.P[idx / C][idx % C];
    __syncthreads();

    // 4. T = (I + A)^-1 (unit lower triangular), stored in P's buffer.
    //    Diagonal 16x16 blocks by forward substitution (warp per block, lane
    //    per column), then off-diagonal blocks by distance from the diagonal:
    //    T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ.
    float *Tm = &sm.P[0][0];
    auto Tat = [&](int r, int j) -> float & { return Tm[r * (C + 1) + j]; };
    for (int idx = tid; idx < C * (C + 1); idx += kPrepThreads) Tm[idx] = 0.f;
    __syncthreads();
    if (warp < 4 && lane < 16) {
        const int I = warp, j = lane, o = 16 * I;
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < r && m >= j) acc -= sm.A[o + r][o + m] * col[m];
            col[r] = (r >= j) ? acc : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tat(o + r, o + j) = col[r];
    }
    __syncthreads();
    for (int dist = 1; dist < 4; ++dist) {
        // blocks (I, J = I - dist); one thread per element, 256 per block
        const int nblk = 4 - dist;
        for (int idx = tid; idx < nblk * 256; idx += kPrepThreads) {
            const int bi = idx / 256, e = idx % 256;
            const int I = bi + dist, J = bi;
            const int r = e / 16, j = e % 16;
            // X = sum_{K=J}^{I-1} A_IK T_KJ  (row r of block I, col j of block J)
            // then T_IJ = -T_II X; compute X row r on the fly
            float out = 0.f;
            for (int m = 0; m <= r; ++m) {
                const float tim = Tat(16 * I + r, 16 * I + m);
                float x = 0.f;
                for (int K = J; K < I; ++K)
                    for (int kk = 0; kk < 16; ++kk)
                        x = fmaf(sm.A[16 * I + m][16 * K + kk], Tat(16 * K + kk, 16 * J + j), x);
                out = fmaf(tim, x, out);
            }
            Tat(16 * I + r, 16 * J + j) = -out;
        }
        __syncthreads();
    }

    // 5. WY factors and chunk-boundary quantities to the workspace.
    float *W = reinterpret_cast<float *>(blk + L.off_w);
    float *Up = reinterpret_cast<float *>(blk + L.off_u);
    float *Qt = reinterpret_cast<float *>(blk + L.off_q);
    float *Kh = reinterpret_cast<float *>(blk + L.off_k);
    float *Eg = reinterpret_cast<float *>(blk + L.off_e);
    const int last = len - 1;
    // Q~, K^ (decayed to the chunk end), P and e^{gamma_C}
    for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
        const int r = idx / DK, c = idx % DK;
        Qt[idx] = sm.qh[r][c] * expf(sm.gam[r][c]);
        Kh[idx] = (r < len) ? sm.kh[r][c] * expf(sm.gam[last][c] - sm.gam[r][c]) : 0.f;
    }
    for (int c = tid; c < DK; c += kPrepThreads) Eg[c] = expf(sm.gam[last][c]);
    for (int idx = tid; idx < C * DV; idx += kPrepThreads) {
        const int j = idx / DV, i = idx % DV;
        sm.vb[j][i] = (j < len) ? sm.beta[j] * ld1(v + ((t0 + j) * H + h) * DV + i) : 0.f;
    }
    __syncthreads();
    // beta_j K~_j = beta_j k^_j e^{gamma_j}, in place of q^
    for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
        const int j = idx / DK, c = idx % DK;
        sm.qh[j][c] = sm.beta[j] * sm.kh[j][c] * expf(sm.gam[j][c]);
    }
    __syncthreads();
    // W = T diag(beta) K~,  U' = T diag(beta) V   (T lower triangular)
    for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
        const int r = idx / DK, c = idx % DK;
        float acc = 0.f;
        for (int j = 0; j <= r; ++j) acc = fmaf(Tat(r, j), sm.qh[j][c], acc);
        W[idx] = acc;
    }
    for (int idx = tid; idx < C * DV; idx += kPrepThreads) {
        const int r = idx / DV, i = idx % DV;
        float acc = 0.f;
        for (int j = 0; j <= r; ++j) acc = fmaf(Tat(r, j), sm.vb[j][i], acc);
        Up[idx] = acc;
    }
}

// ---------------------------------------------------------------- chain

template <int DK, int DV>
struct ChainSmem {
    float S[kChainRows][DK + 1];   // this CTA's rows of the state
    float W[C][DK + 1];
    float Q[C][DK + 1];
    float K[C][DK + 1];
    float P[C][C + 1];
    float U[C][kChainRows + 1];
    float E[DK];
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kChainThreads) chunk_chain_kernel(const PrefillParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<ChainSmem<DK, DV> *>(smem_raw);
    const WsLayout L = ws_layout(DK, DV, p.num_seqs, p.total_tokens);
    const int32_t *plan = reinterpret_cast<const int32_t *>(p.workspace);
    const int n = p.num_seqs;
    if (plan[n + 1] == 0) return;
    constexpr int NB = DV / kChainRows;
    const int s = blockIdx.x / NB, rb = blockIdx.x % NB;
    const int h = blockIdx.y, H = p.H;
    const int tid = threadIdx.x;
    const int32_t cs = p.cu_seqlens[s], ce = p.cu_seqlens[s + 1];
    const int slot = p.slot_ids[s];
    T *out = static_cast<T *>(p.out);
    // checked build: the sequence's tokens and its chunks' workspace blocks
    if (!in_bounds(cs, (int64_t)ce - cs, p.total_tokens, p.err_flag) ||
        !in_bounds((int64_t)(L.plan_bytes + (size_t)plan[s] * H * L.chunk_bytes),
                   (int64_t)(plan[s + 1] - plan[s]) * H * (int64_t)L.chunk_bytes, (int64_t)p.workspace_bytes,
                   p.err_flag))
        return;
    if (slot < 0 || (int64_t)slot >= p.num_slots) {
        for (int64_t idx = tid; idx < (int64_t)(ce - cs) * kChainRows; idx += kChainThreads) {
            const int64_t t = cs + idx / kChainRows;
            const int i = rb * kChainRows + (int)(idx % kChainRows);
            Elem<T>::store1(out + (t * H + h) * DV + i, 0.f);
        }
        if (slot >= 0 && rb == 0 && h == 0 && tid == 0 && p.err_flag)
            atomicOr(p.err_flag, KDA_DEVERR_SLOT);
        return;
    }
    float *Sg = p.pool + ((int64_t)slot * H + h) * (int64_t)DV * DK + (int64_t)rb * kChainRows * DK;
    if (!in_bounds(((int64_t)slot * H + h) * DV * DK + (int64_t)rb * kChainRows * DK, (int64_t)kChainRows * DK,
                   p.num_slots * H * (int64_t)DV * DK, p.err_flag))
        return;
    for (int idx = tid; idx < kChainRows * DK; idx += kChainThreads)
        sm.S[idx / DK][idx % DK] = p.init_from_pool ? Sg[idx] : 0.f;
    const float scale = p.scale;
    const int nchunks = plan[s + 1] - plan[s];
    // snapshot requests of this sequence (the same for every thread)
    int snap_ptr = 0, snap_hi = 0;
    bool snap_bad = false;
    if (p.num_snaps > 0) snap_range(p, s, snap_ptr, snap_hi);
    auto store_snapshot = [&](int sl) {
        float *dst = p.pool + ((int64_t)sl * H + h) * (int64_t)DV * DK + (int64_t)rb * kChainRows * DK;
        for (int idx = tid; idx < kChainRows * DK; idx += kChainThreads) dst[idx] = sm.S[idx / DK][idx % DK];
    };
    for (int ci = 0; ci < nchunks; ++ci) {
        const int32_t chunk = plan[s] + ci;
        const int64_t t0 = (int64_t)cs + (int64_t)ci * C;
        const int len = (int)((int64_t)ce - t0 < C ? (int64_t)ce - t0 : C);
        const unsigned char *blk = static_cast<const unsigned char *>(p.workspace) + L.plan_bytes +
                                   ((size_t)chunk * H + h) * L.chunk_bytes;
        const float *W = reinterpret_cast<const float *>(blk + L.off_w);
        const float *Up = reinterpret_cast<const float *>(blk + L.off_u);
        const float *Qt = reinterpret_cast<const float *>(blk + L.off_q);
        const float *Kh = reinterpret_cast<const float *>(blk + L.off_k);
        const float *Pg = reinterpret_cast<const float *>(blk + L.off_p);
        const float *Eg = reinterpret_cast<const float *>(blk + L.off_e);
        __syncthreads();  // previous chunk done with the staged tiles
        for (int idx = tid; idx < C * DK; idx += kChainThreads) {
            sm.W[idx / DK][idx % DK] = W[idx];
            sm.Q[idx / DK][idx % DK] = Qt[idx];
            sm.K[idx / DK][idx % DK] = Kh[idx];
        }
        for (int idx = tid; idx < C * C; idx += kChainThreads) sm.P[idx / C][idx % C] = Pg[idx];
        for (int c = tid; c < DK; c += kChainThreads) sm.E[c] = Eg[c];
        __syncthreads();
        // U = U' - W S^T  (C x rows)
        for (int idx = tid; idx < C * kChainRows; idx += kChainThreads) {
            const int r = idx / kChainRows, i = idx % kChainRows;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) acc = fmaf(sm.W[r][c], sm.S[i][c], acc);
            sm.U[r][i] = Up[r * DV + rb * kChainRows + i] - acc;
        }
        __syncthreads();
        // O = scale (Q~ S^T + P U)
        for (int idx = tid; idx < C * kChainRows; idx += kChainThreads) {
            const int r = idx / kChainRows, i = idx % kChainRows;
            if (r >= len) continue;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) acc = fmaf(sm.Q[r][c], sm.S[i][c], acc);
            float acc2 = 0.f;
            for (int j = 0; j <= r; ++j) acc2 = fmaf(sm.P[r][j], sm.U[j][i], acc2);
            Elem<T>::store1(out + ((t0 + r) * H + h) * DV + rb * kChainRows + i, scale * (acc + acc2));
        }
        __syncthreads();
        // S <- S diag(e^{gamma_C}) + U^T K^
        for (int idx = tid; idx < kChainRows * DK; idx += kChainThreads) {
            const int i = idx / DK, c = idx % DK;
            float acc = sm.S[i][c] * sm.E[c];
            for (int j = 0; j < len; ++j) acc = fmaf(sm.U[j][i], sm.K[j][c], acc);
            sm.S[i][c] = acc;
        }
        // the state after ci + 1 chunks, where a snapshot asks for it
        if (snap_ptr < snap_hi) {
            __syncthreads();
            snap_ptr = snap_due(p, snap_ptr, snap_hi, min((int64_t)(ci + 1) * C, (int64_t)ce - cs), C, snap_bad,
                                store_snapshot);
        }
    }
    // requests past the sequence's last whole chunk can never be met
    if (snap_ptr < snap_hi) snap_bad = true;
    if (snap_bad && rb == 0 && h == 0 && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SNAPSHOT);
    __syncthreads();
    for (int idx = tid; idx < kChainRows * DK; idx += kChainThreads) Sg[idx] = sm.S[idx / DK][idx % DK];
}

// ---------------------------------------------------------------- launch

template <int DK, int DV, typename T>
static cudaError_t launch_t(const PrefillParams &p, cudaStream_t st) {
    const WsLayout L = ws_layout(DK, DV, p.num_seqs, p.total_tokens);
    int32_t *plan = static_cast<int32_t *>(p.workspace);
    plan_kernel<<<1, 32, 0, st>>>(p.cu_seqlens, p.num_seqs, p.total_tokens, plan, p.err_flag);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (L.max_chunks > 0) {
        const size_t sm1 = sizeof(PrepSmem<DK, DV, T>);
        e = cudaFuncSetAttribute(chunk_prep_kernel<DK, DV, T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
        if (e != cudaSuccess) return e;
        dim3 g1((unsigned)L.max_chunks, (unsigned)p.H);
        chunk_prep_kernel<DK, DV, T><<<g1, kPrepThreads, sm1, st>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t sm2 = sizeof(ChainSmem<DK, DV>);
    e = cudaFuncSetAttribute(chunk_chain_kernel<DK, DV, T>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
    if (e != cudaSuccess) return e;
    dim3 g2((unsigned)(p.num_seqs * (DV / kChainRows)), (unsigned)p.H);
    chunk_chain_kernel<DK, DV, T><<<g2, kChainThreads, sm2, st>>>(p);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_dtype(const PrefillParams &p, cudaStream_t st) {
    if (p.dk == 128) {
        if (p.dv == 128) return launch_t<128, 128, T>(p, st);
        if (p.dv == 64) return launch_t<128, 64, T>(p, st);
        return launch_t<128, 32, T>(p, st);
    }
    if (p.dk == 64) {
        if (p.dv == 128) return launch_t<64, 128, T>(p, st);
        if (p.dv == 64) return launch_t<64, 64, T>(p, st);
        return launch_t<64, 32, T>(p, st);
    }
    if (p.dv == 128) return launch_t<32, 128, T>(p, st);
    if (p.dv == 64) return launch_t<32, 64, T>(p, st);
    return launch_t<32, 32, T>(p, st);
}

}  // namespace prefill

size_t prefill_workspace_bytes(int H, int dk, int dv, int dtype, int32_t num_seqs, int64_t total_tokens) {
    const prefill::WsLayout L = prefill::ws_layout(dk, dv, num_seqs, total_tokens);
    if (prefill_tc_supported(dk, dv, dtype)) return prefill_tc_workspace_bytes(H, num_seqs, total_tokens);
    return L.plan_bytes + (size_t)L.max_chunks * (size_t)H * L.chunk_bytes;
}

cudaError_t launch_prefill(const PrefillParams &p, int dtype, cudaStream_t st) {
    if (prefill_tc_supported(p.dk, p.dv, dtype)) {
        // tensor-core path: the plan validates cu_seqlens and numbers the
        // chunks, the prep kernel builds every chunk's operands, the chain
        // kernel walks them
        prefill::plan_kernel<<<1, 32, 0, st>>>(p.cu_seqlens, p.num_seqs, p.total_tokens,
                                               static_cast<int32_t *>(p.workspace), p.err_flag);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_prefill_tc(p, st);
    }
    if (dtype == KDA_DT_BF16) return prefill::launch_dtype<__nv_bfloat16>(p, st);
    return prefill::launch_dtype<float>(p, st);
}

}  // namespace kda
