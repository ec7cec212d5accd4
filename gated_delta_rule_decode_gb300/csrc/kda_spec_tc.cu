// ReplaySSM verify with the row phase on tcgen05 (bf16 inputs, dk = dv = 128,
// draft windows of up to 8 tokens: the benchmarked shape).
//
// "2.8x faster Kimi K3 inference on CANN", section 04 "ReplaySSM": verify
// keeps only the per-token update records and the outputs of every draft
// token; it never writes the pool.
//
// The window is evaluated in chunk form over the committed state S0 (the
// algebra is written out in kda_window.cuh).  Its dense part, the 2D dot
// products of every state row with the decayed keys K~_j and queries Q~_j,
// is one tensor-core product per (sequence, head):
//   D[i][j] = S0[i] . K~_j,  D[i][8 + j] = S0[i] . Q~_j   (M = 128 rows,
//   N = 16, K = 128 channels, kind::tf32, fp32 accumulate in TMEM).
// S0 arrives by TMA (four 128-byte-swizzled boxes of 32 channels x 128 rows,
// exactly the K-major layout the MMA reads), so it never passes through
// registers.  The token coefficients, the window products and the scalar
// recurrence run on the CUDA cores as in the general kernel; the key and
// beta records come from the decode kernel's routine, bit for bit.
#include <cudaTypedefs.h>
#include <stdint.h>

#include "kda.h"
#include "kda_bulk.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"
#include "kda_window.cuh"

namespace kda {
namespace verify_tc {

constexpr int DK = 128;
constexpr int kThreads = 256;
constexpr int kDraft = 8;
constexpr uint32_t kTmemCols = 32;
constexpr uint32_t kStateBytes = 128 * DK * 4;

struct Smem {
    unsigned char st[4][128 * 128];  // S0: 4 channel atoms of [128 rows][128 B], 128B-swizzled
    unsigned char kq[4][16 * 128];   // [K~ rows 0..7; Q~ rows 8..15], same layout
    float kh[kDraft][DK];
    float qh[kDraft][DK];
    float al[kDraft][DK];
    float A[kDraft][kDraft];
    float P[kDraft][kDraft];
    float beta[kDraft];
    float v[kDraft][kMaxDv];
    float o[kDraft][kMaxDv];
    uint64_t sbar;  // S0 landed
    uint64_t mbar;  // product done
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment of the swizzled tiles

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Row `row` of the 16-row swizzled B tile: this lane's four float4 slots
// (channels 4l + 32a .. 4l + 32a + 3 sit in channel atom a, 16-byte chunk l).
__device__ __forceinline__ void store_b_row(unsigned char *tile, int row, int l, const LaneVec<DK> &x) {
#pragma unroll
    for (int a = 0; a < DK / 32; ++a)
        *reinterpret_cast<float4 *>(tile + a * 16 * 128 + row * 128 + ((l ^ (row & 7)) << 4)) =
            make_float4(x.v[2 * a].x, x.v[2 * a].y, x.v[2 * a + 1].x, x.v[2 * a + 1].y);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) verify_tc_kernel(const VerifyParams p,
                                                                const __grid_constant__ CUtensorMap smap) {
    extern __shared__ unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int sh = blockIdx.x;  // (sequence, head)
    const int h = sh % p.H, n = sh / p.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, l = lane & 7;
    const int gid = warp * kGroupsPerWarp + grp;
    const int ngroups = kThreads / 8;
    const int D = p.D;

    const int slot = __ldg(p.slot_ids + n);
    const bool valid = slot >= 0 && (int64_t)slot < p.num_slots;
    if (slot >= 0 && !valid && tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_SLOT);

    if (warp == 0) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid == 0) {
        mbar_init(&sm.sbar, 1);
        mbar_init(&sm.mbar, 1);
        fence_barrier_init();
    }

    // token coefficients (3D group tasks) while the value rows load
    ValueVecs<T> vv;
    window_values_load<T>(p, n, h, tid, kThreads, vv);
    for (int base = 0; base < 3 * D; base += ngroups) {
        if (base + warp * kGroupsPerWarp >= 3 * D) break;  // warp-uniform
        window_coeffs<DK, T>(p, n, h, base + gid, base + gid < 3 * D, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0],
                             sm.beta);
    }
    // S0 is requested only now: issued first, its 64 KB queued ahead of the
    // coefficient loads (measured 95.5 us per launch against 88.3 us this way)
    if (tid == 0 && valid) {
        mbar_arrive_expect_tx(&sm.sbar, kStateBytes);
        const int z = slot * p.H + h;
#pragma unroll
        for (int a = 0; a < 4; ++a) tma_load_3d(sm.st[a], &smap, 32 * a, 0, z, &sm.sbar);
    }
    window_values_store<T>(p, n, h, tid, kThreads, vv, &sm.v[0][0]);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // window products; K~ and Q~ go straight into the MMA's B tile
    const int ntasks = D + D * (D - 1) / 2;
    auto store_kq = [&](float *, float *, int j, int ll, const LaneVec<DK> &kj, const LaneVec<DK> &qj) {
        store_b_row(&sm.kq[0][0], j, ll, kj);
        store_b_row(&sm.kq[0][0], kDraft + j, ll, qj);
    };
    for (int base = 0; base < ntasks; base += ngroups) {
        if (base + warp * kGroupsPerWarp >= ntasks) break;  // warp-uniform
        window_pair<DK>(base + gid, base + gid < ntasks, D, l, &sm.kh[0][0], &sm.qh[0][0], &sm.al[0][0], nullptr,
                        nullptr, &sm.A[0][0], &sm.P[0][0], kDraft, store_kq);
    }
    fence_proxy_async_smem();  // the B tile is read by the tensor core
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem_base;

    bool ok = true;
    bool mma_issued = false;
    if (valid) {
        // the outcome of every wait is made CTA-uniform
        ok = __syncthreads_and(mbar_wait(&sm.sbar, 0)) != 0;
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
            mma_issued = true;
            ok = __syncthreads_and(mbar_wait(&sm.mbar, 0)) != 0;
            tc::fence_after_sync();
        }
        if (ok && warp < 4) {
            // TMEM lane = state row i = tid
            float d[16];
            tc::ld16(tc::lane_addr(tm, warp, 0), d);
            tc::wait_ld();
            const int row = tid;
            float u[kDraft];
#pragma unroll
            for (int j = 0; j < kDraft; ++j) {
                u[j] = 0.f;
                if (j < D) {
                    float r = d[j];
#pragma unroll
                    for (int m = 0; m < j; ++m) r = __fmaf_rn(sm.A[j][m], u[m], r);
                    u[j] = __fmul_rn(sm.beta[j], __fsub_rn(sm.v[j][row], r));
                    float c = d[kDraft + j];
#pragma unroll
                    for (int m = 0; m <= j; ++m) c = __fmaf_rn(sm.P[j][m], u[m], c);
                    sm.o[j][row] = __fmul_rn(p.scale, c);
                }
            }
        }
        if (!ok) {
            if (tid == 0 && p.err_flag) atomicOr(p.err_flag, KDA_DEVERR_TIMEOUT);
            // bounded second chances: no copy or product may still be running
            mbar_wait(&sm.sbar, 0);
            if (mma_issued) mbar_wait(&sm.mbar, 0);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    window_store<T>(p, n, h, tid, kThreads, &sm.o[0][0], valid && ok);
    if (warp == 0) tc::tmem_dealloc(tm, kTmemCols);
}

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_fn() {
    static const EncodeTiled fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

}  // namespace verify_tc

bool verify_tc_supported(const VerifyParams &p, int dk, int dtype) {
    return dtype == KDA_DT_BF16 && dk == verify_tc::DK && p.dv == 128 && p.D <= verify_tc::kDraft &&
           p.num_slots > 0 && p.num_slots * (int64_t)p.H <= 0x7fffffffLL && verify_tc::encode_fn() != nullptr;
}

cudaError_t launch_verify_tc(const VerifyParams &p, cudaStream_t st) {
    using namespace verify_tc;
    // the pool as [num_slots * H][dv][dk] fp32; one box = 32 channels x 128 rows
    CUtensorMap map;
    const cuuint64_t dims[3] = {(cuuint64_t)DK, 128, (cuuint64_t)p.num_slots * (cuuint64_t)p.H};
    const cuuint64_t strides[2] = {(cuuint64_t)DK * 4, (cuuint64_t)128 * DK * 4};
    const cuuint32_t box[3] = {32, 128, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(p.pool), dims,
                                   strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)p.batch * p.H;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    verify_tc_kernel<__nv_bfloat16><<<(unsigned)grid, kThreads, kSmemBytes, st>>>(p, map);
    return cudaGetLastError();
}

}  // namespace kda
