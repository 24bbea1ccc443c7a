// mma_pair_sm103.cu -- the CTA-pair form of the tensor-core product against the
// single-CTA form the attention kernels use.
//
// PDC Lecture 7 §7.13 (CTA pair / MMA.2SM): two CTAs of a cluster on two SMs run
// one product together.  A single thread of the even CTA issues
// tcgen05.mma.cta_group::2 with M = 256: rows 0-127 of A come from the even
// CTA's shared memory and rows 128-255 from the odd CTA's, at the same offset;
// B's N rows are split the same way (N/2 from each CTA); each CTA's Tensor
// Memory receives its own 128 rows of D.  Tensor Memory is allocated and freed
// by one warp of each CTA together (the cta_group::2 forms of tcgen05.alloc and
// tcgen05.dealloc), and a commit can signal the barriers of both CTAs at once
// (multicast over the cluster).
//
// Two kernels:
//   * attn_pair_product_kernel -- D = A Bᵀ for A 256 x 64 and B 128 x 64 (bf16)
//     by four pair products, read back from both CTAs' Tensor Memory, so a test
//     can check the operand split against a host matrix product;
//   * attn_mma_rate_kernel<kPair, kWaits, kWarp> -- the sustained issue rate of
//     either form: the issuer issues `steps` groups of eight 128 x 128 x 16
//     (cta_group::1) or 256 x 128 x 16 (cta_group::2) products, with or
//     without a barrier wait in its loop (after group s, wait for group s-1:
//     the dependency depth of the attention kernels' pipelines), as a lone
//     lane or as a converged warp whose elected lane issues, and optionally
//     with eight more warps per CTA running a softmax-like loop (Tensor
//     Memory loads, packed fp32 FMA, exponentials, bf16 packs: two warps on
//     every SM sub-partition, as the attention kernels place their softmax
//     warps).
// Each product of either form keeps every SM's tensor core busy for 64 cycles,
// so the issuing thread's cycles per product give the tensor-busy fraction.
//
// Every wait is bounded (mbar_wait); a wait that runs out sets a bit in
// g_pair_error and the kernel still frees its Tensor Memory on the common path.
#include <cooperative_groups.h>

#include <algorithm>
#include <vector>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

namespace cg = cooperative_groups;

__device__ unsigned int g_pair_error = 0;

namespace {

constexpr int kTileRows = 128;     // rows of A per CTA
constexpr int kBRowsPair = 64;     // rows of B per CTA in the pair form (N / 2)
constexpr int kK = 64;             // reduction length: one 128-byte swizzle row of bf16
constexpr int kRowBytes = kK * 2;  // 128
constexpr int kTileBytes = kTileRows * kRowBytes;  // 16 KB
constexpr int kProductN = 128;
constexpr uint32_t kRateCols = 512;     // the whole Tensor Memory of the SM
constexpr uint32_t kProductCols = 128;
constexpr uint32_t kBusyMaxIters = 1u << 20;  // busy warps stop after this many at most
constexpr int kRateThreads = 384;       // 12 warps, as attn_fwd
constexpr int kRateSmemBytes = 160 * 1024;  // > half an SM's shared memory: one CTA per SM

// ---- cta_group::2 forms (the attention kernels use only cta_group::1; a kernel
// uses one of the two throughout)

template <uint32_t kCols>
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <uint32_t kCols>
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kCols)
                 : "memory");
}

__device__ __forceinline__ void umma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at offset `bar` of every CTA in `cta_mask` when
// the products this thread issued before have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Write `rows` rows of a row-major bf16 matrix (kK columns) into shared memory
// in the 128-byte-swizzled K-major layout the product descriptors describe:
// 16-byte chunk c of row r lands at r * 128 + ((c ^ (r % 8)) * 16).
__device__ void stage_swizzled(uint8_t* dst, const uint4* src, int rows) {
    for (int i = threadIdx.x; i < rows * 8; i += blockDim.x) {
        const int r = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(dst + r * kRowBytes + ((c ^ (r & 7)) << 4)) = src[i];
    }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace

// D (256 x 128 fp32, row-major) = A (256 x 64) · Bᵀ (B 128 x 64), bf16 row-major.
// One cluster of two CTAs, 128 threads each.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    attn_pair_product_kernel(const uint4* __restrict__ a, const uint4* __restrict__ b,
                             float* __restrict__ d) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sA = smem;                  // 128 rows of A
    uint8_t* sB = smem + kTileBytes;     // 64 rows of B (room for 128)
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * kTileBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 2 * kTileBytes + 8);

    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    stage_swizzled(sA, a + rank * kTileRows * 8, kTileRows);
    stage_swizzled(sB, b + rank * kBRowsPair * 8, kBRowsPair);
    fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's reads
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(bar), 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc_pair<kProductCols>(smem_addr(tmem_slot));
    tc_fence_before();
    cg::this_cluster().sync();  // both CTAs staged, barriers initialised, TMEM held
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (rank == 0 && threadIdx.x == 0) {
        const uint32_t idesc = umma_idesc_bf16(2 * kTileRows, kProductN, false);
        const uint64_t da = umma_desc_sw128(smem_addr(sA), 16, 1024);
        const uint64_t db = umma_desc_sw128(smem_addr(sB), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kK / 16; ++kk)  // 32 bytes of each row per product
            umma_ss_pair(tmem, da + kk * 2, db + kk * 2, idesc, kk > 0 ? 1u : 0u);
        umma_commit_pair(smem_addr(bar), 0x3);
    }
    if (!mbar_wait(smem_addr(bar), 0)) atomicOr(&g_pair_error, kErrBitTimeout);
    tc_fence_after();

    // each warp reads its lane quarter of this CTA's 128 rows
    const int row = rank * kTileRows + warp * 32 + lane;
    float* drow = d + static_cast<size_t>(row) * kProductN;
#pragma unroll
    for (int c = 0; c < kProductN; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) drow[c + j] = __uint_as_float(r[j]);
    }
    tc_fence_before();
    cg::this_cluster().sync();  // neither CTA frees the pair's columns while the other reads
    if (warp == 0) tmem_dealloc_pair<kProductCols>(tmem);
}

// The issue-rate kernel.  kPair: cta_group::2 products issued by the even CTA
// of each cluster (launched with a cluster of 2); otherwise cta_group::1 products
// issued in every CTA.  kWaits: the loop waits for group s-1 after issuing group
// s.  kWarp: all 32 lanes of warp 0 run the loop and the waits and the lane
// elect_one() picks issues; otherwise lane 0 alone.  cycles[i] receives issuing
// CTA i's clock64 cycles from its first product to the completion of its last.
template <bool kPair, bool kWaits, bool kWarp>
__global__ void __launch_bounds__(kRateThreads, 1)
    attn_mma_rate_kernel(int steps, int busy, long long* __restrict__ cycles,
                         unsigned* __restrict__ sink) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kTileBytes);  // step0, step1, done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 2 * kTileBytes + 32);
    volatile uint32_t* stop_flag = reinterpret_cast<volatile uint32_t*>(smem + 2 * kTileBytes + 36);

    const uint32_t rank = kPair ? cluster_rank() : 0u;
    const bool issuer_cta = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // operands: zeros (the rate does not depend on the values)
    for (int i = threadIdx.x; i < 2 * kTileBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(smem_addr(&bars[i]), 1);
        *stop_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        if constexpr (kPair) tmem_alloc_pair<kRateCols>(smem_addr(tmem_slot));
        else tmem_alloc<kRateCols>(smem_addr(tmem_slot));
    }
    tc_fence_before();
    if constexpr (kPair) cg::this_cluster().sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (issuer_cta && (kWarp || lane == 0)) {
            const uint32_t idesc = umma_idesc_bf16(kPair ? 2 * kTileRows : kTileRows, kProductN, false);
            const uint64_t da = umma_desc_sw128(smem_addr(sA), 16, 1024);
            const uint64_t db = umma_desc_sw128(smem_addr(sB), 16, 1024);
            auto wait = [&](uint32_t bar, uint32_t parity) {
                const bool w = mbar_wait(bar, parity);
                return kWarp ? __all_sync(0xffffffffu, w) : w;
            };
            const long long t0 = clock64();
            bool ok = true;
            for (int s = 0; s < steps && ok; ++s) {
                if (!kWarp || elect_one()) {
                    // eight products into two 128-column accumulators, as one
                    // key-tile step of one query tile issues (S = Q Kᵀ, O += P V)
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        const uint32_t dst = tmem + static_cast<uint32_t>((p >> 2) * 128);
                        const int kk = p & 3;
                        if constexpr (kPair) umma_ss_pair(dst, da + kk * 2, db + kk * 2, idesc, 1u);
                        else umma_ss(dst, da + kk * 2, db + kk * 2, idesc, 1u);
                    }
                    const uint32_t sb = smem_addr(&bars[s & 1]);
                    if constexpr (kPair) umma_commit_pair(sb, 0x1);
                    else umma_commit(sb);
                }
                if constexpr (kWarp) __syncwarp();
                if constexpr (kWaits)
                    if (s >= 1) ok = wait(smem_addr(&bars[(s - 1) & 1]), ((s - 1) >> 1) & 1);
            }
            const uint32_t db_done = smem_addr(&bars[2]);
            if (!kWarp || elect_one()) {
                if constexpr (kPair) umma_commit_pair(db_done, 0x3);
                else umma_commit(db_done);
            }
            if constexpr (kWarp) __syncwarp();
            ok = wait(db_done, 0) && ok;
            const long long t1 = clock64();
            if (lane == 0) {
                if (!ok) atomicOr(&g_pair_error, kErrBitTimeout);
                cycles[kPair ? blockIdx.x / 2 : blockIdx.x] = t1 - t0;
                *stop_flag = 1;
            }
        } else if (!issuer_cta && lane == 0) {
            // the odd CTA of a pair: its tensor core and Tensor Memory take the
            // even CTA's products; wait for the last one
            if (!mbar_wait(smem_addr(&bars[2]), 0)) atomicOr(&g_pair_error, kErrBitTimeout);
            *stop_flag = 1;
        }
        __syncwarp();
    } else if (warp >= 4 && busy) {
        // softmax-like work on this warp's lane quarter, columns 256-511 (the
        // products write columns 0-255 only)
        const uint32_t quarter = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t acc = 0;
        const float2 scale = make_float2(0.18f, 0.18f), shift = make_float2(-3.0f, -3.0f);
        for (uint32_t it = 0; it < kBusyMaxIters; ++it) {
            if (*stop_flag) break;
            uint32_t r[32];
            tmem_ld32(tmem + quarter + 256 + 32 * (it & 7), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                float2 v = make_float2(__uint_as_float(r[j] & 0x3fffffffu),
                                       __uint_as_float(r[j + 1] & 0x3fffffffu));
                v = ffma2(v, scale, shift);
                acc ^= pack_bf16x2(ex2_approx(v.x), ex2_approx(v.y));
            }
        }
        if (acc == 0x9e3779b9u) sink[0] = acc;  // keeps the loop's work; practically never written
    }
    tc_fence_before();
    if constexpr (kPair) cg::this_cluster().sync();
    else __syncthreads();
    if (warp == 0) {
        if constexpr (kPair) tmem_dealloc_pair<kRateCols>(tmem);
        else tmem_dealloc<kRateCols>(tmem);
    }
}

namespace {

int read_and_clear_pair_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_pair_error, sizeof v) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_pair_error, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
    return v ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

constexpr int kProductSmemBytes = 2 * kTileBytes + 64 + 1024;

}  // namespace

int launch_pair_product(const void* a, const void* b, float* d, cudaStream_t stream) {
    if (cudaFuncSetAttribute(attn_pair_product_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kProductSmemBytes) != cudaSuccess)
        return ATTN_ERR_CUDA;
    attn_pair_product_kernel<<<2, 128, kProductSmemBytes, stream>>>(
        static_cast<const uint4*>(a), static_cast<const uint4*>(b), d);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return read_and_clear_pair_error();
}

using RateKernel = void (*)(int, int, long long*, unsigned*);

template <bool kPair>
RateKernel rate_kernel(int waits, int issuer) {
    if (waits) return issuer ? attn_mma_rate_kernel<kPair, true, true> : attn_mma_rate_kernel<kPair, true, false>;
    return issuer ? attn_mma_rate_kernel<kPair, false, true> : attn_mma_rate_kernel<kPair, false, false>;
}

int run_mma_rate(int form, int issuer, int busy, int waits, int steps, int reps, float* ms_out,
                 double* cycles_out, int* sms_out, cudaStream_t stream) {
    const bool pair = form == 2;
    const RateKernel kern = pair ? rate_kernel<true>(waits, issuer) : rate_kernel<false>(waits, issuer);
    const RateKernel probe = attn_mma_rate_kernel<true, false, false>;  // occupancy query
    for (RateKernel k : {kern, probe})
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmemBytes) !=
            cudaSuccess)
            return ATTN_ERR_CUDA;

    // the same SMs for both forms: as many CTA pairs as fit at once
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kRateThreads);
    cfg.dynamicSmemBytes = kRateSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int sms = 0;
    if (current_sm_count(&sms) != ATTN_OK || sms < 2) return ATTN_ERR_CUDA;
    cfg.gridDim = dim3(sms & ~1);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, probe, &cfg) != cudaSuccess ||
        clusters <= 0) {
        (void)cudaGetLastError();  // not sticky: leave no error for the next call
        return ATTN_ERR_CUDA;
    }
    clusters = std::min(clusters, sms / 2);
    const int ctas = 2 * clusters;
    cfg.gridDim = dim3(ctas);
    cfg.numAttrs = pair ? 1 : 0;
    const int issuers = pair ? clusters : ctas;

    long long* d_cycles = nullptr;
    unsigned* d_sink = nullptr;
    if (cudaMalloc(&d_cycles, sizeof(long long) * issuers) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMalloc(&d_sink, sizeof(unsigned)) != cudaSuccess) {
        cudaFree(d_cycles);
        return ATTN_ERR_CUDA;
    }
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    int rc = ATTN_OK;
    float total_ms = 0.0f;
    double total_cycles = 0.0;
    std::vector<long long> h(issuers);
    for (int rep = -1; rep < reps && rc == ATTN_OK; ++rep) {  // rep -1 warms up
        cudaEventRecord(e0, stream);
        if (cudaLaunchKernelEx(&cfg, kern, steps, busy, d_cycles, d_sink) != cudaSuccess) {
            rc = ATTN_ERR_CUDA;
            break;
        }
        cudaEventRecord(e1, stream);
        if (cudaEventSynchronize(e1) != cudaSuccess) {
            rc = ATTN_ERR_CUDA;
            break;
        }
        rc = read_and_clear_pair_error();
        if (rc != ATTN_OK || rep < 0) continue;
        float ms = 0.0f;
        cudaEventElapsedTime(&ms, e0, e1);
        total_ms += ms;
        if (cudaMemcpy(h.data(), d_cycles, sizeof(long long) * issuers, cudaMemcpyDeviceToHost) !=
            cudaSuccess) {
            rc = ATTN_ERR_CUDA;
            break;
        }
        double s = 0.0;
        for (long long c : h) s += static_cast<double>(c);
        total_cycles += s / issuers;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(d_cycles);
    cudaFree(d_sink);
    if (rc != ATTN_OK) return rc;
    *ms_out = total_ms / reps;
    if (cycles_out) *cycles_out = total_cycles / reps;
    if (sms_out) *sms_out = ctas;
    return ATTN_OK;
}

}  // namespace gbattn
