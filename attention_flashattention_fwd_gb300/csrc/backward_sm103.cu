// backward_sm103.cu -- FlashAttention backward for sm_103a.
//
// What it computes is the backward pass of the CS336 Lecture 5 notes,
// section 8.4 (the FlashAttention-2 form): the forward stores no P; it is
// recomputed as P_ij = e^{S_ij - L_i} from the logsumexp L, and with
// D_i = rowsum(dO_i * O_i) (exercise 9 of the same notes)
//     dV_j += P_ij^T dO_i,   dP_ij = dO_i V_j^T,   dS_ij = P_ij * (dP_ij - D_i),
//     dQ_i += scale dS_ij K_j,   dK_j += scale dS_ij^T Q_i.
//
// Three kernels, in stream order:
//   * prep: -D_i and -L_i log2(e) for every query row (negated for the fused
//     multiply-adds that use them), padded to whole 128-row tiles (padded rows
//     get D = 0 and L = +inf, so their P is 0), and a zeroed fp32 dQ
//     accumulator;
//   * main: one CTA per (b, h, 128-key tile j), key/value-outer as in the
//     notes' FlashAttention-2 form.  K_j and V_j stay in shared memory; for
//     every query tile i that can see the key tile, TMA brings Q_i and dO_i
//     (two-stage ring) and tcgen05.mma computes, with one thread per key row
//     (= one Tensor Memory lane) in the softmax warpgroup:
//         S^T = K_j Q_i^T,  dP^T = V_j dO_i^T            (into Tensor Memory)
//         P^T = 2^{S^T c - L log2 e},  dS^T = P^T (dP^T - D)   (registers)
//         dV_j += P^T dO_i,  dK_j += dS^T Q_i              (A operand in TMEM)
//         dQ_i  = dS K_j                                   (A = dS in shared memory)
//     and a second warpgroup adds dQ_i into the fp32 accumulator with TMA
//     bulk reduce-adds, staged through the dS tile once dQ_i has read it;
//   * convert: dQ = scale * accumulator, rounded to bf16.
// Working transposed (a thread owns a key row) keeps the dV and dK products'
// A operands in Tensor Memory and makes the row statistics L_i and D_i
// per-column values that every thread reads at the same address.
#include <cuda_bf16.h>
#include <cuda.h>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

__device__ unsigned int g_bwd_error = 0;

// Error bit of the backward kernel: its shared-memory layout did not fit.
constexpr unsigned kErrLayout = 2u;

namespace {

constexpr int kTile = 128;       // keys per CTA, queries per step
constexpr int kThreads = 384;    // warps 0-3 key rows, 4-7 dQ rows, 8 MMA, 9 TMA, 10-11 idle
// Register split.  The launch gives each thread 168 registers (65536 / 384,
// rounded down to 8); the key-row warpgroup (P and dS) and the dQ warpgroup
// (all of dQ_i in registers) take more from the control warpgroup:
// 128 x 240 + 128 x 152 + 128 x 96 = 62464 <= 384 x 168 = 64512.
constexpr uint32_t kKeyRowRegs = 240;
constexpr uint32_t kDqRegs = 152;
constexpr uint32_t kCtrlRegs = 96;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct BCfg {
    static constexpr int kSub = D / 64;               // 128-byte swizzle atoms along d
    static constexpr int kSubBytes = 128 * 128;       // one atom column: 128 rows x 128 B
    static constexpr int kTileBytes = kTile * D * 2;  // a 128-row bf16 tile of K, V, Q or dO
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTileBytes;
    static constexpr int kRingOff = 2 * kTileBytes;   // stage s: Q_i, then dO_i
    static constexpr int kDsOff = kRingOff + 4 * kTileBytes;  // dS, 128 keys x 128 queries bf16
    // stage s: -L log2(e) and -D of the stage's 128 queries (fp32, 512 B each)
    static constexpr int kLdOff = kDsOff + 2 * kSubBytes;
    static constexpr int kTilesBytes = kLdOff + 2 * 1024;
    // Barriers, the TMEM address slot and the abort flag (128 bytes) go into
    // the gap below the 1024-byte aligned tiles when it has room, else after
    // them.  The dynamic shared memory base is 16-byte aligned, so the gap is
    // at most 1008 bytes: the allocation covers both cases.
    static constexpr int kNumBars = 14;
    static constexpr int kSmallBytes = 128;
    static constexpr int kSmemBytes =
        kTilesBytes + (1008 > kSmallBytes + 80 ? 1008 : kSmallBytes + 80);
    // Tensor Memory columns.  S^T is overwritten by P^T (bf16 pairs, first 64
    // columns); dP^T by dS^T (bf16 pairs, first 64 columns) and, once the dK
    // product has read dS^T, by the dQ_i product.
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColDP = 128;
    static constexpr uint32_t kColDQ = 128;
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
};
static_assert(BCfg<128>::kSmemBytes <= 232448, "shared memory of one CTA");
static_assert(BCfg<128>::kNumBars * 8 + 8 <= BCfg<128>::kSmallBytes, "small objects");

struct BBars {
    uint32_t base;
    __device__ uint32_t kv_full() const { return base; }
    __device__ uint32_t q_full(int s) const { return base + 8u * (1 + s); }
    __device__ uint32_t q_empty(int s) const { return base + 8u * (3 + s); }
    __device__ uint32_t s_full() const { return base + 8u * 5; }    // S^T in TMEM
    __device__ uint32_t dp_full() const { return base + 8u * 6; }   // dP^T in TMEM
    __device__ uint32_t pa_ready() const { return base + 8u * 7; }  // P^T written
    __device__ uint32_t pb_tmem() const { return base + 8u * 8; }   // dS^T written (TMEM)
    __device__ uint32_t pb_smem() const { return base + 8u * 9; }   // dS tile written (smem)
    __device__ uint32_t dq_full() const { return base + 8u * 10; }  // dQ_i in TMEM
    __device__ uint32_t dq_free() const { return base + 8u * 11; }  // dQ_i out of TMEM
    __device__ uint32_t ds_free() const { return base + 8u * 12; }  // dS tile free again
    __device__ uint32_t done() const { return base + 8u * 13; }
};

__device__ __forceinline__ void flag_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_bwd_error, kErrTimeout);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                flag_abort(abort_flag);
                return false;
            }
        }
    }
}

// The same wait run by every lane of the MMA warp, its result made
// warp-uniform so that no lane leaves the warp's loops alone.
__device__ __forceinline__ bool wait_uniform(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
}

// Wait for this thread's Tensor Memory loads into `a` and `b`; the registers
// are tied to the wait so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_into(uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
          "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]),
          "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]),
          "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]),
          "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]),
          "+r"(a[31]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]),
          "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]),
          "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]),
          "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]),
          "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]),
          "+r"(b[30]), "+r"(b[31])
        :
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld_into(uint32_t (&a)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
          "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]),
          "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]),
          "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]),
          "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]),
          "+r"(a[31])
        :
        : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the
// tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared completing `bar`'s transaction count
// (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Ties registers to the preceding tcgen05.wait::ld without emitting code, so
// no use of them is scheduled above that wait.
__device__ __forceinline__ void after_wait_ld(uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile(""
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                   "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                   "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]),
                   "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]),
                   "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]),
                   "+r"(a[30]), "+r"(a[31]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]),
                   "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]),
                   "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]),
                   "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]),
                   "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]),
                   "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
                 :
                 : "memory");
}

// Element-wise product of fp32 pairs (one packed instruction).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// Barrier 1 among the 128 threads of the dQ warpgroup (barrier 0 is
// __syncthreads).
__device__ __forceinline__ void dq_group_sync() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// AND of `ok` over the 128 threads of the dQ warpgroup (barrier 1 with a
// reduction): every warp of the group takes the same branch after a bounded
// wait, so none can be left alone at a later `bar.sync 1`.
__device__ __forceinline__ bool dq_group_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(ok))
        : "memory");
    return r != 0;
}

// Element-wise add of a shared-memory box into global memory through the
// tensor map (TMA reduce), tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int x, int y,
                                                  int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The shared-memory sources of this thread's committed bulk copies have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// All but the most recent of this thread's committed bulk copies have read
// their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// This thread's committed bulk copies have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Instruction descriptor with A in MN-major (transposed) layout as well.
__host__ __device__ constexpr uint32_t idesc_bf16_a_mn(uint32_t M, uint32_t N) {
    return umma_idesc_bf16(M, N, true) | (1u << 15);
}

__device__ __forceinline__ uint4 bf16x8(const float* x) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

}  // namespace

// ----------------------------------------------------------------- prep kernel
//
// Row i of head bh (i < Nq_pad): -D_i with D_i = sum_c dO_ic O_ic in fp32 and
// -lse_i log2(e); rows i >= Nq get 0 and -inf.  The fp32 dQ
// accumulator row is zeroed.  D / 8 consecutive threads share a row (16-byte
// loads); the trip count is rounded up to whole warps so the row sum's
// shuffles always see the full warp.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(BwdPrepParams a) {
    constexpr int kLanes = D / 8;
    const long long total = a.rows * kLanes;
    const long long padded = (total + 31) / 32 * 32;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < padded;
         g += stride) {
        const bool valid = g < total;
        const long long row = g / kLanes;
        const int c = static_cast<int>(g % kLanes);
        const long long bh = row / a.Nq_pad;
        const int i = static_cast<int>(row % a.Nq_pad);
        float acc = 0.f;
        const long long n_rows_q = a.rows / a.Nq_pad * a.Nq;  // B H Nq rows of o, dO, lse
        const long long off_q = (bh * a.Nq + i) * D + c * 8;
        if (valid && i < a.Nq && gb_index_ok(&g_bwd_error, off_q, off_q + 7, n_rows_q * D)) {
            const size_t off = static_cast<size_t>(off_q);
            const uint4 ov = *reinterpret_cast<const uint4*>(a.o + off);
            const uint4 dv = *reinterpret_cast<const uint4*>(a.dout + off);
            const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
            const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 of = __bfloat1622float2(o2[t]);
                const float2 df = __bfloat1622float2(d2[t]);
                acc = fmaf(of.x, df.x, acc);
                acc = fmaf(of.y, df.y, acc);
            }
        }
#pragma unroll
        for (int sh = kLanes / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
        if (valid && gb_index_ok(&g_bwd_error, row * D + c * 8, row * D + c * 8 + 7, a.rows * D)) {
            float4* z = reinterpret_cast<float4*>(a.dq_acc + row * D + c * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c == 0) {
                a.nD[row] = -acc;
                const bool lse_ok = i < a.Nq && gb_index_ok(&g_bwd_error, bh * a.Nq + i,
                                                            bh * a.Nq + i, n_rows_q);
                a.nl2[row] = lse_ok
                                 ? a.lse[static_cast<size_t>(bh) * a.Nq + i] * -1.4426950408889634f
                                 : -INFINITY;
            }
        }
    }
}

// ----------------------------------------------------------------- main kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dqacc, BwdParams p) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int gap = static_cast<int>(smem - smem_raw);
    uint8_t* small = gap >= C::kSmallBytes ? smem - C::kSmallBytes : smem + C::kTilesBytes;
    if (gap + C::kTilesBytes + (gap >= C::kSmallBytes ? 0 : C::kSmallBytes) > C::kSmemBytes) {
        // the base was less aligned than assumed: report and do nothing
        if (threadIdx.x == 0) atomicOr(&g_bwd_error, kErrLayout);
        return;
    }
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sK = sbase + C::kKOff;
    const uint32_t sV = sbase + C::kVOff;
    const uint32_t sRing = sbase + C::kRingOff;
    const uint32_t sDs = sbase + C::kDsOff;
    const uint32_t sLd = sbase + C::kLdOff;
    const BBars bars{smem_addr(small)};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(small + C::kNumBars * 8 + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work item: key tile j of head bh.  The grid runs through groups of
    // head_group heads; within a group, most query tiles (lowest j under a
    // causal mask) first, the group's heads side by side.  Key tile j is seen
    // by query q iff some key k of it has k <= q + causal_off, i.e. from
    // query tile (kj0 - off) / 128 on.
    const int per_group = p.head_group * p.n_kt;
    const int grp = static_cast<int>(blockIdx.x) / per_group;
    const int within = static_cast<int>(blockIdx.x) - grp * per_group;
    const int g_heads = min(p.head_group, p.BH - grp * p.head_group);
    const int j = within / g_heads;
    const int bh = grp * p.head_group + within % g_heads;
    const int kj0 = j * kTile;
    const int n_qt = p.Nq_pad / kTile;
    int i_first = 0;
    if (p.causal) {
        const int f = kj0 - p.causal_off;
        i_first = f > 0 ? f / kTile : 0;
    }
    const int n_iter = n_qt - i_first;  // >= 1: the last query sees every key

    // ---- set-up: barriers (one thread), Tensor Memory (warp 0)
    if (threadIdx.x == kLoadWarp * 32) {
        mbar_init(bars.kv_full(), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bars.q_full(s), 1);
            mbar_init(bars.q_empty(s), 1);
        }
        mbar_init(bars.s_full(), 1);
        mbar_init(bars.dp_full(), 1);
        mbar_init(bars.pa_ready(), 4);  // one arrival per key-row warp
        mbar_init(bars.pb_tmem(), 4);
        mbar_init(bars.pb_smem(), 4);
        mbar_init(bars.dq_full(), 1);
        mbar_init(bars.dq_free(), 4);   // one arrival per dQ warp
        mbar_init(bars.ds_free(), 1);   // the dQ warpgroup's TMA thread
        mbar_init(bars.done(), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc<kTmemCols>(smem_addr(tmem_slot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
    // ====================================================== control warpgroup
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == kLoadWarp) {
        // ===================================================== TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(bars.kv_full(), 2 * C::kTileBytes);
            for (int s = 0; s < C::kSub; ++s) {
                tma_load_3d(sK + s * C::kSubBytes, &tm_k, bars.kv_full(), s * 64, kj0, bh);
                tma_load_3d(sV + s * C::kSubBytes, &tm_v, bars.kv_full(), s * 64, kj0, bh);
            }
            bool ok = true;
            int issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it & 1;
                // the stage's previous tiles (step it - 2) have been read by their last product
                if (it >= 2 &&
                    !(ok = wait_or_abort(bars.q_empty(s), ((it >> 1) - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bars.q_full(s), 2 * C::kTileBytes + 1024);
                const uint32_t dst = sRing + s * 2 * C::kTileBytes;
                const int y = (i_first + it) * kTile;
                const size_t row0 = static_cast<size_t>(bh) * p.Nq_pad + y;
                // (debug builds: an out-of-range tile is not loaded; its stage
                // then never completes and the consumers' bounded waits report it)
                if (gb_index_ok(&g_bwd_error, static_cast<long long>(row0),
                                static_cast<long long>(row0) + 127,
                                static_cast<long long>(p.BH) * p.Nq_pad)) {
                    bulk_load(sLd + s * 1024, p.nl2 + row0, 512, bars.q_full(s));
                    bulk_load(sLd + s * 1024 + 512, p.nD + row0, 512, bars.q_full(s));
                }
                for (int sub = 0; sub < C::kSub; ++sub) {
                    tma_load_3d(dst + sub * C::kSubBytes, &tm_q, bars.q_full(s), sub * 64, y, bh);
                    tma_load_3d(dst + C::kTileBytes + sub * C::kSubBytes, &tm_do, bars.q_full(s),
                                sub * 64, y, bh);
                }
                ++issued;
            }
            if (!ok) {
                // drain: every copy in flight must land before the CTA exits
                mbar_wait(bars.kv_full(), 0);
                for (int it = max(0, issued - 2); it < issued; ++it)
                    mbar_wait(bars.q_full(it & 1), (it >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ===================================================== MMA issuer
        // Per step i (stage s), with S^T(i) issued during step i - 1:
        //   [dQ_{i-1} out of TMEM]  dP^T -> dp_full
        //   [P^T written]           dV += P^T dO_i
        //   [Q_{i+1} loaded]        S^T(i+1) -> s_full
        //   [dS^T written]          dK += dS^T Q_i -> q_empty(s)
        //   [dS tile written]       dQ_i = dS K_j -> dq_full
        // dQ_i lands in the dP^T columns after the dK product has read dS^T from
        // them, S^T(i+1) in the S^T columns after the dV product has read P^T
        // (one thread's MMAs run in issue order); only dP^T(i+1) waits for the
        // dQ warpgroup to have taken dQ_i.
        {  // the whole warp; elect_one() issues
            const uint32_t id_s = umma_idesc_bf16(kTile, kTile, false);  // both K-major
            const uint32_t id_acc = umma_idesc_bf16(kTile, D, true);     // B MN-major
            const uint32_t id_dq = idesc_bf16_a_mn(kTile, D);            // A and B MN-major
            const uint64_t dk_k = umma_desc_sw128(sK, 16, 1024);
            const uint64_t dv_k = umma_desc_sw128(sV, 16, 1024);
            const uint64_t dk_mn = umma_desc_sw128(sK, C::kSubBytes, 1024);
            const uint64_t dds_mn = umma_desc_sw128(sDs, C::kSubBytes, 1024);
            auto issue_s = [&](int it) {  // S^T = K_j Q_i^T, K = d in steps of 16
                const uint64_t dq_k = umma_desc_sw128(sRing + (it & 1) * 2 * C::kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kSubBytes + (kk & 3) * 32) >> 4;
                    umma_ss(tmem + C::kColS, dk_k + off, dq_k + off, id_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(bars.s_full());
            };
            bool ok = wait_uniform(bars.kv_full(), 0, abort_flag) &&
                      wait_uniform(bars.q_full(0), 0, abort_flag);
            if (ok) {
                tc_fence_after();
                if (elect_one()) issue_s(0);
                __syncwarp();
            }
            for (int it = 0; it < n_iter && ok; ++it) {
                const int s = it & 1;
                if (it > 0 && !(ok = wait_uniform(bars.dq_free(), (it - 1) & 1, abort_flag)))
                    break;
                tc_fence_after();
                const uint32_t sq = sRing + s * 2 * C::kTileBytes;
                const uint32_t sdo = sq + C::kTileBytes;
                const uint64_t ddo_k = umma_desc_sw128(sdo, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V_j dO_i^T
                        const uint32_t off = ((kk >> 2) * C::kSubBytes + (kk & 3) * 32) >> 4;
                        umma_ss(tmem + C::kColDP, dv_k + off, ddo_k + off, id_s, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bars.dp_full());
                }
                __syncwarp();
                const uint64_t dq_mn = umma_desc_sw128(sq, C::kSubBytes, 1024);
                const uint64_t ddo_mn = umma_desc_sw128(sdo, C::kSubBytes, 1024);
                // K = 128 queries in steps of 16: 8 packed P / dS columns, 16 rows of 128 B
                if (!(ok = wait_uniform(bars.pa_ready(), it & 1, abort_flag))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        umma_ts(tmem + C::kColDV, tmem + C::kColS + kk * 8,
                                ddo_mn + ((kk * 2048) >> 4), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
                // S^T(i+1) right behind the dV product that read P^T(i): the key-row
                // warps start on it as soon as they are done with dS(i)
                if (it + 1 < n_iter) {
                    if (!(ok = wait_uniform(bars.q_full((it + 1) & 1), ((it + 1) >> 1) & 1,
                                            abort_flag)))
                        break;
                    tc_fence_after();
                    if (elect_one()) issue_s(it + 1);
                    __syncwarp();
                }
                if (!(ok = wait_uniform(bars.pb_tmem(), it & 1, abort_flag))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        umma_ts(tmem + C::kColDK, tmem + C::kColDP + kk * 8,
                                dq_mn + ((kk * 2048) >> 4), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(bars.q_empty(s));
                }
                __syncwarp();
                if (!(ok = wait_uniform(bars.pb_smem(), it & 1, abort_flag))) break;
                tc_fence_after();
                if (elect_one()) {
                    // K = 128 keys in steps of 16 rows of the dS and K_j tiles
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        umma_ss(tmem + C::kColDQ, dds_mn + ((kk * 2048) >> 4),
                                dk_mn + ((kk * 2048) >> 4), id_dq, kk > 0 ? 1u : 0u);
                    umma_commit(bars.dq_full());
                }
                __syncwarp();
            }
            // every MMA the elected lane issued has completed once `done` flips
            if (elect_one()) umma_commit(bars.done());
            __syncwarp();
            mbar_wait(bars.done(), 0);
        }
        __syncwarp();
    }  // warps 10 and 11 have no role
    } else if (warp < 4) {
        setmaxnreg_inc<kKeyRowRegs>();
        // ===================================================== key rows: P^T, dS^T
        // Phase A (S^T in TMEM): P^T = 2^{S^T c - L}, kept as bf16 pairs in
        // registers and written over the first 64 columns of S^T (the dV
        // product's A operand).  Phase B (dP^T in TMEM): dS^T = P^T (dP^T - D)
        // from the bf16 P, written over the first 64 columns of dP^T (the dK
        // product's A operand) and as the dS tile in shared memory (the dQ
        // product's A operand).
        const int r = warp * 32 + lane;  // key row within the tile = TMEM lane
        const int key = kj0 + r;
        const bool key_ok = key < p.Nk;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::kColS;
        const uint32_t tDP = tmem + lane_off + C::kColDP;
        const float cl2 = p.scale_log2;
        const int first_vis = key - p.causal_off;  // causal: query q sees this key iff q >= first_vis
        bool ok = true;
        for (int it = 0; it < n_iter; ++it) {
            // the stage's L and D arrived with its Q and dO tiles (q_full)
            ok = wait_or_abort(bars.s_full(), it & 1, abort_flag) &&
                 wait_or_abort(bars.q_full(it & 1), (it >> 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int i0 = (i_first + it) * kTile;
            const bool diag = p.causal && (kj0 + kTile - 1 > i0 + p.causal_off);
            const float4* L4 = reinterpret_cast<const float4*>(smem + C::kLdOff + (it & 1) * 1024);
            const float4* D4 = L4 + 32;
            uint32_t pk[64];  // P^T row as bf16 pairs, 128 queries
            // ---- phase A: p = 2^{s c - L log2 e}, pairs of columns per instruction
            const float2 c2 = make_float2(cl2, cl2);
            {
                // the whole S^T row (128 queries): four loads in flight, one wait
                uint32_t sr[4][32];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tS + q4 * 32, sr[q4]);
                tmem_wait_ld_into(sr[0], sr[1]);
                after_wait_ld(sr[2], sr[3]);
#pragma unroll
                for (int c4 = 0; c4 < 32; ++c4) {  // four queries per shared-memory read
                    const float4 l4 = L4[c4];  // same address in every lane
                    const uint32_t* sv = sr[c4 >> 3] + (c4 & 7) * 4;
                    const float2 x0 = ffma2(make_float2(__uint_as_float(sv[0]), __uint_as_float(sv[1])),
                                            c2, make_float2(l4.x, l4.y));
                    const float2 x1 = ffma2(make_float2(__uint_as_float(sv[2]), __uint_as_float(sv[3])),
                                            c2, make_float2(l4.z, l4.w));
                    float pv[4] = {ex2_approx(x0.x), ex2_approx(x0.y), ex2_approx(x1.x),
                                   ex2_approx(x1.y)};
                    if (diag) {  // tiles that straddle the causal boundary
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (i0 + c4 * 4 + e < first_vis) pv[e] = 0.f;
                    }
                    pk[2 * c4] = pack_bf16x2(pv[0], pv[1]);
                    pk[2 * c4 + 1] = pack_bf16x2(pv[2], pv[3]);
                }
            }
            if (!key_ok) {  // rows past the last key
#pragma unroll
                for (int x = 0; x < 64; ++x) pk[x] = 0u;
            }
            // P^T over the first 64 columns of S^T (all of S^T has been read)
#pragma unroll
            for (int x = 0; x < 4; ++x)
                tmem_st16(tS + x * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[x * 16]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.pa_ready());
            // ---- phase B
            ok = wait_or_abort(bars.dp_full(), it & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t dk[64];  // dS^T row as bf16 pairs, 128 queries
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t d0[32], d1[32];
                tmem_ld32(tDP + hf * 64, d0);
                tmem_ld32(tDP + hf * 64 + 32, d1);
                tmem_wait_ld_into(d0, d1);
#pragma unroll
                for (int c2i = 0; c2i < 32; ++c2i) {  // pairs of columns
                    const float2 nd = reinterpret_cast<const float2*>(D4)[hf * 32 + c2i];  // -D, broadcast
                    const int c = 2 * c2i;
                    auto dv = [&](int e) { return __uint_as_float(c < 32 ? d0[c + e] : d1[c - 32 + e]); };
                    const uint32_t pp = pk[hf * 32 + c2i];
                    const float2 pe = make_float2(__uint_as_float(pp << 16),
                                                  __uint_as_float(pp & 0xffff0000u));
                    const float2 t = fadd2(make_float2(dv(0), dv(1)), nd);
                    const float2 ds = fmul2(pe, t);
                    dk[hf * 32 + c2i] = pack_bf16x2(ds.x, ds.y);
                }
                tmem_st16(tDP + hf * 32, *reinterpret_cast<uint32_t(*)[16]>(&dk[hf * 32]));
                tmem_st16(tDP + hf * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&dk[hf * 32 + 16]));
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.pb_tmem());
            // the dS tile, once the dQ warpgroup has added dQ_{i-1} out of it: the
            // MN-major A operand of dQ_i = dS K_j; row r holds 64 queries per 16 KB
            // half, its 16-byte chunks permuted by the 128-byte swizzle (chunk ^ (row % 8))
            if (it > 0) {
                ok = wait_or_abort(bars.ds_free(), (it - 1) & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint8_t* row = smem + C::kDsOff + hf * C::kSubBytes + r * 128;
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    *reinterpret_cast<uint4*>(row + ((x ^ (r & 7)) * 16)) =
                        make_uint4(dk[hf * 32 + 4 * x], dk[hf * 32 + 4 * x + 1],
                                   dk[hf * 32 + 4 * x + 2], dk[hf * 32 + 4 * x + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.pb_smem());
        }
        // ---- epilogue: dV_j and dK_j rows (dK scaled), bf16
        if (ok) {
            ok = wait_or_abort(bars.done(), 0, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const size_t row_off = (static_cast<size_t>(bh) * p.Nk + key) * D;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which ? C::kColDK : C::kColDV;
                const float mul = which ? p.scale : 1.f;
                __nv_bfloat16* out = (which ? p.dk : p.dv) + row_off;
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + col + ch * 32, v);
                    tmem_wait_ld_into(v);
                    const long long oe = static_cast<long long>(row_off) + ch * 32;
                    if (key_ok && gb_index_ok(&g_bwd_error, oe, oe + 31,
                                              static_cast<long long>(p.BH) * p.Nk * D)) {
                        float f[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) f[c] = __uint_as_float(v[c]) * mul;
                        uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
                        for (int x = 0; x < 4; ++x) dst[x] = bf16x8(f + 8 * x);
                    }
                }
            }
        }
    } else {
        setmaxnreg_dec<kDqRegs>();
        // ===================================================== query rows: dQ_i
        // All of dQ_i comes out of Tensor Memory into registers at once (its
        // columns are then free for the next dP^T); it is then added to the
        // accumulator through the dS tile (free once the dQ product has read
        // it): 32-column fp32 boxes of 128 rows in the 128-byte swizzle layout,
        // each added by one TMA reduce-add, two in flight.
        const int wq = warp - 4;
        const int r = wq * 32 + lane;  // query row within the tile = TMEM lane
        const uint32_t tQ = tmem + (static_cast<uint32_t>(wq * 32) << 16) + C::kColDQ;
        const bool leader = threadIdx.x == 4 * 32;
        constexpr int kBoxBytes = 128 * 128;  // 128 rows x 32 fp32
        constexpr int kBoxes = D / 32;
        bool ok = true;
        for (int it = 0; it < n_iter; ++it) {
            ok = dq_group_all(wait_or_abort(bars.dq_full(), it & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[kBoxes][32];
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx) tmem_ld32(tQ + bx * 32, v[bx]);
            if constexpr (kBoxes == 4) {
                tmem_wait_ld_into(v[0], v[1]);
                after_wait_ld(v[2], v[3]);
            } else {
                tmem_wait_ld_into(v[0], v[1]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.dq_free());
            const int q0 = (i_first + it) * kTile;
            // box bx goes through slot bx % 2 of the dS tile; a slot is rewritten
            // once the box before the previous one has been read out of it
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx) {
                if (bx >= 2) {
                    if (leader) bulk_wait_read_but_one();
                    dq_group_sync();
                }
                uint8_t* row = smem + C::kDsOff + (bx & 1) * kBoxBytes + r * 128;
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    *reinterpret_cast<uint4*>(row + ((x ^ (r & 7)) * 16)) =
                        make_uint4(v[bx][4 * x], v[bx][4 * x + 1], v[bx][4 * x + 2], v[bx][4 * x + 3]);
                fence_proxy_async_smem();
                dq_group_sync();
                if (leader) {
                    tma_reduce_add_3d(&tm_dqacc, sDs + (bx & 1) * kBoxBytes, bx * 32, q0, bh);
                    bulk_commit();
                }
            }
            // the dS tile is free once the last boxes have been read
            if (leader) {
                bulk_wait_read_all();
                mbar_arrive(bars.ds_free());
            }
        }
        // the reduce-adds must be complete before the CTA exits
        if (leader) bulk_wait_all();
    }

    // ---- teardown: all Tensor Memory traffic is complete; free the columns
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc<kTmemCols>(tmem);
}

// ----------------------------------------------------------------- convert kernel
//
// dQ = scale * accumulator, rounded to bf16; eight elements per thread.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const float* __restrict__ dq_acc,
                                                          __nv_bfloat16* __restrict__ dq,
                                                          float scale, int Nq, int Nq_pad,
                                                          long long n8) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n8;
         g += stride) {
        const long long e = g * 8;
        const long long row = e / D;  // b*H*Nq + ... in the unpadded layout
        const int col = static_cast<int>(e % D);
        const long long bh = row / Nq;
        const int i = static_cast<int>(row % Nq);
        const long long acc_e = (bh * Nq_pad + i) * D + col;
        if (!gb_index_ok(&g_bwd_error, acc_e, acc_e + 7, n8 / Nq * Nq_pad * 8) ||
            !gb_index_ok(&g_bwd_error, e, e + 7, n8 * 8))
            continue;
        const float4* src = reinterpret_cast<const float4*>(dq_acc + acc_e);
        const float4 a = src[0], b = src[1];
        const float f[8] = {a.x * scale, a.y * scale, a.z * scale, a.w * scale,
                            b.x * scale, b.y * scale, b.z * scale, b.w * scale};
        *reinterpret_cast<uint4*>(dq + e) = bf16x8(f);
    }
}

// ------------------------------------------------------------------ host side

int bwd_set_attributes() {
    if (cudaFuncSetAttribute(attn_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BCfg<128>::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BCfg<64>::kSmemBytes) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t bwd_workspace_bytes(long long BH, int Nq, int d) {
    const long long nq_pad = (static_cast<long long>(Nq) + kTile - 1) / kTile * kTile;
    return static_cast<size_t>(BH * nq_pad) * static_cast<size_t>(d + 2) * sizeof(float);
}

template <int D>
static int launch_backward_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const CUtensorMap& tdqacc,
                             const BwdPrepParams& a, const BwdParams& p, __nv_bfloat16* dq,
                             int num_sms, cudaStream_t stream) {
    const long long prep_threads = (a.rows * (D / 8) + 31) / 32 * 32;
    long long prep_blocks = (prep_threads + 255) / 256;
    if (prep_blocks > 8LL * num_sms) prep_blocks = 8LL * num_sms;
    attn_bwd_prep_kernel<D><<<static_cast<unsigned>(prep_blocks), 256, 0, stream>>>(a);
    const long long grid = static_cast<long long>(p.n_kt) * p.BH;
    attn_bwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, BCfg<D>::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, tdqacc, p);
    const long long n8 = static_cast<long long>(p.BH) * p.Nq * D / 8;
    long long cblocks = (n8 + 255) / 256;
    if (cblocks > 8LL * num_sms) cblocks = 8LL * num_sms;
    attn_bwd_dq_kernel<D><<<static_cast<unsigned>(cblocks), 256, 0, stream>>>(
        p.dq_acc, dq, p.scale, p.Nq, p.Nq_pad, n8);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_backward(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                    const CUtensorMap& tdo, const CUtensorMap& tdqacc, const BwdPrepParams& a,
                    const BwdParams& p, __nv_bfloat16* dq, int num_sms, cudaStream_t stream) {
    return d == 128 ? launch_backward_d<128>(tq, tk, tv, tdo, tdqacc, a, p, dq, num_sms, stream)
                    : launch_backward_d<64>(tq, tk, tv, tdo, tdqacc, a, p, dq, num_sms, stream);
}

unsigned read_and_clear_bwd_error() {
    unsigned v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof v);
    cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof zero);
    return v;
}

}  // namespace gbattn
