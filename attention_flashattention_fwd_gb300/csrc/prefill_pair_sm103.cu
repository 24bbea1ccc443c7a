// prefill_pair_sm103.cu -- the fused attention forward on CTA pairs (bf16, d = 128).
//
// It computes what prefill_sm103.cu computes -- the FlashAttention forward of
// the CS336 Lecture 5 notes, section 8.3: per query block, S = Q K_j^T, a
// running reference max and row sum, P = e^{S - m}, O += P V_j, then O / l and
// the logsumexp; key blocks in the causal future are skipped -- with every
// tensor-core product issued as tcgen05.mma.cta_group::2, the CTA-pair form of
// PDC Lecture 7 §7.13 (CTA pair / MMA.2SM).
//
// A cluster of two CTAs on two SMs works on one item: four consecutive 128-row
// query tiles of one (b, h).  Each CTA keeps two of them (query tile slots t = 0,
// 1, ping-ponging as in the single-CTA kernel); "pair tile" t is the even CTA's
// slot t (rows row0 + 256 t + [0, 128)) over the odd CTA's slot t (the next 128
// rows), the M = 256 of one product.  Of every key tile each CTA holds half:
// keys [0, 64) of K_j in the even CTA and [64, 128) in the odd one (B of
// S = Q K^T, split along N), and of V_j the columns d [0, 64) and [64, 128) (B of
// O += P V, split along N); each CTA's Tensor Memory receives its own 128 rows
// of S and of O in full.  So K/V tiles cost each SM half the shared memory and
// half the L2 reads of the single-CTA kernel, and the ring is twice as deep.
//
// Roles, per CTA (12 warps, as the single-CTA kernel):
//   * warp 9 (one thread): TMA producer of this CTA's Q tiles and K/V halves;
//   * warp 8: in the even CTA, the MMA warp -- all 32 lanes run the loop and the
//     barrier waits, the lane elect_one() picks issues every product of the pair
//     and every commit; commits signal both CTAs' barriers (multicast).  In the
//     odd CTA it only waits for the last product before the teardown;
//   * warp 10 (one thread): in the even CTA, the ring relay of the single-CTA
//     kernel; in the odd CTA, it forwards each of its own Q and K/V landings to
//     the even CTA's barrier of the same tile (a remote arrival), so a full or
//     q_full barrier of the even CTA completes once both halves are in;
//   * warps 0-7: the softmax warpgroups of slots 0 and 1, one query row per
//     thread; the odd CTA's softmax warps signal P on the even CTA's p_ready.
// A wait that runs out sets the abort flag of both CTAs.
//
// On the issue rate: with one elected lane of a converged warp issuing, the
// pair product keeps both SMs' tensor cores busy where the single-CTA product
// leaves them waiting on the issuer (attn_bench_mma_rate).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda.h>

#include <atomic>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

__device__ unsigned int g_prefill_pair_error = 0;

namespace {

namespace cg = cooperative_groups;

constexpr int kD = 128;
constexpr int kBM = 128;               // query rows per tile and CTA
constexpr int kBN = 128;               // keys per key tile (N of S = Q K^T over the pair)
constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kRelayWarp = 10;
constexpr uint32_t kSoftmaxRegs = 192;  // the single-CTA kernel's split at d = 128: 128 x 96 + 256 x 192
constexpr uint32_t kControlRegs = 96;
constexpr uint32_t kTmemCols = 512;
constexpr int kStageBufBytes = 32 * 64;
constexpr float kTileSumLimit = 4.611686018427387904e18f;  // 2^62, as the single-CTA kernel

// shared memory of one CTA
constexpr int kQTileBytes = kBM * kD * 2;  // 32 KB: 128 rows, two 128-byte atoms along d
constexpr int kQSubBytes = kBM * 128;      // one atom column of a query tile
constexpr int kHalfBytes = 16384;          // a K half (64 keys x 128 d) or V half (128 keys x 64 d)
constexpr int kKSubBytes = 64 * 128;       // one atom column of a K half
constexpr int kSlots = 8;                  // ring slots (K or V halves)
constexpr int kQOff = 0;
constexpr int kRingOff = 2 * kQTileBytes;
constexpr int kStageOff = kRingOff + kSlots * kHalfBytes;
constexpr int kStageBytes = 8 * 2 * kStageBufBytes;
constexpr int kBarOff = kStageOff + kStageBytes;
constexpr int kNumBars = 2 * kSlots + 10 + 1;
constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
constexpr int kAbortOff = kTmemSlotOff + 4;
constexpr int kSmemBytes = kAbortOff + 4 + 1024;
// Tensor Memory: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512)
__device__ __forceinline__ uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * kD; }

struct Bars {
    uint32_t full0, empty0, tile0, fin;
    __device__ uint32_t full(int i) const { return full0 + 8u * i; }
    __device__ uint32_t empty(int i) const { return empty0 + 8u * i; }
    __device__ uint32_t q_full(int t) const { return tile0 + 8u * (5 * t + 0); }
    __device__ uint32_t q_empty(int t) const { return tile0 + 8u * (5 * t + 1); }
    __device__ uint32_t s_full(int t) const { return tile0 + 8u * (5 * t + 2); }
    __device__ uint32_t p_ready(int t) const { return tile0 + 8u * (5 * t + 3); }
    __device__ uint32_t pv_done(int t) const { return tile0 + 8u * (5 * t + 4); }
};

// ---- cta_group::2 forms and cluster helpers

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

__device__ __forceinline__ void umma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at offset `bar` of both CTAs when every product
// this thread issued before has completed.
__device__ __forceinline__ void umma_commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(static_cast<uint16_t>(0x3))
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The address of this CTA's shared-memory word `addr` in CTA `cta` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t cta) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
    return r;
}

// One arrival on the barrier at cluster address `raddr` (another CTA's), ordered
// after this thread's earlier memory operations at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t raddr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr)
                 : "memory");
}

// try_wait whose completion also orders the arrivals of the other CTA (their
// writes to its shared or Tensor Memory) before this thread's later operations.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---- work items: four query tiles (two pair tiles) of one (b, h)

struct Item {
    int bh, row0, n_kv0, n_kv1, off;
    bool empty;  // every row past Nq (the second half of a split last quad): skipped
    __device__ int n_kv(int t) const { return t ? n_kv1 : n_kv0; }
    __device__ int n_kv_max() const { return max(n_kv0, n_kv1); }
};

// Items below split_start are quads (pair tiles 0 and 1); from split_start on
// they are single pair tiles, the two halves of the quads left for the last
// wave (slot 0 only, n_kv1 = 0).
__device__ __forceinline__ Item item_at(const PrefillParams& p, int idx) {
    Item it;
    int qidx = idx, half = -1;
    if (idx >= p.split_start) {
        qidx = p.split_start + (idx - p.split_start) / 2;
        half = (idx - p.split_start) & 1;
    }
    int quad;
    if (p.causal) {  // heaviest quads first
        quad = p.num_pairs - 1 - qidx / p.BH;
        it.bh = qidx % p.BH;
    } else {  // a head's quads are consecutive: its K/V stay in L2
        quad = qidx % p.num_pairs;
        it.bh = qidx / p.num_pairs;
    }
    it.row0 = quad * 4 * kBM + (half > 0 ? 2 * kBM : 0);
    it.empty = it.row0 >= p.Nq;
    it.off = p.causal ? p.Nk - p.Nq : 0;
    const int n_kv_all = (p.Nk + kBN - 1) / kBN;
    // pair tile t visits the key tiles up to the one holding the last key its
    // last row (the odd CTA's row 127) sees
    const int last0 = it.row0 + 2 * kBM - 1 + it.off;
    it.n_kv0 = p.causal ? min(n_kv_all, last0 / kBN + 1) : n_kv_all;
    const bool has1 = half < 0 && it.row0 + 2 * kBM < p.Nq;
    it.n_kv1 = !has1 ? 0 : p.causal ? min(n_kv_all, (last0 + 2 * kBM) / kBN + 1) : n_kv_all;
    return it;
}

// k-th item of this cluster in the snake deal over clusters, or -1.
__device__ __forceinline__ int item_index(int k, int n_items) {
    const int G = static_cast<int>(gridDim.x) / 2;
    const int c = static_cast<int>(blockIdx.x) / 2;
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
    return idx < n_items ? static_cast<int>(idx) : -1;
}

__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            tmap),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Both CTAs' abort flags: set this CTA's and the other's.
__device__ __forceinline__ void flag_abort(uint32_t abort_addr, uint32_t other) {
    asm volatile("st.shared.u32 [%0], 1;" ::"r"(abort_addr) : "memory");
    asm volatile("st.shared::cluster.u32 [%0], 1;" ::"r"(peer_addr(abort_addr, other)) : "memory");
    atomicOr(&g_prefill_pair_error, kErrTimeout);
}

// Bounded wait that also gives up once either CTA has aborted.  kCluster: the
// barrier takes arrivals from the other CTA.
template <bool kCluster>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                              uint32_t other) {
    auto test = [&]() {
        return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const uint64_t t0 = globaltimer_ns();
    volatile int* flag = reinterpret_cast<volatile int*>(__cvta_shared_to_generic(abort_addr));
    for (uint32_t it = 1;; ++it) {
        if (test()) return true;
        if ((it & 63u) == 0u) {
            if (*flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                flag_abort(abort_addr, other);
                return false;
            }
        }
    }
}

// The same wait by every lane of a warp, its result warp-uniform.
template <bool kCluster>
__device__ __forceinline__ bool wait_uniform(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                             uint32_t other) {
    return __all_sync(0xffffffffu, wait_or_abort<kCluster>(bar, parity, abort_addr, other));
}

}  // namespace

// tm_k maps K in 64-row boxes (a K half); tm_q and tm_v in 128-row boxes.
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                                 const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v,
                                 const __grid_constant__ CUtensorMap tm_o, PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + kQOff;
    const uint32_t sRing = sbase + kRingOff;
    const uint32_t sStage = sbase + kStageOff;
    Bars bars;
    bars.full0 = sbase + kBarOff;
    bars.empty0 = bars.full0 + 8 * kSlots;
    bars.tile0 = bars.empty0 + 8 * kSlots;
    bars.fin = bars.tile0 + 8 * 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlotOff);
    const uint32_t abort_addr = sbase + kAbortOff;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);

    const uint32_t rank = cluster_rank();
    const uint32_t other = rank ^ 1u;
    const bool even = rank == 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_items = p.n_items;

    // ---- set-up: barriers, abort flag, Tensor Memory of the pair
    if (threadIdx.x == kLoadWarp * 32) {
        for (int i = 0; i < kSlots; ++i) {
            // the even CTA's full barrier also takes the odd CTA's forwarded landing
            mbar_init(bars.full(i), even ? 2 : 1);
            mbar_init(bars.empty(i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bars.q_full(t), even ? 2 : 1);
            mbar_init(bars.q_empty(t), 1);
            mbar_init(bars.s_full(t), 1);
            // four softmax warps of each CTA and the even CTA's relay
            mbar_init(bars.p_ready(t), 9);
            mbar_init(bars.pv_done(t), 1);
        }
        mbar_init(bars.fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc_pair<kTmemCols>(smem_addr(tmem_slot));
    tc_fence_before();
    cg::this_cluster().sync();  // both CTAs' barriers initialised, the columns held
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
    // ====================================================== control warpgroup
    setmaxnreg_dec<kControlRegs>();
    if (warp == kLoadWarp) {
        // ================================================= TMA producer (both CTAs)
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            bool ok = true;
            int kq[2] = {0, 0};
            auto load_q = [&](int t, const Item& it) {
                const int kp = kq[t]++;
                if (kp > 0 &&
                    !(ok = wait_or_abort<false>(bars.q_empty(t), (kp - 1) & 1, abort_addr, other)))
                    return;
                mbar_arrive_expect_tx(bars.q_full(t), kQTileBytes);
                for (int s = 0; s < 2; ++s)
                    tma_load_3d(sQ + t * kQTileBytes + s * kQSubBytes, &tm_q, bars.q_full(t), s * 64,
                                it.row0 + t * 2 * kBM + static_cast<int>(rank) * kBM, it.bh);
            };
            auto load_kv = [&](int which, int j, const Item& it) {  // K_j (0) or V_j (1) half
                const int u = issued;
                const int slot = u % kSlots;
                if (u >= kSlots && !(ok = wait_or_abort<false>(bars.empty(slot),
                                                               ((u / kSlots) & 1) ^ 1, abort_addr,
                                                               other)))
                    return;
                mbar_arrive_expect_tx(bars.full(slot), kHalfBytes);
                if (which) {  // V_j: all 128 keys, this CTA's 64 columns of d
                    tma_load_3d(sRing + slot * kHalfBytes, &tm_v, bars.full(slot),
                                static_cast<int>(rank) * 64, j * kBN, it.bh);
                } else {      // K_j: this CTA's 64 keys, both atoms of d
                    for (int s = 0; s < 2; ++s)
                        tma_load_3d(sRing + slot * kHalfBytes + s * kKSubBytes, &tm_k, bars.full(slot),
                                    s * 64, j * kBN + static_cast<int>(rank) * 64, it.bh);
                }
                ++issued;
            };
            for (int k = 0; ok; ++k) {
                const int idx = item_index(k, n_items);
                if (idx < 0) break;
                const Item it = item_at(p, idx);
                if (it.empty) continue;
                load_q(0, it);
                if (ok) load_kv(0, 0, it);
                if (ok && it.n_kv1 > 0) load_q(1, it);
                if (ok) load_kv(1, 0, it);
                const int nidx = item_index(k + 1, n_items);
                if (ok && nidx >= 0) {
                    const Item nx = item_at(p, nidx);
                    for (int t = 0; t < (nx.empty ? 0 : nx.n_kv1 > 0 ? 2 : 1); ++t)
                        for (int s = 0; s < 2; ++s)
                            tma_prefetch_l2_3d(&tm_q, s * 64,
                                               nx.row0 + t * 2 * kBM + static_cast<int>(rank) * kBM,
                                               nx.bh);
                }
                for (int j = 1; j < it.n_kv_max() && ok; ++j) {
                    load_kv(0, j, it);
                    if (ok) load_kv(1, j, it);
                }
            }
            if (!ok) {
                // drain: every slot's most recent copy must land before exit
                for (int u = max(0, issued - kSlots); u < issued; ++u)
                    mbar_wait(bars.full(u % kSlots), (u / kSlots) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp && even) {
        // ================================================= MMA warp (even CTA)
        // The single-CTA kernel's issue order per key tile j (after the item's
        // S_0(0), S_1(0)):  O_0 += P_0(j) V_j,  S_0(j+1),  O_1 += P_1(j) V_j,  S_1(j+1),
        // each a pair product over both CTAs.
        const uint32_t idesc_qk = umma_idesc_bf16(2 * kBM, kBN, false);
        const uint32_t idesc_pv = umma_idesc_bf16(2 * kBM, kD, true);
        int u = 0;
        int iter[2] = {0, 0};
        auto wait_use = [&](int use) {  // both halves of ring use `use` are in
            return wait_uniform<true>(bars.full(use % kSlots), (use / kSlots) & 1, abort_addr, other);
        };
        const uint64_t dq0 = umma_desc_sw128(sQ, 16, 1024);
        const uint64_t dk0 = umma_desc_sw128(sRing, 16, 1024);
        // V half: one 128-byte atom of d (MN-major), 16 key rows per product
        const uint64_t dv0 = umma_desc_sw128(sRing, kHalfBytes, 1024);
        auto issue_s = [&](int t, int use) {  // S_t = Q_t K^T over the pair
            const uint64_t da = dq0 + ((t * kQTileBytes) >> 4);
            const uint64_t db = dk0 + (((use % kSlots) * kHalfBytes) >> 4);
            const uint32_t dst = tmem + col_s(t);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint32_t offa = ((kk >> 2) * kQSubBytes + (kk & 3) * 32) >> 4;
                const uint32_t offb = ((kk >> 2) * kKSubBytes + (kk & 3) * 32) >> 4;
                umma_ss_pair(dst, da + offa, db + offb, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit_both(bars.s_full(t));
        };
        auto issue_pv = [&](int t, int use, bool first) {  // O_t (+)= P_t V over the pair
            const uint64_t db = dv0 + (((use % kSlots) * kHalfBytes) >> 4);
            const uint32_t dst = tmem + col_o(t);
            const uint32_t pa = tmem + col_s(t);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                umma_ts_pair(dst, pa + kk * 8, db + ((kk * 16 * 128) >> 4), idesc_pv,
                             (!first || kk > 0) ? 1u : 0u);
        };
        bool ok = true;
        int kq[2] = {0, 0};
        for (int k = 0; ok; ++k) {
            const int idx = item_index(k, n_items);
            if (idx < 0) break;
            const Item it = item_at(p, idx);
            if (it.empty) continue;
            const int nmax = it.n_kv_max();
            for (int t = 0; t < 2 && ok; ++t) {
                if (it.n_kv(t) == 0) continue;
                ok = wait_uniform<true>(bars.q_full(t), kq[t]++ & 1, abort_addr, other) &&
                     (t == 1 || wait_use(u));
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_s(t, u);
                    if (it.n_kv(t) == 1) umma_commit_both(bars.q_empty(t));
                }
                __syncwarp();
            }
            if (!ok) break;
            for (int j = 0; j < nmax && ok; ++j) {
                const int uv = u + 1, uk = u + 2;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= it.n_kv(t)) continue;
                    // P_t(j) in both CTAs' Tensor Memory, V_j and K_{j+1} halves in both
                    // CTAs' shared memory, and at j = 0 the previous item's O_t read
                    if (!(ok = wait_uniform<true>(bars.p_ready(t), iter[t] & 1, abort_addr, other)))
                        break;
                    tc_fence_after();
                    if (elect_one()) {
                        issue_pv(t, uv, j == 0);
                        if (j + 1 < it.n_kv(t)) {
                            issue_s(t, uk);
                            if (j + 2 == it.n_kv(t)) umma_commit_both(bars.q_empty(t));
                        } else {
                            umma_commit_both(bars.pv_done(t));
                        }
                    }
                    __syncwarp();
                    ++iter[t];
                }
                u += 2;
            }
        }
        if (elect_one()) umma_commit_both(bars.fin);
        __syncwarp();
        mbar_wait(bars.fin, 0);
        __syncwarp();
    } else if (warp == kRelayWarp && even) {
        // ================================================= ring relay (even CTA)
        // waits for V_j and K_{j+1} (both halves) and adds its arrival to p_ready(t)
        // of each pair tile visiting key tile j, as in the single-CTA kernel
        if (lane == 0) {
            auto wait_use = [&](int use) {
                return wait_or_abort<true>(bars.full(use % kSlots), (use / kSlots) & 1, abort_addr,
                                           other);
            };
            int u = 0;
            int iter[2] = {0, 0};
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int idx = item_index(k, n_items);
                if (idx < 0) break;
                const Item it = item_at(p, idx);
                if (it.empty) continue;
                const int nmax = it.n_kv_max();
                for (int j = 0; j < nmax && ok; ++j) {
                    ok = wait_use(u + 1) && (j + 1 >= nmax || wait_use(u + 2));
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= it.n_kv(t)) continue;
                        if (iter[t] > 0 && !(ok = wait_or_abort<true>(bars.p_ready(t),
                                                                      (iter[t] - 1) & 1,
                                                                      abort_addr, other)))
                            break;
                        mbar_arrive(bars.p_ready(t));
                        ++iter[t];
                    }
                    u += 2;
                }
            }
        }
        __syncwarp();
    } else if (warp == kRelayWarp) {
        // ================================================= forwarder (odd CTA)
        // each of this CTA's landings, in the producer's order, becomes an arrival
        // on the even CTA's barrier of the same tile
        if (lane == 0) {
            int u = 0;
            int kq[2] = {0, 0};
            bool ok = true;
            auto fwd = [&](uint32_t bar, uint32_t parity) {
                if (!(ok = wait_or_abort<false>(bar, parity, abort_addr, other))) return;
                mbar_arrive_cluster(peer_addr(bar, other));
            };
            auto fwd_use = [&]() {
                fwd(bars.full(u % kSlots), (u / kSlots) & 1);
                ++u;
            };
            for (int k = 0; ok; ++k) {
                const int idx = item_index(k, n_items);
                if (idx < 0) break;
                const Item it = item_at(p, idx);
                if (it.empty) continue;
                fwd(bars.q_full(0), kq[0]++ & 1);
                if (ok) fwd_use();                                            // K_0
                if (ok && it.n_kv1 > 0) fwd(bars.q_full(1), kq[1]++ & 1);
                if (ok) fwd_use();                                            // V_0
                for (int j = 1; j < it.n_kv_max() && ok; ++j) {
                    fwd_use();                                                // K_j
                    if (ok) fwd_use();                                        // V_j
                }
            }
        }
        __syncwarp();
    }  // warp 11 has no role
    } else {
        // ================================================= softmax warpgroups
        setmaxnreg_inc<kSoftmaxRegs>();
        const int t = warp >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + col_s(t);
        const uint32_t tO = tmem + lane_off + col_o(t);
        const uint32_t p_ready_dst = even ? bars.p_ready(t) : peer_addr(bars.p_ready(t), other);
        const float cl2 = p.scale_log2;
        int iter = 0;
        int kp = 0;
        int ring = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int idx = item_index(k, n_items);
            if (idx < 0) break;
            const Item it = item_at(p, idx);
            if (it.empty) continue;
            const int base = it.row0 + t * 2 * kBM + static_cast<int>(rank) * kBM;  // this CTA's rows
            const int row = base + r;
            const int nkv = it.n_kv(t);
            const int item_ring = ring;
            ring += 2 * it.n_kv_max();
            if (nkv == 0) continue;
            const bool releaser = (it.n_kv1 > 0 ? t == 1 : t == 0) && wq == 0 && lane == 0;
            float m_ref = -INFINITY;
            float l = 0.f;
            for (int j = 0; j < nkv; ++j, ++iter) {
                ok = wait_or_abort<false>(bars.s_full(t), iter & 1, abort_addr, other);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // S_t(j) completing frees this CTA's halves of K_j and V_{j-1}
                if (releaser) {
                    mbar_arrive(bars.empty((item_ring + 2 * j) % kSlots));
                    if (j > 0) mbar_arrive(bars.empty((item_ring + 2 * j - 1) % kSlots));
                }
                uint32_t sr[kBN];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    tmem_ld32(tS + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[q4 * 32]));
                tmem_wait_ld();
                float* s = reinterpret_cast<float*>(sr);
                const int key0 = j * kBN;
                const bool ragged = key0 + kBN > p.Nk;
                const bool diag = p.causal && (key0 + kBN - 1 > base + it.off);
                if (ragged || diag) {
                    // last visible key of this row (the even CTA's rows see no key of
                    // their pair tile's last key tile when it lies past their diagonal)
                    const int lim = p.causal ? min(p.Nk - 1, row + it.off) : p.Nk - 1;
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (key0 + c > lim) s[c] = -INFINITY;
                }
                auto row_max = [&]() {
                    float mc[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mc[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
                    for (int c = 16; c < kBN; c += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mc[i] = fmax3(mc[i], s[c + i], s[c + 8 + i]);
                    return fmaxf(fmax3(mc[0], mc[1], mc[2]),
                                 fmaxf(fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7])));
                };
                auto emit_p = [&]() {
                    const float mneg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                    const float2 c2 = make_float2(cl2, cl2), m2 = make_float2(mneg, mneg);
                    float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const float2 x = ffma2(
                                make_float2(s[h * 32 + 2 * c], s[h * 32 + 2 * c + 1]), c2, m2);
                            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            if (c & 1) ls1 = fadd2(ls1, pp); else ls0 = fadd2(ls0, pp);
                            pk[c] = pack_bf16x2(pp.x, pp.y);
                        }
                        tmem_st16(tS + h * 16, pk);
                    }
                    return (ls0.x + ls0.y) + (ls1.x + ls1.y);
                };
                // the stale reference max of the single-CTA kernel: the row max of
                // the item's first key tile, moved only when a tile would overflow
                if (j == 0) m_ref = row_max() * cl2;
                float lt = emit_p();
                if (__any_sync(0xffffffffu, !(lt <= kTileSumLimit))) {
                    float alpha = 1.f;
                    if (!(lt <= kTileSumLimit)) {
                        const float m_tile = row_max() * cl2;
                        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_tile);
                        m_ref = m_tile;
                        l *= alpha;
                    }
                    if (j > 0) {
#pragma unroll 1
                        for (int ch = 0; ch < kD / 16; ++ch) {
                            uint32_t o[16];
                            tmem_ld16(tO + ch * 16, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                            tmem_st16(tO + ch * 16, o);
                        }
                    }
                    lt = emit_p();
                }
                l += lt;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (even) mbar_arrive(p_ready_dst);
                    else mbar_arrive_cluster(p_ready_dst);
                }
            }
            if (!ok) break;
            // ---- epilogue: O / l of this CTA's 128 rows and their logsumexp
            ok = wait_or_abort<false>(bars.pv_done(t), kp & 1, abort_addr, other);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            if (releaser) mbar_arrive(bars.empty((item_ring + 2 * nkv - 1) % kSlots));
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            // staged through shared memory (64-byte swizzle) and stored by TMA, as
            // in the single-CTA kernel; the store clips rows past Nq
            const int wrow0 = base + wq * 32;
            const bool store = wrow0 < p.Nq;
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int ch = 0; ch < kD / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(tO + ch * 32, o);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    pk[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                        __uint_as_float(o[2 * c + 1]) * inv_l);
                const uint32_t buf =
                    sStage + static_cast<uint32_t>((warp * 2 + (ch & 1)) * kStageBufBytes);
                if (ch >= 2) {
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                }
                const uint32_t rbase = buf + static_cast<uint32_t>(lane * 64);
                const int sw = (lane >> 1) & 3;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_shared_v4(rbase + static_cast<uint32_t>(((q ^ sw) * 16)), pk[4 * q],
                                 pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && store) {
                    tma_store_3d(&tm_o, buf, ch * 32, wrow0, it.bh);
                    bulk_commit();
                }
            }
            if (row < p.Nq && gb_index_ok(&g_prefill_pair_error,
                                          static_cast<long long>(it.bh) * p.Nq + row,
                                          static_cast<long long>(it.bh) * p.Nq + row,
                                          static_cast<long long>(p.BH) * p.Nq))
                p.lse[static_cast<size_t>(it.bh) * p.Nq + row] =
                    (m_ref + log2f(l)) * 0.69314718055994530942f;
            ++kp;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---- teardown: both CTAs are done with the pair's Tensor Memory.  The odd
    // CTA's shared and Tensor Memory serve the even CTA's products until the last
    // one completes: once this CTA's roles are done, wait for it (a short wait:
    // its softmax warps saw every item's last product complete).
    tc_fence_before();
    __syncthreads();
    if (!even && threadIdx.x == kMmaWarp * 32 && !mbar_wait(bars.fin, 0))
        atomicOr(&g_prefill_pair_error, kErrTimeout);
    cg::this_cluster().sync();
    tc_fence_after();
    if (warp == 0) tmem_dealloc_pair<kTmemCols>(tmem);
}

// ------------------------------------------------------------------ host side

namespace {

std::atomic<int> g_pair_clusters[kMaxDevices];

// CTA pairs the device holds at once with this kernel (one CTA per SM).
int pair_clusters(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = g_pair_clusters[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *out = c;
            return ATTN_OK;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_fwd_prefill_pair_kernel, &cfg) != cudaSuccess ||
        n <= 0) {
        (void)cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (dev >= 0 && dev < kMaxDevices) g_pair_clusters[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return ATTN_OK;
}

}  // namespace

int prefill_pair_set_attributes() {
    return cudaFuncSetAttribute(attn_fwd_prefill_pair_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

// p.num_pairs counts quads (four query tiles) per head here.  Without a causal
// mask every quad costs the same, so quads that would leave the last wave
// part-full run as two single pair tiles when those fit in one wave.
int launch_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv,
                        const CUtensorMap& to, const PrefillParams& params, cudaStream_t stream) {
    PrefillParams p = params;
    int clusters = 0;
    int st = pair_clusters(&clusters);
    if (st != ATTN_OK) return st;
    const long long quads = static_cast<long long>(p.num_pairs) * p.BH;
    const long long grid = quads < clusters ? quads : clusters;
    long long items = quads, split = quads;
    if (!p.causal && quads > grid) {
        const long long full = quads / grid * grid, tail = quads - full;
        if (tail > 0 && 2 * tail <= grid && full + 2 * tail <= 0x7fffffffLL) {
            split = full;
            items = full + 2 * tail;
        }
    }
    p.n_items = static_cast<int>(items);
    p.split_start = static_cast<int>(split);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn_fwd_prefill_pair_kernel, tq, tk64, tv, to, p) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

unsigned read_and_clear_prefill_pair_error() {
    unsigned v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_prefill_pair_error, sizeof v);
    cudaMemcpyToSymbol(g_prefill_pair_error, &zero, sizeof zero);
    return v;
}

}  // namespace gbattn
