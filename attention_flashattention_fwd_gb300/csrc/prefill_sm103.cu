// prefill_sm103.cu -- fused attention forward (prefill) for sm_103a.
//
// What it computes is the FlashAttention forward of the CS336 Lecture 5
// notes, section 8.3: for each query block Q_i, for each key/value block
// (K_j, V_j): S_ij = Q_i K_j^T (scaled), a running row max m and row sum l,
// P_ij = e^{S_ij - m}, l and O rescaled when m grows, O += P_ij V_j; at the
// end O /= l and L_i = m_i + log l_i.  Key blocks wholly in the causal future
// of a query block are skipped (same section).  The blocked softmax merge it
// relies on is CS149 Lecture 9 notes, concept 9.
//
// How it maps onto a GB300 SM (persistent: one CTA per SM, 12 warps):
//   * a work item is a pair of consecutive 128-row query tiles of one (b, h);
//     the two tiles share every key/value tile they visit.  Items are ordered
//     heaviest first (causal) and dealt to the CTAs in a snake order
//     (0..G-1, G-1..0, ...), which balances the causal triangle as well as a
//     greedy longest-first schedule;
//   * warp 9 (one thread) is the TMA producer: Q_0/Q_1 of an item (as soon as
//     the previous item's last Q K^T products are done), then K_j and V_j tiles
//     through a ring of shared-memory slots guarded by full/empty mbarriers
//     with transaction counts (the double buffering of CS149 Lecture 9
//     concept 2, deeper than two), running ahead across item boundaries;
//   * warp 8 (one thread) issues tcgen05.mma: S_t = Q_t K_j^T into Tensor
//     Memory, then O_t += P_t V_j with P read from Tensor Memory;
//   * warp 10 (one thread) relays the ring: it waits for V_j and K_{j+1} to
//     land and adds its arrival to the barrier the softmax warps signal P_t(j)
//     on, so the MMA thread waits on one barrier per pair of products;
//   * warps 0-3 and 4-7 are the softmax warpgroups of query tiles 0 and 1: a
//     thread owns one query row (= one TMEM lane), so row max and row sum need
//     no shuffles; it writes P back as bf16 over its own S columns, rescales
//     its O row in TMEM when a key tile lies far above the running reference
//     max, and at the end of an item writes O / l and the logsumexp (its next
//     P arrival tells the MMA warp that the O columns are free again);
//   * the two query tiles ping-pong: while one warpgroup runs its softmax the
//     tensor core works on the other tile.
// Scores use base 2: with c = scale * log2(e), p = 2^{s c - m} and
// lse = ln2 (m + log2 l), identical in exact arithmetic to the e-based form.
//
// FP8 operands (kFp8): Q, K and V are E4M3 with one descale per tensor, the
// per-tensor scaling of PDC course Lecture 7, section 7.14.  The products run
// as kind::f8f6f4 (32 keys or 32 of d per instruction, half the instructions
// of bf16 for the same tile), P is rounded to E4M3 for the P V product, the
// query and key descales fold into c and the value descale into the final
// 1 / l.  Both operands of an 8-bit product are K-major, so V comes
// transposed ([B, H, d, Nk]: keys innermost), and its tile is one 128-byte
// swizzle atom wide like the Q and K tiles at d = 128.
#include <cuda_bf16.h>
#include <cuda.h>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

__device__ unsigned int g_prefill_error = 0;

namespace {

constexpr int kBM = 128;            // query rows per tile (MMA M)
constexpr int kBN = 128;            // keys per tile (MMA N of S = Q K^T)
constexpr int kThreads = 384;       // 12 warps: 8 softmax, MMA, TMA, relay, 1 idle
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kRelayWarp = 10;
// Register split.  The launch gives every thread 168 registers (65536 / 384,
// rounded down to 8): 384 x 168 = 64512.  The warpgroup of the MMA, TMA and
// relay warps gives part of its share to the two softmax warpgroups, which
// needs 2 (S - 168) <= 168 - C.  d = 128: 256 x 192 + 128 x 96 = 61440; the
// converged MMA warp fits in 96 and the softmax runs faster with 192 than with
// 176 (measured: 176/112, 184/96, 200/96 and 208/88 slower or no better,
// 168/128 spills).  d = 64: 256 x 176 + 128 x 112 = 59392 (192/96 spills there).
template <int D> constexpr uint32_t softmax_regs() { return D == 128 ? 192u : 176u; }
template <int D> constexpr uint32_t control_regs() { return D == 128 ? 96u : 112u; }
constexpr uint32_t kTmemCols = 512;
constexpr int kStageBufBytes = 32 * 64;  // one O staging buffer: 32 rows x 64 bytes
// A key tile whose row sum against the stale reference max exceeds this moves
// the reference.  bf16 P: 2^62, far from fp32 overflow for O and l.  E4M3 P:
// 448, the largest finite E4M3 value; a row sum within it bounds every p of
// the row, so no p saturates.
constexpr float kTileSumLimitBf16 = 4.611686018427387904e18f;
constexpr float kTileSumLimitE4m3 = 448.f;

template <int D, bool kFp8>
struct Cfg {
    static constexpr int kElem = kFp8 ? 1 : 2;           // bytes per Q, K, V element
    static constexpr int kSubElems = 128 / kElem;        // elements per 128-byte atom row
    static constexpr int kSub = D / kSubElems;           // 128-byte swizzle atoms along d
    static constexpr int kSubBytes = 128 * 128;          // one atom column: 128 rows x 128 B
    static constexpr int kTileBytes = kBM * D * kElem;   // a Q, K or V tile
    static constexpr int kSlots = (kTileBytes >= 32768) ? 4 : 8;  // K/V ring slots
    static constexpr int kKSteps = D * kElem / 32;       // MMA k-steps of S = Q K^T (32 B each)
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    // O staging of the epilogue: per softmax warp two buffers of 32 rows x 32 bf16
    // (64-byte swizzle), the source of the TMA stores of O
    static constexpr int kStageOff = kRingOff + kSlots * kTileBytes;
    static constexpr int kStageBytes = 8 * 2 * kStageBufBytes;
    static constexpr int kBarOff = kStageOff + kStageBytes;
    // barriers: full[kSlots], empty[kSlots], then per query tile q_full, q_empty,
    // s_full, p_ready, pv_done, then fin
    static constexpr int kNumBars = 2 * kSlots + 10 + 1;
    static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
    static constexpr int kAbortOff = kTmemSlotOff + 4;
    static constexpr int kSmemBytes = kAbortOff + 4 + 1024;  // + alignment slack
    // Tensor Memory columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 after it;
    // P_t (bf16 pairs: 64 columns; E4M3 quads: 32) overwrites the first columns of S_t.
    __device__ static uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
    __device__ static uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * D; }
};

struct Bars {
    uint32_t full0, empty0, tile0, fin;
    __device__ uint32_t full(int i) const { return full0 + 8u * i; }
    __device__ uint32_t empty(int i) const { return empty0 + 8u * i; }
    // five barriers per query tile t
    __device__ uint32_t q_full(int t) const { return tile0 + 8u * (5 * t + 0); }
    __device__ uint32_t q_empty(int t) const { return tile0 + 8u * (5 * t + 1); }
    __device__ uint32_t s_full(int t) const { return tile0 + 8u * (5 * t + 2); }
    __device__ uint32_t p_ready(int t) const { return tile0 + 8u * (5 * t + 3); }
    __device__ uint32_t pv_done(int t) const { return tile0 + 8u * (5 * t + 4); }
};

// Geometry of work item `idx` (0 <= idx < n_items).  Items below split_start
// are pairs of query tiles; the ones from split_start on are single query
// tiles, the two halves of a pair (tile slot 0 only, n_kv1 = 0): the pairs a
// non-causal launch leaves for a part-full last wave, or every pair of a
// causal launch of at most one wave (see plan_items).  With per-sequence lengths, nq / nk are sequence b's; an item
// whose rows all lie past nq is empty and every role skips it.
struct Item {
    int bh, row0, n_kv0, n_kv1;
    int nq, nk, off;  // query and key count of the sequence; causal offset nk - nq
    bool empty;
    __device__ int n_kv(int t) const { return t ? n_kv1 : n_kv0; }
    __device__ int n_kv_max() const { return max(n_kv0, n_kv1); }
};

template <bool kRagged, bool kGrouped>
__device__ __forceinline__ Item item_at(const PrefillParams& p, int idx) {
    Item it;
    int pidx = idx, half = -1;  // half >= 0: a single query tile of pair pidx
    if (idx >= p.split_start) {
        pidx = p.split_start + (idx - p.split_start) / 2;
        half = (idx - p.split_start) & 1;
    }
    int pair;
    if (kGrouped) {  // causal, heads in groups (see plan_items); heaviest first in each
        const int hg = p.head_group;
        const int per = hg * p.num_pairs;
        const int g = pidx / per;
        const int w = pidx - g * per;
        const int gsize = min(hg, p.BH - g * hg);
        pair = p.num_pairs - 1 - w / gsize;
        it.bh = g * hg + w % gsize;
    } else if (p.causal) {  // heaviest pairs (most key tiles) first
        pair = p.num_pairs - 1 - pidx / p.BH;
        it.bh = pidx % p.BH;
    } else {  // a head's pairs are consecutive: its K/V stay in L2
        pair = pidx % p.num_pairs;
        it.bh = pidx / p.num_pairs;
    }
    it.row0 = pair * 2 * kBM + (half > 0 ? kBM : 0);
    it.nq = p.Nq;
    it.nk = p.Nk;
    if constexpr (kRagged) {
        const int b = it.bh / p.H;
        const bool b_ok = gb_index_ok(&g_prefill_error, b, b, p.BH / p.H);
        if (p.seqlens_q) it.nq = b_ok ? p.seqlens_q[b] : 0;
        if (p.seqlens_k) it.nk = b_ok ? p.seqlens_k[b] : 0;
        if (it.nq < 1 || it.nq > p.Nq || it.nk < 1 || it.nk > p.Nk || (p.causal && it.nq > it.nk)) {
            atomicOr(&g_prefill_error, kErrBitLengths);  // the sequence is skipped
            it.nq = 0;  // skip the sequence
            it.nk = 1;
        }
    }
    it.empty = it.row0 >= it.nq;
    it.off = p.causal ? it.nk - it.nq : 0;
    const int n_kv_all = (it.nk + kBN - 1) / kBN;
    // key tiles each query tile visits (causal: up to the tile holding the last
    // key its last row sees, key row0 + 127 + off for tile 0); tile 1 visits
    // every tile tile 0 does, and at most one more
    const int last0 = it.row0 + kBM - 1 + it.off;
    it.n_kv0 = p.causal ? min(n_kv_all, last0 / kBN + 1) : n_kv_all;
    it.n_kv1 = half >= 0 ? 0 : p.causal ? min(n_kv_all, (last0 + kBM) / kBN + 1) : n_kv_all;
    return it;
}

// k-th item of this CTA in the snake deal, or -1 when there are no more.
__device__ __forceinline__ int item_index(int k, int n_items) {
    const int G = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
    return idx < n_items ? static_cast<int>(idx) : -1;
}

__device__ __forceinline__ void flag_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_prefill_error, kErrTimeout);
}

// Bounded wait that also gives up as soon as another role has aborted.
// TMA store of a box of O from shared memory, tracked by this thread's bulk
// async-group; coordinates in elements, innermost first.
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            tmap),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// All but the newest N of this thread's committed bulk groups have read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// This thread's committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
// Shared-memory writes of this thread become visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

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
// warp-uniform so that no lane leaves the warp's loops alone (a lane whose wait
// ran out takes the whole warp with it).
__device__ __forceinline__ bool wait_uniform(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
}

}  // namespace

// kRagged: per-sequence lengths (seqlens_q / seqlens_k) are read; the
// instantiation without them is the plain [B, H, Nq, Nk] problem.  kFp8: E4M3
// operands, tm_v maps the transposed values [BH, d, Nk].  kGrouped: causal items
// dealt in head groups (a separate instantiation, so that the others keep the
// plain item arithmetic).
template <int D, bool kRagged, bool kFp8, bool kGrouped = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_o, PrefillParams p) {
    static_assert(!kFp8 || (D == 128 && !kRagged), "E4M3 operands: d = 128, no sequence lengths");
    using C = Cfg<D, kFp8>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + C::kQOff;
    const uint32_t sRing = sbase + C::kRingOff;
    const uint32_t sStage = sbase + C::kStageOff;
    Bars bars;
    bars.full0 = sbase + C::kBarOff;
    bars.empty0 = bars.full0 + 8 * C::kSlots;
    bars.tile0 = bars.empty0 + 8 * C::kSlots;
    bars.fin = bars.tile0 + 8 * 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlotOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_items = p.n_items;

    // ---- set-up: barriers (one thread), Tensor Memory (warp 0)
    if (threadIdx.x == kLoadWarp * 32) {
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(bars.full(i), 1);
            mbar_init(bars.empty(i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bars.q_full(t), 1);
            mbar_init(bars.q_empty(t), 1);
            mbar_init(bars.s_full(t), 1);
            // one arrival per softmax warp and one from the relay warp
            mbar_init(bars.p_ready(t), 5);
            mbar_init(bars.pv_done(t), 1);
        }
        mbar_init(bars.fin, 1);
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
    setmaxnreg_dec<control_regs<D>()>();
    if (warp == kLoadWarp) {
        // ================================================= TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;  // ring uses (K or V tiles) issued so far
            bool ok = true;
            int kq[2] = {0, 0};  // items in which query tile slot t took part
            auto load_q = [&](int t, const Item& it) {
                // the previous item's last Q_t K^T product has finished
                const int kp = kq[t]++;
                if (kp > 0 && !(ok = wait_or_abort(bars.q_empty(t), (kp - 1) & 1, abort_flag)))
                    return;
                mbar_arrive_expect_tx(bars.q_full(t), C::kTileBytes);
                for (int s = 0; s < C::kSub; ++s)
                    tma_load_3d(sQ + t * C::kTileBytes + s * C::kSubBytes, &tm_q, bars.q_full(t),
                                s * C::kSubElems, it.row0 + t * kBM, it.bh);
            };
            auto load_kv = [&](int which, int j, const Item& it) {  // K_j (0) or V_j (1)
                const int u = issued;  // K_j is use 2j, V_j is use 2j + 1 of the item
                const int slot = u % C::kSlots;
                if (u >= C::kSlots &&
                    !(ok = wait_or_abort(bars.empty(slot), ((u / C::kSlots) & 1) ^ 1, abort_flag)))
                    return;
                mbar_arrive_expect_tx(bars.full(slot), C::kTileBytes);
                if (kFp8 && which) {
                    // V^T tile: d rows of 128 keys, one atom wide
                    tma_load_3d(sRing + slot * C::kTileBytes, &tm_v, bars.full(slot), j * kBN, 0,
                                it.bh);
                } else {
                    const CUtensorMap* tm = which ? &tm_v : &tm_k;
                    for (int s = 0; s < C::kSub; ++s)
                        tma_load_3d(sRing + slot * C::kTileBytes + s * C::kSubBytes, tm,
                                    bars.full(slot), s * C::kSubElems, j * kBN, it.bh);
                }
                ++issued;
            };
            for (int k = 0; ok; ++k) {  // empty items are skipped by every role
                const int idx = item_index(k, n_items);
                if (idx < 0) break;
                const Item it = item_at<kRagged, kGrouped>(p, idx);
                if (it.empty) continue;
                // in the order the MMA warp needs them: Q_0, K_0, Q_1, V_0, K_1, V_1, ...
                load_q(0, it);
                if (ok) load_kv(0, 0, it);
                if (ok && it.n_kv1 > 0) load_q(1, it);
                if (ok) load_kv(1, 0, it);
                // warm L2 with the next item's query tiles (read once, from DRAM)
                const int nidx = item_index(k + 1, n_items);
                if (ok && nidx >= 0) {
                    const Item nx = item_at<kRagged, kGrouped>(p, nidx);
                    for (int t = 0; t < (nx.n_kv1 > 0 ? 2 : 1); ++t)
                        for (int s = 0; s < C::kSub; ++s)
                            tma_prefetch_l2_3d(&tm_q, s * C::kSubElems, nx.row0 + t * kBM, nx.bh);
                }
                for (int j = 1; j < it.n_kv_max() && ok; ++j) {
                    load_kv(0, j, it);
                    if (ok) load_kv(1, j, it);
                }
            }
            if (!ok) {
                // drain: every slot's most recent copy must land before exit
                for (int u = max(0, issued - C::kSlots); u < issued; ++u)
                    mbar_wait(bars.full(u % C::kSlots), (u / C::kSlots) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ================================================= MMA issuer
        // Issue order per key tile j of an item (after the item's S_0(0), S_1(0)):
        //   O_0 += P_0(j) V_j,  S_0(j+1) = Q_0 K_{j+1}^T,  O_1 += P_1(j) V_j,  S_1(j+1)
        // so that while warpgroup t runs the softmax of S_t(j+1), the tensor core
        // works on the other tile's two products.  S_t(j+1) overwrites the TMEM
        // columns P_t(j) is read from by the product issued just before it; the
        // MMAs of one thread run in issue order, so the read comes first.
        // The thread issues nothing but MMAs and the commits the softmax needs:
        // one tcgen05.mma takes it about as long to issue as an M128 N128 K16
        // product takes to run, so ring slots are released by the softmax of
        // tile 1 instead (see there) and P V completion is only committed at
        // the end of an item.
        // The whole warp runs this loop and every barrier wait; one elected lane
        // (elect_one) issues each group of products with its commits.
        {
            const uint32_t idesc_qk =
                kFp8 ? umma_idesc_e4m3(kBM, kBN) : umma_idesc_bf16(kBM, kBN, false);
            const uint32_t idesc_pv =
                kFp8 ? umma_idesc_e4m3(kBM, D) : umma_idesc_bf16(kBM, D, true);
            int u = 0;             // ring use of the current K tile
            int iter[2] = {0, 0};  // key tiles processed per query tile, over all items
            auto wait_use = [&](int use) {
                return wait_uniform(bars.full(use % C::kSlots), (use / C::kSlots) & 1,
                                    abort_flag);
            };
            // Descriptors are built once; the k-steps only move the start address
            // (bits 0-13 of the low word, in 16-byte units), which never carries.
            // bf16 V is the MN-major B operand (its two 64-wide halves of d
            // kSubBytes apart); E4M3 V^T is K-major like K.
            const uint64_t dq0 = umma_desc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = umma_desc_sw128(sRing, 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(sRing, kFp8 ? 16u : C::kSubBytes, 1024);
            auto issue_s = [&](int t, int use) {  // S_t = Q_t K^T, K in ring use `use`
                const uint64_t da = dq0 + ((t * C::kTileBytes) >> 4);
                const uint64_t db = dk0 + (((use % C::kSlots) * C::kTileBytes) >> 4);
                const uint32_t dst = tmem + C::col_s(t);
#pragma unroll
                for (int kk = 0; kk < C::kKSteps; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kSubBytes + (kk & 3) * 32) >> 4;
                    if constexpr (kFp8)
                        umma_ss_f8(dst, da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
                    else
                        umma_ss(dst, da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit(bars.s_full(t));
            };
            auto issue_pv = [&](int t, int use, bool first) {  // O_t (+)= P_t V
                const uint64_t db = dv0 + (((use % C::kSlots) * C::kTileBytes) >> 4);
                const uint32_t dst = tmem + C::col_o(t);
                const uint32_t pa = tmem + C::col_s(t);
                if constexpr (kFp8) {
#pragma unroll
                    for (int kk = 0; kk < kBN / 32; ++kk) {
                        // P: 32 keys = 8 packed columns; V^T: the next 32 bytes
                        // (keys) of every d row
                        umma_ts_f8(dst, pa + kk * 8, db + ((kk * 32) >> 4), idesc_pv,
                                   (!first || kk > 0) ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        // P: 16 keys = 8 packed columns; V: 16 key rows of 128 B,
                        // the two 64-wide halves of d are kSubBytes apart (LBO)
                        umma_ts(dst, pa + kk * 8, db + ((kk * 16 * 128) >> 4), idesc_pv,
                                (!first || kk > 0) ? 1u : 0u);
                    }
                }
            };
            bool ok = true;
            int kq[2] = {0, 0};  // items in which query tile slot t took part
            for (int k = 0; ok; ++k) {
                const int idx = item_index(k, n_items);
                if (idx < 0) break;
                const Item it = item_at<kRagged, kGrouped>(p, idx);
                if (it.empty) continue;
                const int nmax = it.n_kv_max();
                // prologue of the item: S_0(0) once Q_0 and K_0 are in, then S_1(0)
                // (a single-tile item has no tile 1)
                for (int t = 0; t < 2 && ok; ++t) {
                    if (it.n_kv(t) == 0) continue;
                    ok = wait_uniform(bars.q_full(t), kq[t]++ & 1, abort_flag) &&
                         (t == 1 || wait_use(u));
                    if (!ok) break;
                    tc_fence_after();
                    if (elect_one()) {
                        issue_s(t, u);  // n_kv0 >= 1
                        if (it.n_kv(t) == 1) umma_commit(bars.q_empty(t));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                for (int j = 0; j < nmax && ok; ++j) {
                    const int uv = u + 1, uk = u + 2;  // V_j, K_{j+1}
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= it.n_kv(t)) continue;
                        // one wait covers P_t(j) in Tensor Memory, V_j and K_{j+1} in
                        // shared memory (the relay warp's arrival) and, at j = 0, the
                        // previous item's O_t read by its epilogue (the softmax warps
                        // arrive here only after their epilogue's loads completed)
                        if (!(ok = wait_uniform(bars.p_ready(t), iter[t] & 1, abort_flag)))
                            break;
                        tc_fence_after();
                        if (elect_one()) {
                            issue_pv(t, uv, j == 0);
                            if (j + 1 < it.n_kv(t)) {
                                issue_s(t, uk);
                                if (j + 2 == it.n_kv(t)) umma_commit(bars.q_empty(t));
                            } else {
                                umma_commit(bars.pv_done(t));  // O_t of this item is complete
                            }
                        }
                        __syncwarp();
                        ++iter[t];
                    }
                    u += 2;
                }
            }
            // every MMA this thread issued has completed once `fin` flips
            if (elect_one()) umma_commit(bars.fin);
            __syncwarp();
            mbar_wait(bars.fin, 0);
        }
        __syncwarp();
    } else if (warp == kRelayWarp) {
        // ================================================= ring relay
        // Every barrier wait costs the MMA thread about as long as two products
        // take to run once the softmax warps share its sub-partition, and the
        // tensor core's queue holds only a few products.  This thread takes the
        // ring waits off it: it waits for V_j and K_{j+1} to land and adds one
        // arrival to p_ready(t) of each query tile t that visits key tile j, so
        // the MMA thread waits once per product pair.  An arrival for phase g
        // must not land before phase g - 1 completes, hence the wait on the
        // previous phase (the softmax arrivals already come in phase order).
        if (lane == 0) {
            auto wait_use = [&](int use) {
                return wait_or_abort(bars.full(use % C::kSlots), (use / C::kSlots) & 1,
                                     abort_flag);
            };
            int u = 0;             // ring use of the current K tile
            int iter[2] = {0, 0};  // p_ready phases per query tile, over all items
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int idx = item_index(k, n_items);
                if (idx < 0) break;
                const Item it = item_at<kRagged, kGrouped>(p, idx);
                if (it.empty) continue;
                const int nmax = it.n_kv_max();
                for (int j = 0; j < nmax && ok; ++j) {
                    ok = wait_use(u + 1) && (j + 1 >= nmax || wait_use(u + 2));  // V_j, K_{j+1}
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= it.n_kv(t)) continue;
                        if (iter[t] > 0 &&
                            !(ok = wait_or_abort(bars.p_ready(t), (iter[t] - 1) & 1, abort_flag)))
                            break;
                        mbar_arrive(bars.p_ready(t));
                        ++iter[t];
                    }
                    u += 2;
                }
            }
        }
        __syncwarp();
    }  // warp 11 has no role
    } else {
        // ================================================= softmax warpgroups
        setmaxnreg_inc<softmax_regs<D>()>();
        const int t = warp >> 2;          // query tile 0 or 1
        const int wq = warp & 3;          // TMEM lane quarter
        const int r = wq * 32 + lane;     // row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::col_s(t);
        const uint32_t tO = tmem + lane_off + C::col_o(t);
        const float cl2 = p.scale_log2;
        int iter = 0;  // key tiles processed by this tile over all items
        int kp = 0;    // items in which this tile took part
        int ring = 0;  // ring use of the current item's K_0 (2 per key tile of an item)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int idx = item_index(k, n_items);
            if (idx < 0) break;
            const Item it = item_at<kRagged, kGrouped>(p, idx);
            if (it.empty) continue;
            const int row = it.row0 + t * kBM + r;
            const int nkv = it.n_kv(t);
            const int item_ring = ring;
            ring += 2 * it.n_kv_max();
            if (nkv == 0) continue;  // tile slot 1 of a single-tile item
            // the tile that visits every key tile of the item returns the ring
            // slots: tile 1, or tile 0 of a single-tile item
            const bool releaser = (it.n_kv1 > 0 ? t == 1 : t == 0) && wq == 0 && lane == 0;
            float m_ref = -INFINITY;  // running reference max, log2 units
            float l = 0.f;
            for (int j = 0; j < nkv; ++j, ++iter) {
                ok = wait_or_abort(bars.s_full(t), iter & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // S_t(j) was issued after every earlier product of this CTA, so its
                // completion means K_j (last read by S_t(j)) and V_{j-1} (last read
                // by P_t(j-1) V_{j-1}) are free: the releasing tile hands their ring
                // slots back to the producer.  K_j and V_j are ring uses
                // item_ring + 2 j and + 2 j + 1.
                if (releaser) {
                    mbar_arrive(bars.empty((item_ring + 2 * j) % C::kSlots));
                    if (j > 0) mbar_arrive(bars.empty((item_ring + 2 * j - 1) % C::kSlots));
                }
                // S row: four 32-column loads in flight, one wait
                uint32_t sr[kBN];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    tmem_ld32(tS + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[q4 * 32]));
                tmem_wait_ld();
                float* s = reinterpret_cast<float*>(sr);
                const int key0 = j * kBN;
                const bool ragged = key0 + kBN > it.nk;
                const bool diag = p.causal && (key0 + kBN - 1 > it.row0 + t * kBM + it.off);
                if (ragged || diag) {
                    // last visible key of this row
                    const int lim = p.causal ? min(it.nk - 1, row + it.off) : it.nk - 1;
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (key0 + c > lim) s[c] = -INFINITY;
                }
                // row max: eight independent 3-input max chains, then a short tree
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
                // P = 2^(s c - m_ref) into TMEM, with packed fp32 FMA and adds (two
                // lanes of work per instruction); returns this tile's row sum
                auto emit_p = [&]() {
                    const float mneg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                    const float2 c2 = make_float2(cl2, cl2), m2 = make_float2(mneg, mneg);
                    float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
                    if constexpr (kFp8) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t pk[16];  // 4 E4M3 values per column
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const float* sc = s + h * 64 + 4 * c;
                                const float2 x0 = ffma2(make_float2(sc[0], sc[1]), c2, m2);
                                const float2 x1 = ffma2(make_float2(sc[2], sc[3]), c2, m2);
                                const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
                                const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
                                ls0 = fadd2(ls0, p0);
                                ls1 = fadd2(ls1, p1);
                                pk[c] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
                            }
                            tmem_st16(tS + h * 16, pk);  // P over the first 32 columns of S
                        }
                    } else {
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
                            tmem_st16(tS + h * 16, pk);  // P over the first 64 columns of S
                        }
                    }
                    return (ls0.x + ls0.y) + (ls1.x + ls1.y);
                };
                constexpr float kTileSumLimit = kFp8 ? kTileSumLimitE4m3 : kTileSumLimitBf16;
                // The reference m_ref is the row max of the item's first key tile and
                // is only moved when a later tile would overflow against it: O and l
                // share the reference, so any reference gives the same O / l, and
                // fp32 / bf16 keep full relative precision for p up to 2^62.  Most
                // tiles therefore need no row max at all.
                if (j == 0) m_ref = row_max() * cl2;
                float lt = emit_p();
                if (__any_sync(0xffffffffu, !(lt <= kTileSumLimit))) {
                    // rare: move this row's reference to the tile max, rescale O and l,
                    // and write P again (rows that did not move write the same P)
                    float alpha = 1.f;
                    if (!(lt <= kTileSumLimit)) {
                        const float m_tile = row_max() * cl2;
                        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_tile);
                        m_ref = m_tile;
                        l *= alpha;
                    }
                    if (j > 0) {
                        // O_t row *= alpha, 16 columns at a time (the score row
                        // is still live).  The previous P V product is complete:
                        // S_t(j) was issued after it.
#pragma unroll 1
                        for (int ch = 0; ch < D / 16; ++ch) {
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
                if (lane == 0) mbar_arrive(bars.p_ready(t));
            }
            if (!ok) break;
            // ---- epilogue of the item: O / l and the logsumexp
            ok = wait_or_abort(bars.pv_done(t), kp & 1, abort_flag);  // one phase per item
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // the item's last V tile is free once its last P V product is done
            if (releaser) mbar_arrive(bars.empty((item_ring + 2 * nkv - 1) % C::kSlots));
            float inv_l = l > 0.f ? 1.f / l : 0.f;
            if constexpr (kFp8) inv_l *= p.o_scale;
            if constexpr (kRagged) {
                // rows past the sequence's length must stay untouched: direct stores
                __nv_bfloat16* orow = p.o + (static_cast<size_t>(it.bh) * p.Nq + row) * D;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(tO + ch * 32, o);
                    tmem_wait_ld();
                    const long long oi = (static_cast<long long>(it.bh) * p.Nq + row) * D + ch * 32;
                    if (row < it.nq && gb_index_ok(&g_prefill_error, oi, oi + 31,
                                                   static_cast<long long>(p.BH) * p.Nq * D)) {
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            pk[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l,
                                                __uint_as_float(o[2 * c + 1]) * inv_l);
                        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                                 pk[4 * v4 + 3]);
                    }
                }
            } else {
                // A thread holds one row of O, so direct stores would write 32 rows
                // 2 d bytes apart per instruction.  Instead each warp stages 32 rows
                // x 32 columns in shared memory (64-byte swizzle: the 16-byte granule
                // q of row i sits at granule q ^ ((i >> 1) & 3), so 8 neighbouring
                // rows hit distinct banks) and one lane stores the box with TMA, two
                // buffers per warp so the next chunk is written while one drains.
                // The store clips rows past Nq.
                const int wrow0 = it.row0 + t * kBM + wq * 32;
                const bool store = wrow0 < it.nq;
                if (lane == 0) bulk_wait_read<0>();  // the previous item's stores have read
                __syncwarp();
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
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
                    if (ch >= 2) {  // buffer ch & 1 was last the source of chunk ch - 2
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
            }
            // O_t has been read (each load above was waited for): the MMA thread
            // learns it from this warp's next p_ready arrival, which follows
            if (row < it.nq && gb_index_ok(&g_prefill_error,
                                           static_cast<long long>(it.bh) * p.Nq + row,
                                           static_cast<long long>(it.bh) * p.Nq + row,
                                           static_cast<long long>(p.BH) * p.Nq))
                p.lse[static_cast<size_t>(it.bh) * p.Nq + row] =
                    (m_ref + log2f(l)) * 0.69314718055994530942f;
            ++kp;
        }
        // the TMA stores of O have completed before the CTA (and its shared memory) ends
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---- teardown: all Tensor Memory traffic is complete; free the columns
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc<kTmemCols>(tmem);
}

// ------------------------------------------------------------------ host side

int prefill_set_attributes() {
    const auto a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    const int s128 = Cfg<128, false>::kSmemBytes, s64 = Cfg<64, false>::kSmemBytes;
    if (cudaFuncSetAttribute(attn_fwd_prefill_kernel<128, false, false>, a, s128) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_prefill_kernel<64, false, false>, a, s64) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_prefill_kernel<128, true, false>, a, s128) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_prefill_kernel<64, true, false>, a, s64) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_prefill_kernel<128, false, false, true>, a, s128) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_prefill_kernel<128, false, true>, a,
                             Cfg<128, true>::kSmemBytes) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

// The persistent grid (one CTA per SM, at most one per item) and the work
// items.  Without a causal mask or per-sequence lengths every pair costs the
// same, so pairs that would leave the last wave part-full run as two
// single-tile items instead, when those fit in one wave: e.g. 512 pairs on 152
// SMs take 3 waves of pairs and one of 112 single tiles instead of 4 waves.
// A causal launch of at most one wave of pairs (few heads) lasts as long as its
// heaviest pair, so there every pair runs as two single tiles, heaviest first:
// 5-8 % faster on B1 H1-H2 N16384 and B1 H1-H8 N4096 (d = 128), same output.
// A tile alone still takes ~0.95 of a pair's time per key tile (nothing
// overlaps its softmax), so where the tiles would fill more than one wave the
// split measured slower (0.6-0.75x) and pairs stay whole.
// kv_bytes: one head's K and V (0: no head groups).  Causal items are dealt
// heaviest first; for bf16 operands without sequence lengths, when the
// K and V of all heads exceed 96 MB (three quarters of L2) by three times or
// more, heads go in groups that fit it, heaviest first within each group, so a
// head's K/V tiles are re-read from L2 instead of DRAM.  On the causal B1 H32
// N16384 d128 workload (12-head groups) the DRAM traffic fell from 2.31 to
// 1.06 GB per launch at the same speed; 16-head groups (two) ran 7 % slower,
// hence the three-group minimum.
static long long plan_items(PrefillParams& p, int num_sms, long long kv_bytes) {
    const long long pairs = static_cast<long long>(p.num_pairs) * p.BH;
    long long grid = pairs < num_sms ? pairs : num_sms;
    long long items = pairs, split = pairs;
    if (p.causal && !p.seqlens_q && !p.seqlens_k && pairs <= num_sms) {
        split = 0;
        items = 2 * pairs;
        grid = items < num_sms ? items : num_sms;
    } else if (!p.causal && !p.seqlens_q && !p.seqlens_k && pairs > grid) {
        const long long full = pairs / grid * grid, tail = pairs - full;
        if (tail > 0 && 2 * tail <= grid && full + 2 * tail <= 0x7fffffffLL) {
            split = full;
            items = full + 2 * tail;
        }
    }
    p.n_items = static_cast<int>(items);
    p.split_start = static_cast<int>(split);
    const long long budget = 96LL << 20;
    long long hg = (kv_bytes > 0 && p.causal && !p.seqlens_q && !p.seqlens_k) ? budget / kv_bytes
                                                                              : p.BH;
    if (hg < 1) hg = 1;
    if (hg >= p.BH || (p.BH + hg - 1) / hg < 3 || split < pairs) hg = p.BH;
    p.head_group = static_cast<int>(hg);
    return grid;
}

template <int D>
static int launch_prefill_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const PrefillParams& params, int num_sms,
                            cudaStream_t stream) {
    using C = Cfg<D, false>;
    PrefillParams p = params;
    // head groups only for the bf16 d = 128 kernel without sequence lengths
    const long long grid = plan_items(p, num_sms, D == 128 ? 2LL * p.Nk * D * 2 : 0);
    const dim3 g(static_cast<unsigned>(grid));
    if (p.seqlens_q || p.seqlens_k) {
        attn_fwd_prefill_kernel<D, true, false><<<g, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv,
                                                                                     to, p);
    } else if (p.head_group < p.BH) {
        if constexpr (D == 128)
            attn_fwd_prefill_kernel<D, false, false, true>
                <<<g, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, p);
    } else {
        attn_fwd_prefill_kernel<D, false, false><<<g, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv,
                                                                                      to, p);
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& to, const PrefillParams& p, int num_sms,
                   cudaStream_t stream) {
    return d == 128 ? launch_prefill_d<128>(tq, tk, tv, to, p, num_sms, stream)
                    : launch_prefill_d<64>(tq, tk, tv, to, p, num_sms, stream);
}

int launch_prefill_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                       const CUtensorMap& to, const PrefillParams& params, int num_sms,
                       cudaStream_t stream) {
    using C = Cfg<128, true>;
    PrefillParams p = params;
    const long long grid = plan_items(p, num_sms, 0);  // no head groups here
    attn_fwd_prefill_kernel<128, false, true>
        <<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(tq, tk, tvt, to, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int prefill_smem_bytes(int d) {
    return d == 128 ? Cfg<128, false>::kSmemBytes : Cfg<64, false>::kSmemBytes;
}

unsigned read_and_clear_prefill_error() {
    unsigned v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof v);
    cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof zero);
    return v;
}

}  // namespace gbattn
