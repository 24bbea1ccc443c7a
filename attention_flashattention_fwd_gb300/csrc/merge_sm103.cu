// merge_sm103.cu -- merge of attention results computed over disjoint key sets.
//
// With the keys (and values) of every (b, h) split into S disjoint parts,
// part s gives o_s = softmax over its keys applied to its values and its
// logsumexp lse_s.  The two-block merge rule of the CS149 Lecture 9 notes,
// concept 9 (m = max(m1, m2), l = e^{m1-m} l1 + e^{m2-m} l2), applied to S
// blocks, with m_s + log l_s = lse_s:
//     lse = M + log sum_s e^{lse_s - M},    M = max_s lse_s
//     o   = sum_s e^{lse_s - lse} o_s
// is the attention over all keys.  This is the one exchange step of key
// (context) parallel attention: each rank attends to its key shard, the
// (o_s, lse_s) are gathered, and this kernel merges them.  A part with
// lse_s = -inf (no visible key) has weight 0.
//
// Memory bound: every row reads S * (2 d + 4) bytes and writes 2 d + 4.
// D / 8 neighbouring lanes share a row, 16-byte loads of 8 bf16 each, read
// once and not kept in L1; a persistent grid (4 CTAs per SM) strides over the
// (row, 8-column chunk) units.  With at most 4 parts a thread loads every part
// of two units before using any (8 loads in flight) and merges each unit
// against its own largest lse: about 6 TB/s on 4 parts of the B=2, H=16,
// N=4096, d=128 shape, against 5.2 with one unit per thread and a CTA per
// 256 units.  With more parts the rule runs in its online form, 4 parts at a
// time (a running max, earlier partial sums rescaled when it grows).
#include <cuda_bf16.h>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

__device__ unsigned int g_merge_error = 0;  // debug builds: kErrBitBounds

namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

constexpr int kMergeThreads = 256;
constexpr int kMergeCtasPerSm = 4;

}  // namespace

// Every part's weight against the row's largest lse, one (row, 8-column
// chunk) unit: w_s = e^{lse_s - M}, o = sum_s w_s o_s / sum_s w_s.
template <int D, int kParts>
__device__ __forceinline__ void merge_unit(const MergeParams& p, long long g, const float (&ls)[kParts],
                                           const uint4 (&raw)[kParts]) {
    constexpr int kLanes = D / 8;
    const long long row = g / kLanes;
    const int c = static_cast<int>(g % kLanes) * 8;
    float M = -INFINITY;
#pragma unroll
    for (int b = 0; b < kParts; ++b) M = fmaxf(M, ls[b]);
    float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
#pragma unroll
        for (int b = 0; b < kParts; ++b) {
            if (ls[b] == -INFINITY) continue;  // an empty part: no weight, its o unused
            const float w = ex2_approx((ls[b] - M) * 1.4426950408889634f);
            L += w;
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[b]);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 f = __bfloat1622float2(h[t]);
                acc[2 * t] = fmaf(w, f.x, acc[2 * t]);
                acc[2 * t + 1] = fmaf(w, f.y, acc[2 * t + 1]);
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4 out;
    out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    if (gb_index_ok(&g_merge_error, row * D + c, row * D + c + 7, p.rows * D))
        *reinterpret_cast<uint4*>(p.o + row * D + c) = out;
    if (c == 0 && gb_index_ok(&g_merge_error, row, row, p.rows))
        p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;
}

// At most 4 parts: every load of two units (2 x 4 parts) in flight before any
// is used, then each unit merged against its own maximum.
template <int D>
__global__ void __launch_bounds__(kMergeThreads, kMergeCtasPerSm)
    attn_merge_small_kernel(MergeParams p) {
    constexpr int kLanes = D / 8;
    constexpr int kParts = 4;
    const long long total = p.rows * kLanes;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const size_t part_rows = static_cast<size_t>(p.rows);
    for (long long g0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g0 < total;
         g0 += 2 * stride) {
        float ls[2][kParts];
        uint4 raw[2][kParts];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const long long g = g0 + u * stride;
            const long long row = g / kLanes;
            const int c = static_cast<int>(g % kLanes) * 8;
#pragma unroll
            for (int s = 0; s < kParts; ++s) {
                ls[u][s] = -INFINITY;
                raw[u][s] = make_uint4(0u, 0u, 0u, 0u);
                const long long pr = s * static_cast<long long>(part_rows) + row;
                if (g < total && s < p.n_parts &&
                    gb_index_ok(&g_merge_error, pr * D + c, pr * D + c + 7,
                                p.n_parts * p.rows * D)) {
                    ls[u][s] = p.lse_parts[pr];
                    raw[u][s] = ld_stream(p.o_parts + pr * D + c);
                }
            }
        }
        merge_unit<D>(p, g0, ls[0], raw[0]);
        if (g0 + stride < total) merge_unit<D>(p, g0 + stride, ls[1], raw[1]);
    }
}

// Any number of parts: one unit per thread, the parts in batches of 4 whose
// loads are in flight together, a running max across batches (earlier sums
// rescaled when it grows: the online form of the rule).
template <int D>
__global__ void __launch_bounds__(kMergeThreads, kMergeCtasPerSm) attn_merge_kernel(MergeParams p) {
    constexpr int kLanes = D / 8;
    constexpr int kBatch = 4;
    const long long total = p.rows * kLanes;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const size_t part_rows = static_cast<size_t>(p.rows);
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
         g += stride) {
        const long long row = g / kLanes;
        const int c = static_cast<int>(g % kLanes) * 8;
        float M = -INFINITY, L = 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < p.n_parts; s0 += kBatch) {
            float ls[kBatch];
            uint4 raw[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int s = s0 + b;
                ls[b] = -INFINITY;
                raw[b] = make_uint4(0u, 0u, 0u, 0u);
                const long long pr = s * static_cast<long long>(part_rows) + row;
                if (s < p.n_parts && gb_index_ok(&g_merge_error, pr * D + c, pr * D + c + 7,
                                                 p.n_parts * p.rows * D)) {
                    ls[b] = p.lse_parts[pr];
                    raw[b] = ld_stream(p.o_parts + pr * D + c);
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (ls[b] == -INFINITY) continue;  // an empty part: no weight, its o unused
                const float m_new = fmaxf(M, ls[b]);
                const float keep = ex2_approx((M - m_new) * 1.4426950408889634f);  // 0 when M = -inf
                const float w = ex2_approx((ls[b] - m_new) * 1.4426950408889634f);
                L = L * keep + w;
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[b]);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 f = __bfloat1622float2(h[t]);
                    acc[2 * t] = fmaf(w, f.x, acc[2 * t] * keep);
                    acc[2 * t + 1] = fmaf(w, f.y, acc[2 * t + 1] * keep);
                }
                M = m_new;
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        uint4 out;
        out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        if (gb_index_ok(&g_merge_error, row * D + c, row * D + c + 7, p.rows * D))
            *reinterpret_cast<uint4*>(p.o + row * D + c) = out;
        if (c == 0 && gb_index_ok(&g_merge_error, row, row, p.rows))
            p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;
    }
}

template <int D>
static void launch_merge_d(const MergeParams& p, unsigned blocks, cudaStream_t stream) {
    if (p.n_parts <= 4)
        attn_merge_small_kernel<D><<<blocks, kMergeThreads, 0, stream>>>(p);
    else
        attn_merge_kernel<D><<<blocks, kMergeThreads, 0, stream>>>(p);
}

int launch_merge(int d, const MergeParams& p, int num_sms, cudaStream_t stream) {
    const long long threads = p.rows * (d / 8);
    long long blocks = (threads + kMergeThreads - 1) / kMergeThreads;
    if (blocks > static_cast<long long>(kMergeCtasPerSm) * num_sms)
        blocks = static_cast<long long>(kMergeCtasPerSm) * num_sms;
    if (d == 128)
        launch_merge_d<128>(p, static_cast<unsigned>(blocks), stream);
    else
        launch_merge_d<64>(p, static_cast<unsigned>(blocks), stream);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

unsigned read_and_clear_merge_error() {
    unsigned v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_merge_error, sizeof v);
    cudaMemcpyToSymbol(g_merge_error, &zero, sizeof zero);
    return v;
}

}  // namespace gbattn
