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
// The kernel applies the rule in its online form (a running max, earlier
// partial sums rescaled when it grows), so all loads of a batch of parts are
// issued before any of them is used.
// D / 8 neighbouring lanes share a row, 16-byte loads of 8 bf16 each.
#include <cuda_bf16.h>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

template <int D>
__global__ void __launch_bounds__(256, 4) attn_merge_kernel(MergeParams p) {
    constexpr int kLanes = D / 8;
    constexpr int kBatch = 4;  // parts whose loads are in flight together
    const long long total = p.rows * kLanes;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const size_t part_rows = static_cast<size_t>(p.rows);
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
         g += stride) {
        const long long row = g / kLanes;
        const int c = static_cast<int>(g % kLanes) * 8;
        // one pass with a running max (the online form of the merge rule): a
        // batch's lse and o loads do not wait on each other
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
                if (s < p.n_parts) {
                    ls[b] = p.lse_parts[s * part_rows + row];
                    raw[b] = *reinterpret_cast<const uint4*>(p.o_parts + (s * part_rows + row) * D + c);
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
        *reinterpret_cast<uint4*>(p.o + row * D + c) = out;
        if (c == 0) p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;
    }
}

int launch_merge(int d, const MergeParams& p, int num_sms, cudaStream_t stream) {
    const long long threads = p.rows * (d / 8);
    long long blocks = (threads + 255) / 256;
    if (blocks > 64LL * num_sms) blocks = 64LL * num_sms;
    if (d == 128)
        attn_merge_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    else
        attn_merge_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace gbattn
