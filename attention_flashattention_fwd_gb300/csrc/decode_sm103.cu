// decode_sm103.cu -- single-query attention forward, split over the keys.
//
// Decode reads every key and value once and does about one FLOP per byte
// (CS336 Lecture 5 notes, section 5.3: decode is memory-bound), so the job is
// to stream K and V at HBM speed:
//   * the keys of one (b, h) are cut into `splits` contiguous ranges; one CTA
//     streams one range with coalesced 16-byte loads (a key row of d bf16 is
//     read by d/8 neighbouring lanes; the lanes of a warp read neighbouring
//     rows), bypassing L1 because nothing is read twice;
//   * each group of d/8 lanes keeps its own running max m and sum l and an
//     fp32 output slice (online softmax, CS336 Lecture 5 notes, section 8.2),
//     the groups of a CTA are merged through shared memory with the two-block
//     rule of CS149 Lecture 9 notes, concept 9, and the CTA writes a partial
//     (o_s, lse_s) to the workspace;
//   * a second, tiny kernel merges the splits of each (b, h) with the same rule
//     (the "second launch as a global barrier" of the PDC course, section 5.14)
//     and writes bf16 O and the fp32 logsumexp.  With a single split the first
//     kernel writes the final result itself.
// Scores are kept in base 2 (c = scale * log2 e) as in the prefill kernel.
#include <cuda_bf16.h>

#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

__device__ unsigned int g_decode_error = 0;

namespace {

constexpr int kDecThreads = 256;   // 8 warps
constexpr int kUnroll = 8;         // key rows in flight per lane group and iteration
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kDecMinKeysPerSplit = 512;  // a split streams at least this many keys

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// dot of 8 bf16 values packed in a uint4 with 8 fp32 values
__device__ __forceinline__ float dot8(const float (&q)[8], uint4 k) {
    float s = q[0] * bf_lo(k.x);
    s = fmaf(q[1], bf_hi(k.x), s);
    s = fmaf(q[2], bf_lo(k.y), s);
    s = fmaf(q[3], bf_hi(k.y), s);
    s = fmaf(q[4], bf_lo(k.z), s);
    s = fmaf(q[5], bf_hi(k.z), s);
    s = fmaf(q[6], bf_lo(k.w), s);
    s = fmaf(q[7], bf_hi(k.w), s);
    return s;
}

__device__ __forceinline__ void axpy8(float (&acc)[8], float p, uint4 v) {
    acc[0] = fmaf(p, bf_lo(v.x), acc[0]);
    acc[1] = fmaf(p, bf_hi(v.x), acc[1]);
    acc[2] = fmaf(p, bf_lo(v.y), acc[2]);
    acc[3] = fmaf(p, bf_hi(v.y), acc[3]);
    acc[4] = fmaf(p, bf_lo(v.z), acc[4]);
    acc[5] = fmaf(p, bf_hi(v.z), acc[5]);
    acc[6] = fmaf(p, bf_lo(v.w), acc[6]);
    acc[7] = fmaf(p, bf_hi(v.w), acc[7]);
}

__device__ __forceinline__ uint32_t ld_stream_u8(const uint8_t* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// Four E4M3 codes (lowest byte first) to fp32.  Every E4M3 value is an fp16
// value, so both conversions (E4M3 pairs to fp16 pairs, fp16 to fp32) are exact.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
    asm("{\n\t.reg .b16 lo, hi, a0, a1, a2, a3;\n\t.reg .b32 h01, h23;\n\t"
        "mov.b32 {lo, hi}, %4;\n\t"
        "cvt.rn.f16x2.e4m3x2 h01, lo;\n\tcvt.rn.f16x2.e4m3x2 h23, hi;\n\t"
        "mov.b32 {a0, a1}, h01;\n\tmov.b32 {a2, a3}, h23;\n\t"
        "cvt.f32.f16 %0, a0;\n\tcvt.f32.f16 %1, a1;\n\tcvt.f32.f16 %2, a2;\n\t"
        "cvt.f32.f16 %3, a3;\n\t}"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3])
        : "r"(w));
}

// Value of an E8M0 scale code (OCP MX v1.0): 2^(code - 127), built from its
// exponent bits; code 0 is 2^-127 (an fp32 subnormal), 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
    return __uint_as_float(code == 0u ? 0x00400000u : code == 255u ? 0x7fc00000u : code << 23);
}

// sum over 16 E4M3 codes (a uint4) of q[c] * value(code c), two lanes of
// work per instruction (packed fp32 FMA on (even, odd) element pairs)
__device__ __forceinline__ float dot16_e4m3(const float2 (&q)[8], uint4 k) {
    const uint32_t w[4] = {k.x, k.y, k.z, k.w};
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float f[4];
        e4m3x4_to_f32(w[i], f);
        s = ffma2(q[2 * i], make_float2(f[0], f[1]), s);
        s = ffma2(q[2 * i + 1], make_float2(f[2], f[3]), s);
    }
    return s.x + s.y;
}

// acc[c] += p * value(code c) over 16 E4M3 codes, acc as (even, odd) pairs
__device__ __forceinline__ void axpy16_e4m3(float2 (&acc)[8], float p, uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float2 p2 = make_float2(p, p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float f[4];
        e4m3x4_to_f32(w[i], f);
        acc[2 * i] = ffma2(p2, make_float2(f[0], f[1]), acc[2 * i]);
        acc[2 * i + 1] = ffma2(p2, make_float2(f[2], f[3]), acc[2 * i + 1]);
    }
}

}  // namespace

// One CTA = one (b, h, split).  Lane group g (d/8 lanes) handles keys
// ks + g, ks + g + G, ... where G = lane groups per CTA.
template <int D>
__global__ void __launch_bounds__(kDecThreads)
    attn_fwd_decode_split_kernel(DecodeParams p) {
    constexpr int kLanesPerRow = D / 8;              // 16 (d=128) or 8 (d=64)
    constexpr int kGroupsPerWarp = 32 / kLanesPerRow;
    constexpr int kGroups = (kDecThreads / 32) * kGroupsPerWarp;

    __shared__ float sm_m[kGroups];
    __shared__ float sm_l[kGroups];
    __shared__ float sm_acc[kGroups][D];

    const int bh = blockIdx.x / p.splits;
    const int split = blockIdx.x % p.splits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp * kGroupsPerWarp + lane / kLanesPerRow;
    const int sub = lane % kLanesPerRow;  // which 8-element slice of the row

    // keys of this (b, h): all Nk, or the sequence's own count (a count out
    // of range is reported and gives the sequence no keys: o = 0, lse = -inf)
    int nk = p.Nk;
    if (p.seqlens_k) {
        nk = gb_index_ok(&g_decode_error, bh / p.H, bh / p.H, p.BH / p.H) ? p.seqlens_k[bh / p.H] : 0;
        if (nk < 1 || nk > p.Nk) {
            if (threadIdx.x == 0) atomicOr(&g_decode_error, kErrBitLengths);
            nk = 0;
        }
    }
    const int ks = split * p.keys_per_split;
    const int ke = min(nk, ks + p.keys_per_split);

    const long long n_kv = static_cast<long long>(p.BH) * p.Nk * D;  // elements of k, v
    float q[8];
    {
        const long long qi = static_cast<long long>(bh) * D + sub * 8;
        const uint4 qr = gb_index_ok(&g_decode_error, qi, qi + 7, static_cast<long long>(p.BH) * D)
                             ? *reinterpret_cast<const uint4*>(p.q + qi)
                             : make_uint4(0, 0, 0, 0);
        q[0] = bf_lo(qr.x); q[1] = bf_hi(qr.x); q[2] = bf_lo(qr.y); q[3] = bf_hi(qr.y);
        q[4] = bf_lo(qr.z); q[5] = bf_hi(qr.z); q[6] = bf_lo(qr.w); q[7] = bf_hi(qr.w);
        // fold scale * log2(e) into q once
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] *= p.scale_log2;
    }
    const __nv_bfloat16* kbase = p.k + static_cast<size_t>(bh) * p.Nk * D + sub * 8;
    const __nv_bfloat16* vbase = p.v + static_cast<size_t>(bh) * p.Nk * D + sub * 8;

    float m = -INFINITY, l = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;

    for (int base = ks; base < ke; base += kGroups * kUnroll) {
        uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = base + u * kGroups + g;
            const long long e0 = (static_cast<long long>(bh) * p.Nk + j) * D + sub * 8;
            if (j < ke && gb_index_ok(&g_decode_error, e0, e0 + 7, n_kv)) {
                kr[u] = ld_stream(kbase + static_cast<size_t>(j) * D);
                vr[u] = ld_stream(vbase + static_cast<size_t>(j) * D);
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float s[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) s[u] = dot8(q, kr[u]);
        // sum the d/8 partial dots of each row across its lane group
#pragma unroll
        for (int off = kLanesPerRow / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
        float mx = m;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (base + u * kGroups + g >= ke) s[u] = -INFINITY;
            mx = fmaxf(mx, s[u]);
        }
        if (mx == -INFINITY) continue;  // every key of this group is past the range
        const float alpha = ex2_approx(m - mx);  // m = -inf on the first visit gives 0
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float pu = ex2_approx(s[u] - mx);
            l += pu;
            axpy8(acc, pu, vr[u]);
        }
        m = mx;
    }

    // ---- merge the lane groups of the CTA
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_acc[g][sub * 8 + e] = acc[e];
    if (sub == 0) {
        sm_m[g] = m;
        sm_l[g] = l;
    }
    __syncthreads();
    if (threadIdx.x < D) {
        const int c = threadIdx.x;
        float M = -INFINITY;
#pragma unroll 4
        for (int i = 0; i < kGroups; ++i) M = fmaxf(M, sm_m[i]);
        float Lsum = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int i = 0; i < kGroups; ++i) {
                if (sm_m[i] == -INFINITY) continue;
                const float w = ex2_approx(sm_m[i] - M);
                Lsum = fmaf(w, sm_l[i], Lsum);
                O = fmaf(w, sm_acc[i][c], O);
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        if (p.splits == 1) {
            const long long oi = static_cast<long long>(bh) * D + c;
            if (gb_index_ok(&g_decode_error, oi, oi, static_cast<long long>(p.BH) * D))
                p.o[oi] = __float2bfloat16_rn(O * inv);
            if (c == 0 && gb_index_ok(&g_decode_error, bh, bh, p.BH))
                p.lse[bh] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
        } else {
            const long long ps = static_cast<long long>(bh) * p.splits + split;
            const long long n_ps = static_cast<long long>(p.BH) * p.splits;
            if (gb_index_ok(&g_decode_error, ps * D + c, ps * D + c, n_ps * D))
                p.part_o[ps * D + c] = O * inv;
            if (c == 0 && gb_index_ok(&g_decode_error, ps, ps, n_ps))
                p.part_lse[ps] = Lsum > 0.f ? M + log2f(Lsum) : -INFINITY;
        }
    }
}

// MXFP8 keys and values (E4M3 codes, one E8M0 scale per 32 consecutive
// elements of a row: the microscaling formats of the PDC course, Lecture 7,
// section 7.14): the split kernel above with one byte per element.  A key row
// of d codes is read by d/16 neighbouring lanes (16 codes per 16-byte load), so
// a lane's slice lies in one scale block: the lane multiplies its partial dot
// by the key's block scale before the lane group sums the slices, and folds
// the value's block scale into the probability before its axpy.  Every code
// is widened exactly (E4M3 -> fp16 -> fp32); the arithmetic is the bf16
// kernel's, so the decode reads 1 + 1/32 bytes per K and V element instead of 2.
template <int D>
__global__ void __launch_bounds__(kDecThreads, 2)
    attn_fwd_decode_mx_split_kernel(DecodeParams p) {
    constexpr int kLanesPerRow = D / 16;             // 8 (d=128) or 4 (d=64)
    constexpr int kGroupsPerWarp = 32 / kLanesPerRow;
    constexpr int kGroups = (kDecThreads / 32) * kGroupsPerWarp;
    constexpr int kNb = D / 32;                      // scale blocks per row

    __shared__ float sm_m[kGroups];
    __shared__ float sm_l[kGroups];
    __shared__ float sm_acc[kGroups][D];

    const int bh = blockIdx.x / p.splits;
    const int split = blockIdx.x % p.splits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp * kGroupsPerWarp + lane / kLanesPerRow;
    const int sub = lane % kLanesPerRow;  // which 16-element slice of the row
    const int ks = split * p.keys_per_split;
    const int ke = min(p.Nk, ks + p.keys_per_split);

    const long long n_kv = static_cast<long long>(p.BH) * p.Nk * D;  // codes of k8, v8
    float2 q[8];  // the lane's 16 elements as (even, odd) pairs
    {
        const long long qi = static_cast<long long>(bh) * D + sub * 16;
        const uint4* qp = reinterpret_cast<const uint4*>(p.q + qi);
        const bool q_ok = gb_index_ok(&g_decode_error, qi, qi + 15, static_cast<long long>(p.BH) * D);
        const uint4 a = q_ok ? qp[0] : make_uint4(0, 0, 0, 0);
        const uint4 b = q_ok ? qp[1] : make_uint4(0, 0, 0, 0);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)  // fold scale * log2(e) into q once
            q[i] = make_float2(bf_lo(w[i]) * p.scale_log2, bf_hi(w[i]) * p.scale_log2);
    }
    const uint8_t* k8 = reinterpret_cast<const uint8_t*>(p.k);
    const uint8_t* v8 = reinterpret_cast<const uint8_t*>(p.v);
    const uint8_t* kbase = k8 + static_cast<size_t>(bh) * p.Nk * D + sub * 16;
    const uint8_t* vbase = v8 + static_cast<size_t>(bh) * p.Nk * D + sub * 16;
    const uint8_t* ksbase = p.k_scale + static_cast<size_t>(bh) * p.Nk * kNb + sub / 2;
    const uint8_t* vsbase = p.v_scale + static_cast<size_t>(bh) * p.Nk * kNb + sub / 2;

    float m = -INFINITY, l = 0.f;
    float2 acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = make_float2(0.f, 0.f);

    for (int base = ks; base < ke; base += kGroups * kUnroll) {
        uint4 kr[kUnroll], vr[kUnroll];
        uint32_t kx[kUnroll], vx[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = base + u * kGroups + g;
            const long long e0 = (static_cast<long long>(bh) * p.Nk + j) * D + sub * 16;
            const long long x0 = (static_cast<long long>(bh) * p.Nk + j) * kNb + sub / 2;
            if (j < ke && gb_index_ok(&g_decode_error, e0, e0 + 15, n_kv) &&
                gb_index_ok(&g_decode_error, x0, x0, n_kv / 32)) {
                kr[u] = ld_stream(kbase + static_cast<size_t>(j) * D);
                vr[u] = ld_stream(vbase + static_cast<size_t>(j) * D);
                kx[u] = ld_stream_u8(ksbase + static_cast<size_t>(j) * kNb);
                vx[u] = ld_stream_u8(vsbase + static_cast<size_t>(j) * kNb);
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
                kx[u] = 127u;
                vx[u] = 127u;
            }
        }
        float s[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) s[u] = dot16_e4m3(q, kr[u]) * e8m0_to_f32(kx[u]);
        // sum the d/16 partial dots of each row across its lane group
#pragma unroll
        for (int off = kLanesPerRow / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
        float mx = m;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (base + u * kGroups + g >= ke) s[u] = -INFINITY;
            mx = fmaxf(mx, s[u]);
        }
        if (mx == -INFINITY) continue;  // every key of this group is past the range
        const float alpha = ex2_approx(m - mx);  // m = -inf on the first visit gives 0
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = make_float2(acc[e].x * alpha, acc[e].y * alpha);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float pu = ex2_approx(s[u] - mx);
            l += pu;
            axpy16_e4m3(acc, pu * e8m0_to_f32(vx[u]), vr[u]);
        }
        m = mx;
    }

    // ---- merge the lane groups of the CTA (as in the bf16 kernel)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        sm_acc[g][sub * 16 + 2 * e] = acc[e].x;
        sm_acc[g][sub * 16 + 2 * e + 1] = acc[e].y;
    }
    if (sub == 0) {
        sm_m[g] = m;
        sm_l[g] = l;
    }
    __syncthreads();
    if (threadIdx.x < D) {
        const int c = threadIdx.x;
        float M = -INFINITY;
#pragma unroll 4
        for (int i = 0; i < kGroups; ++i) M = fmaxf(M, sm_m[i]);
        float Lsum = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int i = 0; i < kGroups; ++i) {
                if (sm_m[i] == -INFINITY) continue;
                const float w = ex2_approx(sm_m[i] - M);
                Lsum = fmaf(w, sm_l[i], Lsum);
                O = fmaf(w, sm_acc[i][c], O);
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        if (p.splits == 1) {
            const long long oi = static_cast<long long>(bh) * D + c;
            if (gb_index_ok(&g_decode_error, oi, oi, static_cast<long long>(p.BH) * D))
                p.o[oi] = __float2bfloat16_rn(O * inv);
            if (c == 0 && gb_index_ok(&g_decode_error, bh, bh, p.BH))
                p.lse[bh] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
        } else {
            const long long ps = static_cast<long long>(bh) * p.splits + split;
            const long long n_ps = static_cast<long long>(p.BH) * p.splits;
            if (gb_index_ok(&g_decode_error, ps * D + c, ps * D + c, n_ps * D))
                p.part_o[ps * D + c] = O * inv;
            if (c == 0 && gb_index_ok(&g_decode_error, ps, ps, n_ps))
                p.part_lse[ps] = Lsum > 0.f ? M + log2f(Lsum) : -INFINITY;
        }
    }
}

// Merge the splits of one (b, h): lse = log2 sum_s 2^{lse_s},
// o = sum_s 2^{lse_s - lse} o_s.  One CTA per (b, h), one thread per column.
template <int D>
__global__ void __launch_bounds__(D) attn_fwd_decode_combine_kernel(DecodeParams p) {
    const int bh = blockIdx.x;
    const int c = threadIdx.x;
    const float* pl = p.part_lse + static_cast<size_t>(bh) * p.splits;
    const float* po = p.part_o + static_cast<size_t>(bh) * p.splits * D;
    const long long n_ps = static_cast<long long>(p.BH) * p.splits;
    const long long ps0 = static_cast<long long>(bh) * p.splits;
    if (!gb_index_ok(&g_decode_error, ps0, ps0 + p.splits - 1, n_ps) ||
        !gb_index_ok(&g_decode_error, bh, bh, p.BH))
        return;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, pl[s]);
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < p.splits; ++s) {
            if (pl[s] == -INFINITY) continue;
            const float w = ex2_approx(pl[s] - M);
            Lsum += w;
            O = fmaf(w, po[static_cast<size_t>(s) * D + c], O);
        }
    }
    p.o[static_cast<size_t>(bh) * D + c] = __float2bfloat16_rn(Lsum > 0.f ? O / Lsum : 0.f);
    if (c == 0) p.lse[bh] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ host side

// Split policy: aim for 16 CTAs per SM of the device (num_sms), never fewer
// than 512 keys per split, at most 64 splits.  Pure arithmetic on the sizes.
void decode_split_plan(long long BH, int Nk, int num_sms, int* splits, int* keys_per_split) {
    const long long target_ctas = 16LL * (num_sms > 0 ? num_sms : 1);
    long long s = (target_ctas + BH - 1) / BH;
    const long long max_by_keys = (Nk + kDecMinKeysPerSplit - 1) / kDecMinKeysPerSplit;
    if (s > max_by_keys) s = max_by_keys;
    if (s > kDecodeMaxSplits) s = kDecodeMaxSplits;
    if (s < 1) s = 1;
    int kps = static_cast<int>((Nk + s - 1) / s);
    s = (Nk + kps - 1) / kps;  // no empty split
    *splits = static_cast<int>(s);
    *keys_per_split = kps;
}

size_t decode_partials_bytes(long long BH, int splits, int d) {
    if (splits <= 1) return 0;
    const size_t n = static_cast<size_t>(BH) * splits;
    // partial outputs [BH, splits, d] fp32, then partial lse [BH, splits] fp32
    return n * d * sizeof(float) + n * sizeof(float);
}

// The most splits the plan takes on any device: the bound depends on the
// sizes alone, so the workspace a caller sizes on one machine fits every GPU.
size_t decode_workspace_bytes(long long BH, int Nk, int d) {
    long long s = (Nk + kDecMinKeysPerSplit - 1) / kDecMinKeysPerSplit;
    if (s > kDecodeMaxSplits) s = kDecodeMaxSplits;
    return decode_partials_bytes(BH, static_cast<int>(s), d);
}

int launch_decode(int d, const DecodeParams& p, cudaStream_t stream) {
    const long long grid = static_cast<long long>(p.BH) * p.splits;
    if (d == 128) {
        attn_fwd_decode_split_kernel<128><<<static_cast<unsigned>(grid), kDecThreads, 0, stream>>>(p);
        if (p.splits > 1)
            attn_fwd_decode_combine_kernel<128><<<p.BH, 128, 0, stream>>>(p);
    } else {
        attn_fwd_decode_split_kernel<64><<<static_cast<unsigned>(grid), kDecThreads, 0, stream>>>(p);
        if (p.splits > 1)
            attn_fwd_decode_combine_kernel<64><<<p.BH, 64, 0, stream>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_decode_mx(int d, const DecodeParams& p, cudaStream_t stream) {
    const long long grid = static_cast<long long>(p.BH) * p.splits;
    if (d == 128) {
        attn_fwd_decode_mx_split_kernel<128>
            <<<static_cast<unsigned>(grid), kDecThreads, 0, stream>>>(p);
        if (p.splits > 1)
            attn_fwd_decode_combine_kernel<128><<<p.BH, 128, 0, stream>>>(p);
    } else {
        attn_fwd_decode_mx_split_kernel<64>
            <<<static_cast<unsigned>(grid), kDecThreads, 0, stream>>>(p);
        if (p.splits > 1)
            attn_fwd_decode_combine_kernel<64><<<p.BH, 64, 0, stream>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

unsigned read_and_clear_decode_error() {
    unsigned v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_decode_error, sizeof v);
    cudaMemcpyToSymbol(g_decode_error, &zero, sizeof zero);
    return v;
}

}  // namespace gbattn
