// gbattn_internal.h -- declarations shared by the host API and the kernel
// translation units of libgbattn.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gbattn.h"  // include/ is on the include path

namespace gbattn {

// Arguments of the prefill kernel besides the three TMA descriptors.
struct PrefillParams {
    __nv_bfloat16* o;   // [BH, Nq, d]
    float* lse;         // [BH, Nq]
    int Nq, Nk, BH;
    int num_pairs;      // query-tile pairs per head: ceil(Nq / 256)
    int causal;         // query i sees keys j <= i + (nk - nq) of its sequence
    float scale_log2;   // scale * log2(e)
    int H;
    const int* seqlens_q;  // [B] per-sequence query counts, or null (all Nq)
    const int* seqlens_k;  // [B] per-sequence key counts, or null (all Nk)
    float o_scale;         // FP8 operands: the value descale applied to O / l
    // Set by the launcher: the number of work items, and the first of them that
    // is a single 128-row query tile (items split_start + 2 i and + 2 i + 1 are
    // the two halves of query-tile pair split_start + i; no split when
    // split_start == n_items).
    int n_items, split_start;
    // Set by the launcher: causal items are dealt in groups of this many heads.
    int head_group;
};

// Arguments of the split-K decode kernels.
struct DecodeParams {
    const __nv_bfloat16* q;  // [BH, d]
    const __nv_bfloat16* k;  // [BH, Nk, d]
    const __nv_bfloat16* v;  // [BH, Nk, d]
    __nv_bfloat16* o;        // [BH, d]
    float* lse;              // [BH]
    float* part_o;           // [BH, splits, d]   (workspace)
    float* part_lse;         // [BH, splits]      (workspace), log2 units
    int BH, Nk, splits, keys_per_split;
    float scale_log2;
    int H;
    const int* seqlens_k;    // [B] per-sequence key counts, or null (all Nk)
    // MXFP8 keys and values (attn_fwd_decode_mx): k and v then point at E4M3
    // codes [BH, Nk, d] and these at the E8M0 block scales [BH, Nk, d / 32]
    const uint8_t* k_scale;
    const uint8_t* v_scale;
};

// Arguments of the backward preprocessing kernel.
struct BwdPrepParams {
    const __nv_bfloat16* o;     // [BH, Nq, d]
    const __nv_bfloat16* dout;  // [BH, Nq, d]
    const float* lse;           // [BH, Nq], natural log
    float* nl2;                 // [BH, Nq_pad] -lse * log2(e); -inf on padded rows
    float* nD;                  // [BH, Nq_pad] -rowsum(dO * O); 0 on padded rows
    float* dq_acc;              // [BH, Nq_pad, d], zeroed
    long long rows;             // BH * Nq_pad
    int Nq, Nq_pad;
};

// Arguments of the backward main kernel besides the four TMA descriptors.
struct BwdParams {
    __nv_bfloat16* dk;   // [BH, Nk, d]
    __nv_bfloat16* dv;   // [BH, Nk, d]
    float* dq_acc;       // [BH, Nq_pad, d]
    const float* nl2;    // [BH, Nq_pad] -lse * log2(e)
    const float* nD;     // [BH, Nq_pad] -D
    int Nq, Nk, Nq_pad, BH;
    int n_kt;            // key tiles per head: ceil(Nk / 128)
    // CTAs are ordered in groups of head_group heads: within a group by key
    // tile (most query tiles first), then by head, so the CTAs in flight at
    // once share the Q, dO and dQ accumulator rows of a few heads in L2
    int head_group;
    int causal, causal_off;
    float scale, scale_log2;
};

// Arguments of the merge kernel.
struct MergeParams {
    const __nv_bfloat16* o_parts;  // [n_parts, rows, d]
    const float* lse_parts;        // [n_parts, rows], natural log
    __nv_bfloat16* o;              // [rows, d]
    float* lse;                    // [rows]
    long long rows;                // B * H * Nq
    int n_parts;
};

// gbattn_api.cu: streaming multiprocessors of the current device (cached per
// device ordinal).
int current_sm_count(int* out);

// prefill_sm103.cu
int prefill_set_attributes();
// Persistent launch: min(work items, num_sms) CTAs, one per SM.
// `to` maps O [BH, Nq, d] in boxes of 32 x 32 x 1 with the 64-byte swizzle (the
// target of the epilogue's TMA stores; unused with per-sequence lengths).
int launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& to, const PrefillParams& p, int num_sms,
                   cudaStream_t stream);
// E4M3 operands, d = 128; tvt maps the transposed values [BH, d, Nk].
int launch_prefill_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                       const CUtensorMap& to, const PrefillParams& p, int num_sms,
                       cudaStream_t stream);
int prefill_smem_bytes(int d);
unsigned read_and_clear_prefill_error();

// prefill_pair_sm103.cu: bf16, d = 128, no per-sequence lengths, on CTA pairs.
// p.num_pairs counts quads (four 128-row query tiles) per head; tk64 maps K in
// boxes of 64 x 64 x 1 (the half key tile each CTA of a pair holds).
int prefill_pair_set_attributes();
int launch_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv,
                        const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream);
unsigned read_and_clear_prefill_pair_error();
constexpr int kMaxDevices = 64;  // device ordinals the per-device caches cover
// Device error bits (shared by the kernels' error words)
constexpr unsigned kErrBitTimeout = 1u;  // a bounded barrier wait ran out
constexpr unsigned kErrBitLengths = 4u;  // a per-sequence length was out of range
constexpr unsigned kErrBitBounds = 8u;   // debug builds: an out-of-range access was skipped

// One lane of a converged warp: elect.sync picks the same lane for the same
// member mask every time, so the lane that issues a group of tcgen05.mma
// products also issues every commit that tracks them.  The kernels' MMA warps
// run their loops and barrier waits with all 32 lanes and issue from the
// elected one: a lone issuing lane whose loop holds barrier waits issues every
// product markedly slower (attn_bench_mma_rate measures both forms).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Debug builds (-DGBATTN_DEBUG: libgbattn_debug.so) check every direct global
// memory access of the kernels -- the ones a TMA tensor map does not bound --
// against its buffer: elements first .. last of an n-element buffer.  Out of
// range, the kernel sets kErrBitBounds in its error word and skips the access
// (attn_device_error reports ATTN_ERR_OUT_OF_RANGE); nothing traps.  Release
// builds compile the check away.
__device__ __forceinline__ bool gb_index_ok(unsigned int* err, long long first, long long last,
                                            long long n) {
#ifdef GBATTN_DEBUG
    if (first >= 0 && last < n) return true;
    atomicOr(err, kErrBitBounds);
    return false;
#else
    (void)err;
    (void)first;
    (void)last;
    (void)n;
    return true;
#endif
}

// decode_sm103.cu
// Splits of each (b, h)'s keys for a device with num_sms SMs (at most
// kDecodeMaxSplits).
constexpr int kDecodeMaxSplits = 64;
void decode_split_plan(long long BH, int Nk, int num_sms, int* splits, int* keys_per_split);
// Bytes of the split partials of a plan with `splits` splits (0 for one split).
size_t decode_partials_bytes(long long BH, int splits, int d);
// Workspace the caller provides: the partials of the largest plan any device
// takes for these sizes (depends on the sizes alone).
size_t decode_workspace_bytes(long long BH, int Nk, int d);
int launch_decode(int d, const DecodeParams& p, cudaStream_t stream);
// the same split + combine kernels on MXFP8 keys and values
int launch_decode_mx(int d, const DecodeParams& p, cudaStream_t stream);
unsigned read_and_clear_decode_error();

// selftest_sm103.cu
int launch_selftest_timeout(cudaStream_t stream);
// debug builds: a kernel whose index check fails on purpose (no access made)
int launch_selftest_bounds(cudaStream_t stream);
unsigned read_and_clear_selftest_error();

// mma_pair_sm103.cu: the cta_group::2 product checked and timed against the
// single-CTA form (blocking calls; each synchronises `stream`)
int launch_pair_product(const void* a, const void* b, float* d, cudaStream_t stream);
int run_mma_rate(int form, int issuer, int busy, int waits, int steps, int reps, float* ms_out,
                 double* cycles_out, int* sms_out, cudaStream_t stream);

// merge_sm103.cu
int launch_merge(int d, const MergeParams& p, int num_sms, cudaStream_t stream);
unsigned read_and_clear_merge_error();

// backward_sm103.cu
int bwd_set_attributes();
size_t bwd_workspace_bytes(long long BH, int Nq, int d);
// prep, main (one CTA per key tile and head) and dQ convert kernels, in order.
// tdqacc: the fp32 dQ accumulator [BH, Nq_pad, d] as 32 x 128 x 1 boxes with
// the 128-byte swizzle.
int launch_backward(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                    const CUtensorMap& tdo, const CUtensorMap& tdqacc, const BwdPrepParams& a,
                    const BwdParams& p, __nv_bfloat16* dq, int num_sms, cudaStream_t stream);
unsigned read_and_clear_bwd_error();

}  // namespace gbattn
