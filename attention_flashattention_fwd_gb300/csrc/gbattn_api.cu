// gbattn_api.cu -- the extern "C" entry points of libgbattn (declared in
// include/gbattn.h): argument validation, TMA descriptor encoding and kernel
// launches.  Every check happens before the first CUDA call, so a rejected
// call launches nothing.
#include <atomic>
#include <cmath>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include <cudaTypedefs.h>

#include "gbattn_internal.h"

using namespace gbattn;

namespace {

constexpr int kVersion = 100;  // 0.1.0

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks of attn_fwd and attn_fwd_from_host (no CUDA call).
int validate_fwd(const void* q, const void* k, const void* v, const void* o, const void* lse,
                 int B, int H, int Nq, int Nk, int d, int causal, float scale) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (causal && Nq > Nk) return ATTN_ERR_UNSUPPORTED;  // rows with no visible key
    // query positions i + (Nk - Nq) and padded tile rows stay within int32
    if (static_cast<long long>(Nq) + Nk + 512 > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    // grid and TMA coordinate range: (b*H + h) and the CTA count fit in int32
    const long long pairs = (static_cast<long long>(Nq) + 255) / 256;
    if (BH > 0x7fffffffLL || BH * pairs > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}


// The driver's tensor-map encoder: looked up once per process.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_encode_status = ATTN_OK;
std::once_flag g_encode_once;

void init_encode() {
    cudaDriverEntryPointQueryResult qres;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) != cudaSuccess ||
        qres != cudaDriverEntryPointSuccess || fn == nullptr) {
        g_encode_status = ATTN_ERR_CUDA;
        return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Kernel attributes (the large dynamic shared memory opt-in) belong to the
// device context they are set in, so they are set once per device.
std::once_flag g_attr_once[kMaxDevices];
int g_attr_status[kMaxDevices];

int ensure_init() {
    std::call_once(g_encode_once, init_encode);
    if (g_encode_status != ATTN_OK) return g_encode_status;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::call_once(g_attr_once[dev], [dev] {
        int st = prefill_set_attributes();
        if (st == ATTN_OK) st = prefill_pair_set_attributes();
        if (st == ATTN_OK) st = bwd_set_attributes();
        g_attr_status[dev] = st;
    });
    return g_attr_status[dev];
}

// Streaming multiprocessors of the current device (cached per device).
std::atomic<int> g_num_sms[kMaxDevices];

}  // namespace

namespace gbattn {

int current_sm_count(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_num_sms[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *out = cached;
            return ATTN_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return ATTN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) g_num_sms[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return ATTN_OK;
}

}  // namespace gbattn

namespace {

// [BH, N, d] bf16 viewed as a 3-D tensor (d innermost), boxes of 64 x rows x 1
// (rows 128, or 64 for the half key tiles of the CTA-pair prefill) with the
// 128-byte swizzle the tcgen05 operand descriptors expect.
int encode_bhnd(CUtensorMap* m, const void* base, long long BH, int N, int d, unsigned rows = 128) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// O [BH, Nq, d] bf16 as a 3-D tensor {d, Nq, BH} in boxes of 32 x 32 x 1 with
// the 64-byte swizzle: the target of the prefill epilogue's TMA stores (a warp
// stores 32 rows x 32 columns at a time; rows past Nq are clipped).
int encode_o_store(CUtensorMap* m, void* base, long long BH, int N, int d) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// The fp32 dQ accumulator [BH, Nq_pad, d] of the backward as a 3-D tensor
// {d, Nq_pad, BH} in boxes of 32 x 128 x 1 with the 128-byte swizzle (the
// target of the backward's TMA reduce-adds).
int encode_dq_acc(CUtensorMap* m, void* base, long long BH, int nq_pad, int d) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(nq_pad),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                             static_cast<cuuint64_t>(nq_pad) * static_cast<cuuint64_t>(d) * 4};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// cta_pair: the products as CTA-pair (cta_group::2) products (bf16, d = 128,
// no per-sequence lengths); otherwise the single-CTA kernel.
int enqueue_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int d, int causal, float scale, cudaStream_t stream,
                const int* seqlens_q = nullptr, const int* seqlens_k = nullptr,
                bool cta_pair = false) {
    int st = ensure_init();
    if (st != ATTN_OK) return st;
    int num_sms = 0;
    if ((st = current_sm_count(&num_sms)) != ATTN_OK) return st;
    const long long BH = static_cast<long long>(B) * H;
    CUtensorMap tq, tk, tv, to;
    if ((st = encode_bhnd(&tq, q, BH, Nq, d)) != ATTN_OK) return st;
    if ((st = encode_bhnd(&tk, k, BH, Nk, d)) != ATTN_OK) return st;
    if ((st = encode_bhnd(&tv, v, BH, Nk, d)) != ATTN_OK) return st;
    if ((st = encode_o_store(&to, o, BH, Nq, d)) != ATTN_OK) return st;
    PrefillParams p;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.Nq = Nq;
    p.Nk = Nk;
    p.BH = static_cast<int>(BH);
    p.num_pairs = (Nq + 255) / 256;
    p.causal = causal;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.H = H;
    p.seqlens_q = seqlens_q;
    p.seqlens_k = seqlens_k;
    p.o_scale = 1.f;
    if (cta_pair) {
        // quads of four query tiles per item, K in half tiles of 64 keys
        CUtensorMap tk64;
        if ((st = encode_bhnd(&tk64, k, BH, Nk, d, 64)) != ATTN_OK) return st;
        p.num_pairs = (Nq + 511) / 512;
        return launch_prefill_pair(tq, tk64, tv, to, p, stream);
    }
    return launch_prefill(d, tq, tk, tv, to, p, num_sms, stream);
}

// A 3-D byte tensor {x, y, BH} (x innermost, x bytes per row, y rows per
// (b, h)) in boxes of 128 x 128 x 1 with the 128-byte swizzle: E4M3 Q and K
// ({d, N, BH}) and the transposed values ({Nk, d, BH}).
int encode_u8(CUtensorMap* m, const void* base, long long BH, int x, int y) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(x), static_cast<cuuint64_t>(y),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(x),
                             static_cast<cuuint64_t>(x) * static_cast<cuuint64_t>(y)};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Heads per group of the backward's CTA order: as many as keep their Q and dO
// rows (bf16) and fp32 dQ accumulator rows within a quarter of the L2 cache.
int bwd_head_group(long long BH, int Nq, int d, int* out) {
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const long long per_head = (static_cast<long long>(Nq) + 127) / 128 * 128 * d * (2 + 2 + 4);
    long long g = (static_cast<long long>(l2) / 4) / per_head;
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    *out = static_cast<int>(g);
    return ATTN_OK;
}

int enqueue_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                int d, int causal, float scale, void* workspace, cudaStream_t stream) {
    int st = ensure_init();
    if (st != ATTN_OK) return st;
    int num_sms = 0;
    if ((st = current_sm_count(&num_sms)) != ATTN_OK) return st;
    const long long BH = static_cast<long long>(B) * H;
    CUtensorMap tq, tk, tv, tdo;
    if ((st = encode_bhnd(&tq, q, BH, Nq, d)) != ATTN_OK) return st;
    if ((st = encode_bhnd(&tk, k, BH, Nk, d)) != ATTN_OK) return st;
    if ((st = encode_bhnd(&tv, v, BH, Nk, d)) != ATTN_OK) return st;
    if ((st = encode_bhnd(&tdo, dout, BH, Nq, d)) != ATTN_OK) return st;
    const int nq_pad = (Nq + 127) / 128 * 128;
    float* ws = static_cast<float*>(workspace);
    CUtensorMap tdqacc;
    if ((st = encode_dq_acc(&tdqacc, ws, BH, nq_pad, d)) != ATTN_OK) return st;
    BwdPrepParams a;
    a.o = static_cast<const __nv_bfloat16*>(o);
    a.dout = static_cast<const __nv_bfloat16*>(dout);
    a.lse = lse;
    a.dq_acc = ws;
    a.nl2 = ws + BH * nq_pad * d;
    a.nD = a.nl2 + BH * nq_pad;
    a.rows = BH * nq_pad;
    a.Nq = Nq;
    a.Nq_pad = nq_pad;
    BwdParams p;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.dq_acc = a.dq_acc;
    p.nl2 = a.nl2;
    p.nD = a.nD;
    p.Nq = Nq;
    p.Nk = Nk;
    p.Nq_pad = nq_pad;
    p.BH = static_cast<int>(BH);
    p.n_kt = (Nk + 127) / 128;
    if ((st = bwd_head_group(BH, Nq, d, &p.head_group)) != ATTN_OK) return st;
    p.causal = causal;
    p.causal_off = causal ? Nk - Nq : 0;
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    return launch_backward(d, tq, tk, tv, tdo, tdqacc, a, p, static_cast<__nv_bfloat16*>(dq),
                           num_sms, stream);
}

// Streams and events of the host-buffer path, created on first use per device
// and kept until the process exits.  The mutex serialises the enqueue of
// calls from several host threads (the events are shared).
constexpr int kHostChunks = 5;
struct HostPipe {
    bool ready = false;
    cudaStream_t compute = nullptr, copy_out = nullptr;
    cudaEvent_t start = nullptr, out_done = nullptr;
    cudaEvent_t in_done[kHostChunks] = {}, fwd_done[kHostChunks] = {};
};
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mu;

int host_pipe(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    HostPipe& hp = g_pipes[dev];
    if (!hp.ready) {
        const unsigned ev = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&hp.compute, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp.copy_out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.start, ev) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.out_done, ev) == cudaSuccess;
        for (int c = 0; c < kHostChunks && ok; ++c)
            ok = cudaEventCreateWithFlags(&hp.in_done[c], ev) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.fwd_done[c], ev) == cudaSuccess;
        if (!ok) return ATTN_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Nq, int Nk, int d, int causal, float scale, void* stream) {
    int st = validate_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale);
    if (st != ATTN_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    return enqueue_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale,
                       static_cast<cudaStream_t>(stream));
}

int attn_fwd_cta_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, int causal, float scale, void* stream) {
    int st = validate_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale);
    if (st != ATTN_OK) return st;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    return enqueue_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale,
                       static_cast<cudaStream_t>(stream), nullptr, nullptr, true);
}

size_t attn_fwd_decode_workspace_bytes(int B, int H, int Nk, int d) {
    if (B <= 0 || H <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
    return decode_workspace_bytes(static_cast<long long>(B) * H, Nk, d);
}

}  // extern "C"

namespace {

// k_scale / v_scale non-null: k and v are MXFP8 codes with these block scales.
int decode_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nk, int d, float scale, void* workspace, size_t workspace_bytes,
                const int* seqlens_k, void* stream, const void* k_scale = nullptr,
                const void* v_scale = nullptr) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nk <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    // the workspace bound covers every device's plan; it is checked before any CUDA call
    const size_t need = decode_workspace_bytes(BH, Nk, d);
    if (BH * kDecodeMaxSplits > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        (need > 0 && !aligned16(workspace)))
        return ATTN_ERR_MISALIGNED;
    int num_sms = 0;
    const int sst = current_sm_count(&num_sms);
    if (sst != ATTN_OK) return sst;
    int splits, kps;
    decode_split_plan(BH, Nk, num_sms, &splits, &kps);
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.part_o = static_cast<float*>(workspace);
    p.part_lse = splits > 1 ? static_cast<float*>(workspace) + BH * splits * d : nullptr;
    p.BH = static_cast<int>(BH);
    p.Nk = Nk;
    p.splits = splits;
    p.keys_per_split = kps;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.H = H;
    p.seqlens_k = seqlens_k;
    p.k_scale = static_cast<const uint8_t*>(k_scale);
    p.v_scale = static_cast<const uint8_t*>(v_scale);
    if (k_scale) return launch_decode_mx(d, p, static_cast<cudaStream_t>(stream));
    return launch_decode(d, p, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int attn_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int Nk, int d, float scale, void* workspace, size_t workspace_bytes,
                    void* stream) {
    return decode_impl(q, k, v, o, lse, B, H, Nk, d, scale, workspace, workspace_bytes, nullptr,
                       stream);
}

int attn_fwd_decode_mx(const void* q, const void* k8, const void* k_scale, const void* v8,
                       const void* v_scale, void* o, float* lse, int B, int H, int Nk, int d,
                       float scale, void* workspace, size_t workspace_bytes, void* stream) {
    if (!k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
    return decode_impl(q, k8, v8, o, lse, B, H, Nk, d, scale, workspace, workspace_bytes,
                       nullptr, stream, k_scale, v_scale);
}

int attn_fwd_decode_ragged(const void* q, const void* k, const void* v, void* o, float* lse,
                           const int* seqlens_k, int B, int H, int Nk, int d, float scale,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (seqlens_k && (reinterpret_cast<uintptr_t>(seqlens_k) & 3u)) return ATTN_ERR_MISALIGNED;
    return decode_impl(q, k, v, o, lse, B, H, Nk, d, scale, workspace, workspace_bytes,
                       seqlens_k, stream);
}

int attn_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B,
                 int H, int Nq, int Nk, int d, int causal, float scale, float descale_q,
                 float descale_k, float descale_v, void* stream) {
    int st = validate_fwd(q, k, vt, o, lse, B, H, Nq, Nk, d, causal, scale);
    if (st != ATTN_OK) return st;
    for (float ds : {descale_q, descale_k, descale_v})
        if (!(std::isfinite(ds) && ds > 0.f)) return ATTN_ERR_INVALID_ARG;
    const double c = static_cast<double>(scale) * descale_q * descale_k;
    if (!(c < 3.0e38)) return ATTN_ERR_INVALID_ARG;  // the folded score scale stays finite
    if (d != 128) return ATTN_ERR_UNSUPPORTED;   // one 128-byte atom per row
    if (Nk % 16 != 0) return ATTN_ERR_UNSUPPORTED;  // V^T rows: a multiple of 16 bytes
    if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    if ((st = ensure_init()) != ATTN_OK) return st;
    int num_sms = 0;
    if ((st = current_sm_count(&num_sms)) != ATTN_OK) return st;
    const long long BH = static_cast<long long>(B) * H;
    CUtensorMap tq, tk, tvt, to;
    if ((st = encode_u8(&tq, q, BH, d, Nq)) != ATTN_OK) return st;
    if ((st = encode_u8(&tk, k, BH, d, Nk)) != ATTN_OK) return st;
    if ((st = encode_u8(&tvt, vt, BH, Nk, d)) != ATTN_OK) return st;
    if ((st = encode_o_store(&to, o, BH, Nq, d)) != ATTN_OK) return st;
    PrefillParams p;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.Nq = Nq;
    p.Nk = Nk;
    p.BH = static_cast<int>(BH);
    p.num_pairs = (Nq + 255) / 256;
    p.causal = causal;
    p.scale_log2 = static_cast<float>(c * 1.4426950408889634074);
    p.H = H;
    p.seqlens_q = nullptr;
    p.seqlens_k = nullptr;
    p.o_scale = descale_v;
    return launch_prefill_fp8(tq, tk, tvt, to, p, num_sms, static_cast<cudaStream_t>(stream));
}

int attn_fwd_ragged(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk,
                    int d, int causal, float scale, void* stream) {
    int st = validate_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale);
    if (st != ATTN_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
        return ATTN_ERR_MISALIGNED;
    return enqueue_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale,
                       static_cast<cudaStream_t>(stream), seqlens_q, seqlens_k);
}

int attn_fwd_from_host(const void* q, const void* k, const void* v, void* o, float* lse,
                       void* dq, void* dk, void* dv, void* do_, float* dlse, int B, int H,
                       int Nq, int Nk, int d, int causal, float scale, void* stream) {
    int st = validate_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale);
    if (st != ATTN_OK) return st;
    if (!dq || !dk || !dv || !do_ || !dlse) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(do_) || !aligned16(dlse))
        return ATTN_ERR_MISALIGNED;
    // The (b, h) heads go in up to kHostChunks contiguous chunks.  Chunk c:
    // host->device copies on the caller's stream, the prefill kernel on the
    // compute stream once they have landed, device->host copies on the
    // copy-out stream once it has run -- so the inputs of chunk c + 1 cross
    // the host link while chunk c computes and chunk c - 1's results come back
    // the other way.  The caller's stream finally waits for the last copy out.
    // Chunk sizes fall off in the ratio 5 : 4 : 3 : 2 : 1: the host link is
    // the bottleneck and only the last chunk's kernel and copy out are left
    // exposed after the inputs have crossed, so the last chunk is the smallest.
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long BH = static_cast<long long>(B) * H;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* hp = nullptr;
    if ((st = host_pipe(&hp)) != ATTN_OK) return st;
    const int chunks = static_cast<int>(BH < kHostChunks ? BH : kHostChunks);
    if (cudaEventRecord(hp->start, s) != cudaSuccess ||
        cudaStreamWaitEvent(hp->compute, hp->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->copy_out, hp->start, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const size_t qh = static_cast<size_t>(Nq) * d * 2, kh = static_cast<size_t>(Nk) * d * 2;
    const size_t lh = static_cast<size_t>(Nq) * 4;
    auto at = [](const void* base, size_t off) { return static_cast<const char*>(base) + off; };
    auto atw = [](void* base, size_t off) { return static_cast<char*>(base) + off; };
    // chunk c ends near head BH * W(c) / W(chunks), W(c) = the sum of the first
    // c + 1 weights chunks, chunks - 1, ..., 1, clamped so that every chunk has
    // at least one head
    const long long wsum = static_cast<long long>(chunks) * (chunks + 1) / 2;
    long long h0 = 0, wacc = 0;
    for (int c = 0; c < chunks; ++c) {
        wacc += chunks - c;
        long long h1 = BH * wacc / wsum;
        if (h1 < h0 + 1) h1 = h0 + 1;
        if (h1 > BH - (chunks - 1 - c)) h1 = BH - (chunks - 1 - c);
        const size_t n = static_cast<size_t>(h1 - h0);
        const size_t oq = static_cast<size_t>(h0) * qh, ok = static_cast<size_t>(h0) * kh;
        const size_t ol = static_cast<size_t>(h0) * lh;
        if (cudaMemcpyAsync(atw(dq, oq), at(q, oq), n * qh, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaMemcpyAsync(atw(dk, ok), at(k, ok), n * kh, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaMemcpyAsync(atw(dv, ok), at(v, ok), n * kh, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaEventRecord(hp->in_done[c], s) != cudaSuccess ||
            cudaStreamWaitEvent(hp->compute, hp->in_done[c], 0) != cudaSuccess)
            return ATTN_ERR_CUDA;
        // the chunk as a batch of n heads (B = 1, H = n): the same per-head problem
        st = enqueue_fwd(atw(dq, oq), atw(dk, ok), atw(dv, ok), atw(do_, oq),
                         reinterpret_cast<float*>(atw(dlse, ol)), 1, static_cast<int>(n), Nq, Nk,
                         d, causal, scale, hp->compute);
        if (st != ATTN_OK) return st;
        if (cudaEventRecord(hp->fwd_done[c], hp->compute) != cudaSuccess ||
            cudaStreamWaitEvent(hp->copy_out, hp->fwd_done[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(atw(o, oq), atw(do_, oq), n * qh, cudaMemcpyDeviceToHost,
                            hp->copy_out) != cudaSuccess ||
            cudaMemcpyAsync(atw(lse, ol), atw(dlse, ol), n * lh, cudaMemcpyDeviceToHost,
                            hp->copy_out) != cudaSuccess)
            return ATTN_ERR_CUDA;
        h0 = h1;
    }
    if (cudaEventRecord(hp->out_done, hp->copy_out) != cudaSuccess ||
        cudaStreamWaitEvent(s, hp->out_done, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

int attn_merge(const void* o_parts, const float* lse_parts, int n_parts, void* o, float* lse,
               int B, int H, int Nq, int d, void* stream) {
    if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (n_parts <= 0 || B <= 0 || H <= 0 || Nq <= 0) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * H * Nq;
    if (rows > (1LL << 40) / n_parts) return ATTN_ERR_UNSUPPORTED;  // index range
    if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    int num_sms = 0;
    const int st = current_sm_count(&num_sms);
    if (st != ATTN_OK) return st;
    MergeParams p;
    p.o_parts = static_cast<const __nv_bfloat16*>(o_parts);
    p.lse_parts = lse_parts;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.rows = rows;
    p.n_parts = n_parts;
    return launch_merge(d, p, num_sms, static_cast<cudaStream_t>(stream));
}

size_t attn_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
    return bwd_workspace_bytes(static_cast<long long>(B) * H, Nq, d);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
             int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
    int st = validate_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale);
    if (st != ATTN_OK) return st;
    if (!dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * ((static_cast<long long>(Nk) + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < bwd_workspace_bytes(BH, Nq, d)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(workspace))
        return ATTN_ERR_MISALIGNED;
    return enqueue_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, causal, scale,
                       workspace, static_cast<cudaStream_t>(stream));
}

const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported configuration";
        case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED: pointer not 16-byte aligned";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA call failed";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: kernel abandoned a barrier wait";
        case ATTN_ERR_OUT_OF_RANGE:
            return "ATTN_ERR_OUT_OF_RANGE: debug build skipped an access outside its buffer";
        default: return "unknown status";
    }
}

int attn_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    const unsigned e = read_and_clear_prefill_error() | read_and_clear_prefill_pair_error() |
                       read_and_clear_bwd_error() |
                       read_and_clear_decode_error() | read_and_clear_selftest_error() |
                       read_and_clear_merge_error();
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (e & kErrBitTimeout) return ATTN_ERR_TIMEOUT;
    if (e & kErrBitBounds) return ATTN_ERR_OUT_OF_RANGE;
    return e ? ATTN_ERR_INVALID_ARG : ATTN_OK;
}

int attn_version(void) { return kVersion; }

int attn_selftest_timeout(void* stream) {
    return launch_selftest_timeout(static_cast<cudaStream_t>(stream));
}

int attn_selftest_bounds(void* stream) {
    return launch_selftest_bounds(static_cast<cudaStream_t>(stream));
}

int attn_pair_product(const void* a, const void* b, float* d, void* stream) {
    if (!a || !b || !d) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return ATTN_ERR_MISALIGNED;
    return launch_pair_product(a, b, d, static_cast<cudaStream_t>(stream));
}

int attn_bench_mma_rate(int form, int issuer, int busy, int waits, int steps, int reps,
                        float* ms_out, double* cycles_out, int* sms_out, void* stream) {
    if ((form != 1 && form != 2) || (issuer != 0 && issuer != 1) || (busy != 0 && busy != 1) ||
        (waits != 0 && waits != 1) || steps < 1 || steps > (1 << 16) || reps < 1 || reps > 1000 ||
        !ms_out)
        return ATTN_ERR_INVALID_ARG;
    return run_mma_rate(form, issuer, busy, waits, steps, reps, ms_out, cycles_out, sms_out,
                        static_cast<cudaStream_t>(stream));
}

int attn_debug_build(void) {
#ifdef GBATTN_DEBUG
    return 1;
#else
    return 0;
#endif
}

}  // extern "C"
