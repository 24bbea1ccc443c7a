// decode_no_alloc_sm103.cu -- single-query attention forward for callers
// that cannot allocate device memory.
//
// attn_fwd_decode needs a workspace for the per-split partial results, and the
// caller has to provide it.  Some callers cannot: a plugin inside a host
// application (an inference engine, a game or media pipeline) whose device
// memory is owned and budgeted by that application, or a latency-critical
// serving loop where cudaMalloc/cudaFree are off limits because they can
// synchronise the whole device.  attn_fwd_decode_no_alloc serves them: its
// scratch is a fixed array in the library's own device memory, so the call
// allocates nothing itself.
//
// The array is file-scope, so host code cannot use its name as a device
// address; the address is looked up once per device with
// cudaGetSymbolAddress (on the first call made while that device is current)
// and handed to the same split and combine kernels attn_fwd_decode uses.
// CUDA loads a library's device code lazily, on first use per device, so it
// is that first call's lookup that loads this file's module and reserves the
// array on the device (and may synchronise it): make the first call during
// set-up, outside any serving loop or stream capture.  The cached address
// belongs to the device's primary context; after cudaDeviceReset the module
// is reloaded elsewhere and the cached address is stale, so this call (like
// the rest of the library, whose per-device state is cached the same way)
// must not be used after a reset in the same process.
#include <mutex>

#include "gbattn_internal.h"

namespace {

constexpr size_t kScratchBytes = ATTN_DECODE_NO_ALLOC_SCRATCH_BYTES;

// Partial outputs and logsumexps of the splits.  Every device that loads the
// library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_lock;
void* g_scratch_addr[gbattn::kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= gbattn::kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_lock);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return ATTN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int attn_fwd_decode_no_alloc(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int B, int H, int Nk, int d, float scale,
                                        void* stream) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nk <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f && scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * gbattn::kDecodeMaxSplits > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    // more partial results than the fixed scratch holds (the workspace
    // attn_fwd_decode would ask for, which bounds every device's plan): use
    // attn_fwd_decode with a workspace of the caller's
    if (gbattn::decode_workspace_bytes(BH, Nk, d) > kScratchBytes) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    int num_sms = 0;
    int st = gbattn::current_sm_count(&num_sms);
    if (st != ATTN_OK) return st;
    int splits, kps;
    gbattn::decode_split_plan(BH, Nk, num_sms, &splits, &kps);
    void* scratch = nullptr;
    if (splits > 1 && (st = scratch_address(&scratch)) != ATTN_OK) return st;
    // Nothing in the scratch has to start at zero: every partial the combine
    // kernel reads is written by the split kernel of the same call.
    gbattn::DecodeParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.part_o = static_cast<float*>(scratch);
    p.part_lse = splits > 1 ? static_cast<float*>(scratch) + BH * splits * d : nullptr;
    p.BH = static_cast<int>(BH);
    p.Nk = Nk;
    p.splits = splits;
    p.keys_per_split = kps;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.H = H;
    p.seqlens_k = nullptr;  // every sequence has all Nk keys
    p.k_scale = nullptr;    // bf16 keys and values
    p.v_scale = nullptr;
    return gbattn::launch_decode(d, p, static_cast<cudaStream_t>(stream));
}
