/*
 * gbattn.h -- C ABI of the fused attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation (from the lecture pages this library follows):
 *   O = softmax(scale * Q K^T [+ causal mask]) V,   lse_i = log sum_j e^{scale q_i . k_j}
 * "Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V" (PDC course Lecture 4,
 * section 4.14; CS336 Lecture 5 notes, section 8.1), evaluated block by block
 * with the online softmax and the logsumexp L_i = m_i + log l_i kept per row
 * (CS336 Lecture 5 notes, section 8.3).  The score matrix never reaches HBM.
 *
 * Conventions shared by every entry point:
 *   - Tensors are contiguous, row-major, head dimension innermost:
 *       q  bf16 [B, H, Nq, d]      k, v  bf16 [B, H, Nk, d]
 *       o  bf16 [B, H, Nq, d]      lse   fp32 [B, H, Nq]  (natural log)
 *     "bf16" is IEEE bfloat16 (1-8-7) stored in 2 bytes.
 *   - Device pointers must be 16-byte aligned.  The caller owns every buffer;
 *     the attention calls allocate nothing (attn_bench_mma_rate, a measurement
 *     of the product forms, allocates its own result buffer).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  The attention
 *     calls are asynchronous: ATTN_OK means "enqueued" (attn_pair_product and
 *     attn_bench_mma_rate synchronise before returning).  Faults inside a kernel
 *     surface at the caller's next synchronisation, as in CUDA.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and touches no buffer.
 *   - Nothing is thrown across the ABI; every call returns a status code.
 *   - Thread safety: calls may be made from several host threads, and on
 *     several devices (each call runs on the current device).  The shared host
 *     state is the driver's tensor-map encoder (looked up once), kernel
 *     attributes and an SM count set once per device, and the streams and
 *     events attn_fwd_from_host creates per device on first use (its enqueue
 *     is serialised by a mutex).
 *   - Contexts: that per-device state is cached by device ordinal for the
 *     life of the process and belongs to the device's primary context (the
 *     one the CUDA runtime uses).  After cudaDeviceReset it is stale: do not
 *     call the library again in that process.
 *   - CUDA graphs: after one call on a device (which creates that state),
 *     every call can be captured in a CUDA graph and replayed.  Calls enqueue
 *     only kernel launches; attn_fwd_from_host also enqueues copies (capture
 *     needs pinned host buffers) and event waits that fork its own streams
 *     from the caller's stream and join them back before it returns.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, non-finite or
                                  non-positive scale, too-small workspace */
    ATTN_ERR_UNSUPPORTED = 2,  /* d not in {64, 128}; causal with Nq > Nk;
                                  sizes beyond the index range of the kernels */
    ATTN_ERR_MISALIGNED = 3,   /* a device pointer is not 16-byte aligned */
    ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    ATTN_ERR_TIMEOUT = 5,      /* a kernel gave up waiting on one of its own
                                  pipeline barriers (reported by
                                  attn_device_error, never by a launch) */
    ATTN_ERR_OUT_OF_RANGE = 6  /* debug builds only: a kernel found an index
                                  outside its buffer and skipped the access (a
                                  library bug; reported by attn_device_error) */
} attn_status_t;

/*
 * attn_fwd -- prefill / full attention forward.
 *
 * Computes, for every (b, h) and query row i < Nq:
 *   s_ij   = scale * sum_c q[b,h,i,c] k[b,h,j,c]            for j < Nk
 *   s_ij   = -inf if causal and j > i + (Nk - Nq)          (key j in the future of query i)
 *   o[b,h,i,:] = sum_j softmax_j(s_i.) v[b,h,j,:]          (bf16, round-to-nearest-even)
 *   lse[b,h,i] = log sum_j e^{s_ij}                          (fp32, natural log)
 * FlashAttention forward with the online softmax (CS336 Lecture 5 notes,
 * sections 8.2-8.3; CS149 Lecture 9 notes, concept 9); causal key blocks
 * wholly in the future of a query block are skipped.
 * Causal with Nq < Nk: the queries are the newest Nq tokens of a sequence of
 * Nk tokens whose keys and values are all given (chunked prefill against a
 * KV cache, the cache that grows during inference of the PDC course
 * Lecture 4, section 4.9), so query i sits at position i + (Nk - Nq).  With
 * Nq == Nk this is the usual j > i mask; Nq > Nk would leave rows with no
 * visible key and is rejected.
 *
 *   q, k, v  device, bf16, layouts above; read only.
 *   o        device, bf16 [B,H,Nq,d]; written.
 *   lse      device, fp32 [B,H,Nq]; written.  May not be NULL.
 *   B, H, Nq, Nk >= 1;  d in {64, 128};  causal in {0, 1} (causal needs Nq <= Nk).
 *   scale    > 0 and finite; the usual value is 1/sqrt(d).
 *   stream   cudaStream_t.
 * Internal arithmetic: fp32 scores and accumulators on the tensor cores,
 * probabilities rounded to bf16 before the P V product, fp32 row sums.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 * ATTN_ERR_MISALIGNED or ATTN_ERR_CUDA.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int Nq, int Nk, int d, int causal, float scale, void *stream);

/*
 * attn_fwd_fp8 -- attn_fwd on FP8 (E4M3) operands with one descale per tensor.
 *
 * Blackwell's tensor cores run 8-bit products at twice the bf16 rate, with
 * per-tensor (or finer) scaling (PDC course Lecture 7, section 7.14; E4M3 in
 * CS336 Lecture 5 notes, section 6.2).  With Q = descale_q * q, K = descale_k
 * * k and V = descale_v * v (q, k, v the E4M3 values), computes exactly what
 * attn_fwd computes on Q, K, V:
 *   s_ij = scale * sum_c Q[b,h,i,c] K[b,h,j,c], the same causal rule,
 *   o = softmax(s) V (bf16), lse = log sum_j e^{s_ij} (fp32, natural log).
 *
 *   q        device, E4M3 codes (one byte each) [B,H,Nq,d]; read only.
 *   k        device, E4M3 [B,H,Nk,d]; read only.
 *   vt       device, E4M3, the values TRANSPOSED: [B,H,d,Nk] (keys innermost).
 *            Both operands of an 8-bit tensor-core product are read with the
 *            reduction dimension innermost, and for O += P V that is the key.
 *   o        device, bf16 [B,H,Nq,d]; written.
 *   lse      device, fp32 [B,H,Nq]; written.
 *   B, H, Nq, Nk >= 1;  d = 128;  Nk a multiple of 16 (rows of vt are TMA
 *            rows and must span a multiple of 16 bytes); causal as attn_fwd.
 *   scale, descale_q, descale_k, descale_v  > 0 and finite, with
 *            scale * descale_q * descale_k finite in fp32.
 * Internal arithmetic: exact E4M3 products accumulated in fp32, the query and
 * key descales folded into the fp32 score scale, probabilities rounded to E4M3
 * before the P V product (row sums from the unrounded fp32 values), descale_v
 * applied with 1 / l in the epilogue.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED (d != 128,
 * Nk % 16 != 0, causal with Nq > Nk), ATTN_ERR_MISALIGNED or ATTN_ERR_CUDA.
 */
int attn_fwd_fp8(const void *q, const void *k, const void *vt, void *o, float *lse,
                 int B, int H, int Nq, int Nk, int d, int causal, float scale,
                 float descale_q, float descale_k, float descale_v, void *stream);

/*
 * attn_fwd_cta_pair -- attn_fwd with every tensor-core product issued as a
 * CTA-pair product (tcgen05.mma.cta_group::2, PDC course Lecture 7, section
 * 7.13: two CTAs of a cluster on two SMs share each product, M = 256, each
 * holding half of every key and value tile).  Same arguments, layouts,
 * ownership and result as attn_fwd; the products are the same and accumulate
 * in the same order, so the output is bit-identical to attn_fwd's.
 *   d = 128 only.
 * Measured on GB300 it is slower than attn_fwd (about 0.72x at 4096 tokens):
 * every key-tile step waits for the second SM's softmax to signal across the
 * pair.  attn_fwd keeps the single-CTA products.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED (d != 128, or as
 * attn_fwd), ATTN_ERR_MISALIGNED or ATTN_ERR_CUDA.
 */
int attn_fwd_cta_pair(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int H, int Nq, int Nk, int d, int causal, float scale,
                      void *stream);

/*
 * attn_fwd_decode_workspace_bytes -- bytes of device workspace attn_fwd_decode
 * needs for these sizes: room for the split partials of the largest split
 * plan any device takes (at most one split per 512 keys and 64 splits per
 * (b, h); the plan itself follows the device's SM count), so a workspace
 * sized once fits every GPU.  0 when Nk <= 512 (one split).  Pure host
 * arithmetic; never touches the GPU.  Returns 0 for invalid sizes as well.
 */
size_t attn_fwd_decode_workspace_bytes(int B, int H, int Nk, int d);

/*
 * attn_fwd_decode -- single-query (Nq = 1) attention forward, split over keys.
 *
 * Same result as attn_fwd with Nq = 1, causal = 0.  Decode is memory-bound
 * (CS336 Lecture 5 notes, section 5.3: arithmetic intensity about 1 FLOP per
 * byte), so the keys of each (b, h) are cut into splits that stream K and V
 * once with 16-byte coalesced loads; each split keeps its own running max and
 * sum and writes a partial (o_s, lse_s) to the workspace; a second kernel
 * merges the splits with the two-block rule m = max(m1, m2),
 * l = e^{m1-m} l1 + e^{m2-m} l2 (CS149 Lecture 9 notes, concept 9).
 *
 *   q        device bf16 [B,H,1,d];  k, v device bf16 [B,H,Nk,d].
 *   o        device bf16 [B,H,1,d];  lse device fp32 [B,H,1].
 *   workspace  device scratch of at least attn_fwd_decode_workspace_bytes()
 *              bytes, 16-byte aligned (NULL allowed when that is 0).  Its
 *              contents on entry do not matter; it is overwritten.  Two calls
 *              in flight at once must not share a workspace.
 * Returns as attn_fwd; a too-small workspace is ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int H, int Nk, int d, float scale,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_fwd_decode_mx -- attn_fwd_decode with MXFP8 keys and values.
 *
 * The microscaling (MX) formats give every block of 32 consecutive elements
 * its own power-of-two scale (the fine-grained quantisation of PDC course
 * Lecture 7, section 7.14; the bits follow the OCP Microscaling Formats v1.0
 * specification): an element's value is 2^(X - 127) * E4M3(code), X the E8M0
 * code of its block (0xFF is NaN).  Decode reads every key and value once, so
 * storing the KV cache this way halves the bytes it streams.  Computes what
 * attn_fwd_decode computes on the dequantised keys and values:
 *   s_j = scale * q . K_j,  o = softmax(s) V (bf16),  lse = log sum_j e^{s_j}.
 *
 *   q        device bf16 [B,H,1,d].
 *   k8, v8   device, E4M3 codes (one byte each) [B,H,Nk,d]; read only.
 *   k_scale, v_scale  device, E8M0 codes [B,H,Nk,d/32]: the scale of elements
 *            32 b .. 32 b + 31 of a key's (value's) row is its entry b; read only.
 *   o, lse, workspace, stream, B, H, Nk, scale  as attn_fwd_decode (the same
 *            workspace size: attn_fwd_decode_workspace_bytes(B, H, Nk, d)).
 *   d in {64, 128}.  q, k8, v8, o, lse and the workspace 16-byte aligned.
 * Internal arithmetic: codes widened exactly to fp32, fp32 dot products and
 * accumulators, scales applied per block (exact powers of two).
 * Returns as attn_fwd_decode; a NULL scale pointer is ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_decode_mx(const void *q, const void *k8, const void *k_scale, const void *v8,
                       const void *v_scale, void *o, float *lse, int B, int H, int Nk, int d,
                       float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_fwd_from_host -- attn_fwd on HOST buffers, end to end.
 *
 * Host->device copies of q, k, v into the caller's device buffers dq, dk,
 * dv; attn_fwd on them into do_, dlse; device->host copies of the results
 * into o and lse.  The (b, h) heads go in up to five chunks, each smaller
 * than the one before, so that one chunk's inputs cross the host link while
 * the previous chunk computes and the one before returns its results (the
 * last, smallest chunk's kernel and output copy are all that remain after
 * the inputs have crossed): the input copies run on `stream`, the
 * kernels and the output copies on two streams of the library's own
 * (created with a few events on the first call on each device, kept until
 * the process exits), and `stream` is made to wait for the last output copy.
 * So, as for every call here, the caller synchronises `stream` before
 * reading o and lse.  The host buffers should be pinned (page-locked) for
 * the copies to be asynchronous.  Same arguments, sizes and status codes as
 * attn_fwd; every pointer must be non-NULL and the device ones 16-byte
 * aligned.
 */
int attn_fwd_from_host(const void *q, const void *k, const void *v, void *o, float *lse,
                       void *dq, void *dk, void *dv, void *do_, float *dlse,
                       int B, int H, int Nq, int Nk, int d, int causal, float scale,
                       void *stream);

/*
 * attn_fwd_decode_no_alloc -- attn_fwd_decode for callers that cannot
 * allocate device memory.  The lecture pages have no counterpart of this
 * call; it exists for users of this library.
 *
 * attn_fwd_decode needs the caller to provide a workspace.  Some callers
 * cannot call cudaMalloc: a plugin inside a host application that owns and
 * budgets all device memory, or a latency-critical serving loop in which
 * cudaMalloc/cudaFree are not allowed because they can synchronise the whole
 * device.  This call computes the same result as attn_fwd_decode but keeps
 * the split partials in a fixed scratch array of
 * ATTN_DECODE_NO_ALLOC_SCRATCH_BYTES that lives in the library's own device
 * memory (every GPU that loads the library holds it until the process exits).
 * The call allocates nothing; the caller still passes q, k, v, o and lse.
 *
 *   Arguments and layouts as attn_fwd_decode, without the workspace.
 *   Sizes whose partials need more than ATTN_DECODE_NO_ALLOC_SCRATCH_BYTES
 *   (i.e. attn_fwd_decode_workspace_bytes(B, H, Nk, d) is larger) are
 *   rejected with ATTN_ERR_UNSUPPORTED before anything is launched; use
 *   attn_fwd_decode with your own workspace for them.
 *   The first call on each device looks up the scratch array's device
 *   address (cudaGetSymbolAddress) with that device current.  CUDA loads the
 *   library's device code lazily, so it is this first call that loads the
 *   module holding the array and reserves its memory on that device (and it
 *   may synchronise the device): make the first call during set-up, outside
 *   the serving loop and before any stream capture.  Later calls allocate
 *   and look up nothing.
 *   All calls share the one array and it keeps the previous call's contents;
 *   nothing in it needs to start at zero.  Calls whose kernels overlap on the
 *   GPU (other streams, other host threads) race on the array: order them on
 *   one stream or wait for one to finish before the next.
 * Returns as attn_fwd_decode.
 */
#define ATTN_DECODE_NO_ALLOC_SCRATCH_BYTES (2u << 20) /* 2 MiB */
int attn_fwd_decode_no_alloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int Nk, int d, float scale, void *stream);

/*
 * attn_fwd_ragged -- attn_fwd on a batch of sequences of different lengths.
 *
 * The KV cache grows per request during inference (PDC course Lecture 4,
 * section 4.9), so a serving batch holds sequences of different lengths.
 * The tensors keep the padded layout of attn_fwd ([B,H,Nq,d], [B,H,Nk,d]);
 * sequence b has seqlens_q[b] queries and seqlens_k[b] keys, the first
 * ones of its rows.  For every b, h and i < seqlens_q[b]:
 *   s_ij = scale q_i . k_j  for j < seqlens_k[b]  (later keys do not exist)
 *   s_ij = -inf if causal and j > i + (seqlens_k[b] - seqlens_q[b])
 *   o, lse as attn_fwd over those keys.
 *
 *   seqlens_q, seqlens_k  device int32 [B], 4-byte aligned, or NULL (every
 *               sequence has Nq queries / Nk keys).  1 <= seqlens_q[b] <= Nq,
 *               1 <= seqlens_k[b] <= Nk, and seqlens_q[b] <= seqlens_k[b] when
 *               causal.  The values are read on the GPU: a sequence whose
 *               lengths break these bounds is skipped (nothing of it is
 *               written) and attn_device_error reports ATTN_ERR_INVALID_ARG.
 *   o, lse      rows i >= seqlens_q[b] are not written.
 *   k, v        rows j >= seqlens_k[b] get weight 0 but are read in whole
 *               128-key tiles: they must hold finite values (0 * inf is NaN).
 *   Everything else as attn_fwd.
 */
int attn_fwd_ragged(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int *seqlens_q, const int *seqlens_k, int B, int H, int Nq, int Nk,
                    int d, int causal, float scale, void *stream);

/*
 * attn_fwd_decode_ragged -- attn_fwd_decode on a batch whose sequences hold
 * different numbers of keys: sequence b attends to keys j < seqlens_k[b] of
 * the padded [B,H,Nk,d] k and v; later rows are never read.
 *   seqlens_k   device int32 [B], 4-byte aligned, or NULL (all Nk);
 *               1 <= seqlens_k[b] <= Nk, checked on the GPU: a sequence out
 *               of range gets o = 0 and lse = -inf and attn_device_error
 *               reports ATTN_ERR_INVALID_ARG.
 *   Workspace: attn_fwd_decode_workspace_bytes(B, H, Nk, d).  Everything
 *   else as attn_fwd_decode.
 */
int attn_fwd_decode_ragged(const void *q, const void *k, const void *v, void *o, float *lse,
                           const int *seqlens_k, int B, int H, int Nk, int d, float scale,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_merge -- attention over all keys from results over disjoint key sets.
 *
 * For every row (b, h, i), part s holds o_s = attention of query i over the
 * keys of part s and its logsumexp lse_s (e.g. attn_fwd or attn_fwd_decode
 * on one shard of k and v).  The merge is the two-block rule of the CS149
 * Lecture 9 notes, concept 9 (m = max, l = sum of e^{m_s - m} l_s), applied
 * to all parts:
 *   lse = log sum_s e^{lse_s},    o = sum_s e^{lse_s - lse} o_s
 * which is the attention over the union of the parts' keys.  This is the
 * one exchange step of key- (context-) parallel attention: each rank attends
 * to its shard of the keys, the (o_s, lse_s) are gathered, and this call
 * merges them.  A part with lse_s = -inf (no visible key) has weight 0; a row
 * whose parts are all -inf gets o = 0 and lse = -inf.
 *
 *   o_parts    device, bf16 [n_parts, B, H, Nq, d], contiguous; read only.
 *   lse_parts  device, fp32 [n_parts, B, H, Nq] (natural log); read only.
 *   o          device, bf16 [B, H, Nq, d]; written.
 *   lse        device, fp32 [B, H, Nq]; written.
 *   n_parts, B, H, Nq >= 1;  d in {64, 128};  stream cudaStream_t.
 * Arithmetic in fp32, o rounded to bf16 (round-to-nearest-even).  Memory
 * bound: reads n_parts * (2 d + 4) and writes 2 d + 4 bytes per row.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 * ATTN_ERR_MISALIGNED or ATTN_ERR_CUDA.
 */
int attn_merge(const void *o_parts, const float *lse_parts, int n_parts, void *o, float *lse,
               int B, int H, int Nq, int d, void *stream);

/*
 * attn_bwd_workspace_bytes -- bytes of device workspace attn_bwd needs:
 * an fp32 dQ accumulator plus two fp32 values per query row, over whole
 * 128-row query tiles: B*H*ceil(Nq/128)*128*(d + 2)*4.  Pure host
 * arithmetic; returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/*
 * attn_bwd -- backward pass of attn_fwd: dQ, dK, dV for an upstream
 * gradient dO = dL/dO.
 *
 * The FlashAttention-2 backward of the CS336 Lecture 5 notes, section 8.4:
 * P is not stored but recomputed from the forward's logsumexp,
 * P_ij = e^{s_ij - lse_i}; with D_i = rowsum(dO_i * O_i) (exercise 9 there)
 *   dV_j = sum_i P_ij dO_i,           dP_ij = dO_i . v_j,
 *   dS_ij = P_ij (dP_ij - D_i),       dQ_i = scale sum_j dS_ij k_j,
 *   dK_j = scale sum_i dS_ij q_i,
 * with s and the causal mask exactly as in attn_fwd.
 *
 *   q, k, v     device, bf16, the forward's inputs; read only.
 *   o, lse      device, the forward's outputs for these inputs (bf16
 *               [B,H,Nq,d], fp32 [B,H,Nq]) from attn_fwd; read only.
 *   dout        device, bf16 [B,H,Nq,d], dL/dO; read only.
 *   dq          device, bf16 [B,H,Nq,d]; written.
 *   dk, dv      device, bf16 [B,H,Nk,d]; written.
 *   B .. scale  as attn_fwd (causal needs Nq <= Nk).
 *   workspace   device, at least attn_bwd_workspace_bytes(B, H, Nq, Nk, d)
 *               bytes, 16-byte aligned; owned by the caller, overwritten,
 *               need not be initialised.  Calls that overlap on the GPU must
 *               not share a workspace.
 *   stream      cudaStream_t.
 * Internal arithmetic: S and dP in fp32 on the tensor cores, P and dS
 * rounded to bf16 for the dV, dK and dQ products, fp32 accumulation of dK
 * and dV in Tensor Memory and of dQ in the workspace (TMA bulk reduce-adds
 * from every key tile, in no fixed order, so the last bits of dQ may differ
 * from run to run).
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG (also for a missing or too-small
 * workspace), ATTN_ERR_UNSUPPORTED, ATTN_ERR_MISALIGNED or ATTN_ERR_CUDA.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, int B, int H, int Nq, int Nk,
             int d, int causal, float scale, void *workspace, size_t workspace_bytes,
             void *stream);

/* attn_status_string -- a static, human-readable name for a status code. */
const char *attn_status_string(int status);

/*
 * attn_device_error -- synchronises the current device, then reads and
 * clears the library's device-side error word.  Returns ATTN_OK when no
 * kernel reported a problem since the last call, ATTN_ERR_TIMEOUT when a
 * kernel abandoned a bounded wait on one of its own barriers (it then wrote
 * no valid output), ATTN_ERR_INVALID_ARG when a kernel found a per-sequence
 * length out of range (attn_fwd_ragged, attn_fwd_decode_ragged), or
 * ATTN_ERR_CUDA if the synchronisation failed.
 */
int attn_device_error(void);

/* attn_version -- library version as major*10000 + minor*100 + patch. */
int attn_version(void);

/*
 * attn_selftest_timeout -- a check of the failure path; the lecture pages
 * have no counterpart.  Enqueues a one-thread kernel that waits on a
 * barrier nothing ever arrives on, with the same bounded wait the attention
 * kernels use.  The wait gives up after the library's limit (2 s), the
 * kernel sets the timeout bit of the device error word and returns, and the
 * next attn_device_error returns ATTN_ERR_TIMEOUT (and clears it).  Nothing
 * faults; the context stays usable.  Returns ATTN_OK or ATTN_ERR_CUDA.
 */
int attn_selftest_timeout(void *stream);

/*
 * Debug builds.  The library also builds as libgbattn_debug.so (compiled with
 * GBATTN_DEBUG), whose kernels check the index of every direct global-memory
 * access (those a TMA tensor map does not bound) against its buffer; an index
 * out of range sets a bit of the device error word and the access is skipped,
 * so attn_device_error returns ATTN_ERR_OUT_OF_RANGE instead of the kernel
 * touching memory it does not own.  Nothing traps.  The lecture pages have no
 * counterpart; this is the library's own stand-in for a memory checker.
 *
 * attn_debug_build -- 1 in the debug build, 0 in the release build.
 * attn_selftest_bounds -- debug builds: enqueue a kernel whose index check
 * fails on purpose (it makes no access); the next attn_device_error returns
 * ATTN_ERR_OUT_OF_RANGE and clears it.  Release builds return
 * ATTN_ERR_UNSUPPORTED and enqueue nothing.
 */
int attn_debug_build(void);
int attn_selftest_bounds(void *stream);

/*
 * The CTA-pair product (PDC Lecture 7 §7.13, CTA pair / MMA.2SM): one thread
 * issues tcgen05.mma.cta_group::2 for a cluster of two CTAs on two SMs, M = 256
 * rows of which each CTA holds 128 in its shared memory and receives 128 in its
 * Tensor Memory, while B's N rows are split N/2 per CTA.  The attention kernels
 * use the single-CTA form; these two calls check the pair form and measure both
 * forms' issue rates.  Both block: they synchronise `stream` before returning.
 *
 * attn_pair_product -- D = A · Bᵀ through four pair products (K = 64 in steps
 * of 16).  a: 256 x 64 bf16, b: 128 x 64 bf16, d: 256 x 128 fp32, all
 * row-major device buffers owned by the caller, 16-byte aligned.  Returns
 * ATTN_OK, ATTN_ERR_INVALID_ARG (a null pointer), ATTN_ERR_MISALIGNED,
 * ATTN_ERR_CUDA, or ATTN_ERR_TIMEOUT (a bounded wait ran out; d is then not
 * valid).
 *
 * attn_bench_mma_rate -- the sustained rate of one issuer.
 *   form   1: each CTA issues 128 x 128 x 16 bf16 products (cta_group::1);
 *          2: the even CTA of each pair issues 256 x 128 x 16 products
 *             (cta_group::2).  Either way every product keeps each SM's
 *             tensor core busy for 64 cycles, and both forms run on the same
 *             SMs: as many CTA pairs as the device holds at once (sms_out
 *             receives how many SMs that is).
 *   issuer 0: lane 0 of warp 0 alone runs the issuing loop;
 *          1: all 32 lanes of warp 0 run it (and its waits) and one lane
 *             chosen by elect.sync issues, as the attention kernels do.
 *   busy   0: the issuing warp runs alone; 1: eight more warps per CTA (two
 *          on each SM sub-partition, where the attention kernels' softmax
 *          warps sit) loop over Tensor Memory loads, packed FMAs, exponentials
 *          and bf16 packs until the products are done.
 *   waits  0: the loop holds no barrier wait (a commit after every 8
 *          products); 1: after issuing group s it waits for group s-1.
 *   steps  groups of 8 products per issuer, 1 to 65536.
 *   reps   timed launches (after one untimed), 1 to 1000.
 *   ms_out (host) mean launch time by CUDA events; cycles_out (host, may be
 *   NULL) mean clock64 cycles of an issuer from its first product to the
 *   completion of its last; sms_out (host, may be NULL).
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_CUDA or ATTN_ERR_TIMEOUT.
 */
int attn_pair_product(const void *a, const void *b, float *d, void *stream);
int attn_bench_mma_rate(int form, int issuer, int busy, int waits, int steps, int reps,
                        float *ms_out, double *cycles_out, int *sms_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
