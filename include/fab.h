/*
 * fab.h -- C ABI of libfab, the fused attention backward library for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The operation is ggml_flash_attn_back: given the forward's inputs q, k, v,
 * the upstream gradient d of the forward output, a softmax scale and an
 * optional causal flag and/or additive f16 mask, return dQ, dK and dV as f32,
 * packed into one buffer.  Sources, by page and section:
 *   - the ggml_flash_attn_back constructor (PowerInfer ggml.c): shape
 *     asserts (k rows match q rows, H % Hkv == 0), f32 result type, and the
 *     packed offsets offs_k = PAD(elem_q*4, 16), offs_v = offs_k +
 *     PAD(elem_k*4, 16), end = offs_v + PAD(elem_v*4, 16);
 *   - the ggmlR test file test-flash-attn-back.R: the call shape
 *     (q, k, v, mask, d, scale), layouts q [DK,N,H,B], k [DK,M,Hkv,B],
 *     v [DV,M,Hkv,B], forward output and d [DV,H,N,B], mask f16 [M,N]
 *     added after scaling (attn_ref), contiguous GQA groups, the causal mask
 *     (query n attends keys 0..n), rows with no finite score giving zero
 *     output, and a zero-filled packed buffer whose padding stays 0;
 *   - the labml "Flash Attention" page, sections "Forward pass", "Flash
 *     Attention Optimization" (online softmax) and "Backward pass": the
 *     gradient formulas, with D_i = dO_i . O_i.
 *
 * Layout convention: every tensor is contiguous in ggml ne order (ne[0]
 * fastest), e.g. q[i, n, h, b] is at i + DK*(n + N*(h + H*b)).
 *   q    [DK, N, H, B]     k [DK, M, Hkv, B]     v [DV, M, Hkv, B]
 *   o, d [DV, H, N, B]     (the forward output and its gradient)
 *   lse  [N, H, B] f32     (natural-log row log-sum-exp of the scaled,
 *                           masked scores; +inf for a row with no finite score)
 *   mask [M, N] f16        (mask[m + M*n] is added to score(n, m); shared by
 *                           every head and batch; only -inf and finite values
 *                           are defined)
 *   packed f32: [dQ as q | 0 pad | dK as k | 0 pad | dV as v | 0 pad],
 *               byte offsets from fab_packed_offsets().
 * Causal masking is top-left: query n attends keys m <= n (also when N != M).
 * When both `causal` and a mask are given, both apply.
 *
 * Ownership and execution: the caller owns every buffer.  Device pointers
 * must point to device memory of the current device and be 16-byte aligned.
 * The library never allocates, frees or synchronises: each compute entry point
 * validates its arguments on the host, enqueues kernels on `stream` and
 * returns.  A status other than FAB_OK means nothing was enqueued, except
 * FAB_ERR_CUDA, which reports a launch error (the stream state is then the
 * CUDA runtime's).  Device-side waits are bounded: a wait that runs out sets
 * an error word that fab_last_device_error() returns as FAB_ERR_TIMEOUT.
 *
 * Supported on the GPU: dtype FAB_F32 (any DK, DV <= 256), FAB_BF16 and
 * FAB_F16 (tensor-core path when DK == DV and DK is 64 or 128, with P and dS
 * rounded to the input type for their products; any DK, DV <= 256
 * otherwise).  Anything else returns FAB_ERR_UNSUPPORTED; there is no CPU
 * fallback.  ALiBi and logit soft-capping are not part of this ABI.
 */
#ifndef FAB_H
#define FAB_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FAB_EXPORT __attribute__((visibility("default")))
#else
#define FAB_EXPORT
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FAB_OK = 0,
  FAB_ERR_INVALID = 1,     /* null/misaligned pointer, bad dims, H % Hkv != 0 */
  FAB_ERR_UNSUPPORTED = 2, /* valid op, but no GPU kernel for these dims/dtype */
  FAB_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  FAB_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  FAB_ERR_TIMEOUT = 5      /* a device-side wait ran out (see fab_last_device_error) */
} fab_status;

typedef enum {
  FAB_F32 = 0,  /* q, k, v, d, o are float32 */
  FAB_BF16 = 1, /* q, k, v, d, o are bfloat16 */
  FAB_F16 = 2   /* q, k, v, d, o are float16 (IEEE binary16) */
} fab_dtype;

/* Sizes in ggml terms: B batches, H query heads, Hkv key/value heads
 * (H % Hkv == 0; query head h uses key/value head h / (H / Hkv)), N queries,
 * M keys, DK query/key width, DV value width.  All must be positive. */
typedef struct {
  int64_t B, H, Hkv, N, M, DK, DV;
} fab_dims;

/* An opaque cudaStream_t; NULL is the legacy default stream. */
typedef void* fab_stream;

/* Library version, major*10000 + minor*100 + patch. */
FAB_EXPORT int fab_version(void);

/* Human-readable text for a fab_status value; never NULL. */
FAB_EXPORT const char* fab_status_string(int status);

/* Byte offsets of the dK and dV slices and the total size of the packed
 * result (the ggml_flash_attn_back constructor's offs_k, offs_v, end).
 * Returns FAB_ERR_INVALID for bad dims (the outputs are then untouched). */
FAB_EXPORT int fab_packed_offsets(const fab_dims* dims, size_t* off_k, size_t* off_v, size_t* end);

/* Total packed bytes (== end above), or 0 for bad dims. */
FAB_EXPORT size_t fab_packed_bytes(const fab_dims* dims);

/* Device workspace bytes fab_backward needs: D_i = rowsum(dO * O), f32
 * [N,H,B], then, for a call with a mask, the mask's live-tile maps (a byte
 * per 128 x 128 tile, nonzero where some mask entry is not -inf, by query
 * tile rows then by key tile rows, each row padded to 16 bytes; the
 * tensor-core passes skip the tiles before the first and after the last live
 * tile of each row, which changes no result bit; a workspace that ends after
 * D_i skips nothing), each part a multiple of 256 bytes.  0 for bad dims. */
FAB_EXPORT size_t fab_backward_workspace_bytes(const fab_dims* dims, int dtype);

/* Device workspace bytes fab_backward needs when called without o and lse
 * (it then recomputes them): D_i and the live-tile maps as above, then O
 * (`dtype`, [DV,H,N,B]) and LSE (f32, [N,H,B]), each part a multiple of 256
 * bytes.  0 for bad dims. */
FAB_EXPORT size_t fab_backward_recompute_workspace_bytes(const fab_dims* dims, int dtype);

/* Forward pass saving what the backward needs (labml "Flash Attention",
 * "Forward pass" and "Flash Attention Optimization"; ggmlR attn_ref):
 *   o[:, h, n, b] = sum_m softmax_m(scale * q_n . k_m + mask[m + M*n]) v_m
 *   lse[n, h, b]  = log sum_m exp(scale * q_n . k_m + mask[m + M*n])
 * q, k, v: device, `dtype`; mask: device f16 [M,N] or NULL; o: device,
 * `dtype`, [DV,H,N,B]; lse: device f32 [N,H,B].  A query row with no finite
 * score gets o = 0 and lse = +inf. */
FAB_EXPORT int fab_forward_lse(const void* q, const void* k, const void* v, const uint16_t* mask, int causal, float scale,
                    int dtype, const fab_dims* dims, void* o, float* lse, fab_stream stream);

/* Backward pass (ggml_flash_attn_back; labml "Backward pass"):
 *   dV_m = sum_n P_nm dO_n,  dP_nm = dO_n . V_m,  D_n = dO_n . O_n,
 *   dS_nm = P_nm (dP_nm - D_n),  dQ_n = scale sum_m dS_nm K_m,
 *   dK_m = scale sum_n dS_nm Q_n,
 * with P recomputed from q, k, mask, causal, scale and the saved lse; dK and
 * dV are summed over each GQA group's query heads.  o and lse must come from
 * fab_forward_lse on the same inputs; or both be NULL, as in
 * ggml_flash_attn_back, whose operands are q, k, v, the mask and d alone:
 * the call then enqueues fab_forward_lse into the workspace first (exactly one
 * of them NULL is FAB_ERR_INVALID).  d: device, `dtype`, [DV,H,N,B].
 * workspace: device, >= fab_backward_workspace_bytes() bytes (with o and lse
 * NULL: fab_backward_recompute_workspace_bytes()), contents overwritten.  packed_out: device f32, fab_packed_bytes() bytes, fully
 * overwritten (padding written as 0).  Where the tensor-core kernels apply
 * (bf16 or f16, DK == DV in {64, 128}) it enqueues fab_backward_query_pass then
 * fab_backward_key_pass; otherwise fab_backward_preprocess then
 * fab_backward_main. */
FAB_EXPORT int fab_backward(const void* q, const void* k, const void* v, const void* d, const void* o, const float* lse,
                 const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims, void* workspace,
                 size_t workspace_bytes, float* packed_out, fab_stream stream);

/* First half of fab_backward (labml "Backward pass", D_i = dO_i . O_i):
 * writes D into the workspace, zeroes the padding of packed_out and, where the
 * main kernel accumulates dQ, the dQ slice.  Same arguments as fab_backward
 * minus those the preprocess does not read. */
FAB_EXPORT int fab_backward_preprocess(const void* d, const void* o, int dtype, const fab_dims* dims, void* workspace,
                            size_t workspace_bytes, float* packed_out, fab_stream stream);

/* Second half of fab_backward: the gradient kernels proper.  Requires the
 * workspace and packed_out as fab_backward_preprocess left them. */
FAB_EXPORT int fab_backward_main(const void* q, const void* k, const void* v, const void* d, const float* lse,
                      const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims,
                      const void* workspace, size_t workspace_bytes, float* packed_out, fab_stream stream);

/* The two tensor-core passes that make up fab_backward for bf16 or f16 inputs
 * with DK == DV in {64, 128} (labml "Backward pass"); FAB_ERR_UNSUPPORTED
 * otherwise.  Same arguments as fab_backward.
 * fab_backward_query_pass: D_i = dO_i . O_i into the workspace, the dQ slice
 * of packed_out (dQ_n = scale sum_m dS_nm K_m, recomputing S and dP per query
 * tile) and the padding of packed_out.
 * fab_backward_key_pass: the dK and dV slices of packed_out, reading D_i
 * from the workspace (written by the query pass or fab_backward_preprocess);
 * it does not read o. */
FAB_EXPORT int fab_backward_query_pass(const void* q, const void* k, const void* v, const void* d, const void* o,
                            const float* lse, const uint16_t* mask, int causal, float scale, int dtype,
                            const fab_dims* dims, void* workspace, size_t workspace_bytes, float* packed_out,
                            fab_stream stream);
FAB_EXPORT int fab_backward_key_pass(const void* q, const void* k, const void* v, const void* d, const float* lse,
                          const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims,
                          const void* workspace, size_t workspace_bytes, float* packed_out, fab_stream stream);

/* Largest B*H*N that fab_backward_noalloc accepts (query rows times heads
 * times batches): its fixed scratch holds one float per such row. */
#define FAB_NOALLOC_MAX_ROWS 1048576

/* fab_backward for callers that cannot allocate device memory (o and lse
 * must be given: the fixed scratch holds D_i and, when they fit after it, the
 * mask's live-tile maps, not a recomputed O and LSE), for example
 * code whose device memory belongs to another allocator, or code that must not
 * call cudaMalloc (which can synchronise the device) on its path.  The pages
 * have no counterpart; the operation and every argument are those of
 * fab_backward minus the workspace.  The workspace lives instead in a fixed
 * device array inside the library: FAB_NOALLOC_MAX_ROWS floats (4 MiB), held
 * on every GPU that loads the library until the process exits.  Returns
 * FAB_ERR_WORKSPACE when B*H*N exceeds FAB_NOALLOC_MAX_ROWS; allocates and
 * frees nothing.  The first call on a device looks up the array's device
 * address with that device current; make that first call before any stream
 * capture.  The address is kept for the life of the process: after a
 * cudaDeviceReset of that device, do not call this entry point there again.  Calls on one device share the array, so two calls that may run
 * at the same time on the GPU (on unordered streams) race; order them.  No
 * part of the array needs clearing between calls. */
FAB_EXPORT int fab_backward_noalloc(const void* q, const void* k, const void* v, const void* d, const void* o,
                                    const float* lse, const uint16_t* mask, int causal, float scale, int dtype,
                                    const fab_dims* dims, float* packed_out, fab_stream stream);

/* Synchronises `stream`, then returns and clears the device-side error word
 * of the current device: FAB_OK, FAB_ERR_TIMEOUT (a bounded wait inside a
 * kernel ran out; that kernel's outputs are invalid) or FAB_ERR_CUDA. */
FAB_EXPORT int fab_last_device_error(fab_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* FAB_H */
