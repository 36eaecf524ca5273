// fab_host.cu -- the C ABI of libfab (declared in include/fab.h): argument
// validation, packed-layout arithmetic, and the stream-ordered launches.
// Nothing here allocates device memory or synchronises, except
// fab_last_device_error, whose job is to synchronise.
#include <mutex>

#include "fab.h"
#include "fab_internal.h"

#define FAB_API extern "C" FAB_EXPORT

namespace fab {

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {

constexpr int64_t kMaxWidth = 256;  // DK, DV limit of every kernel
constexpr int64_t kMaxElems = int64_t(1) << 40;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t pad16(int64_t bytes) { return (bytes + 15) / 16 * 16; }

// The ggml_flash_attn_back constructor's shape rules (k rows as wide as q
// rows, matching batch/head counts, H % Hkv == 0) expressed on fab_dims, plus
// positivity and overflow guards.
int check_dims(const fab_dims* d) {
  if (!d) return FAB_ERR_INVALID;
  if (d->B <= 0 || d->H <= 0 || d->Hkv <= 0 || d->N <= 0 || d->M <= 0 || d->DK <= 0 || d->DV <= 0)
    return FAB_ERR_INVALID;
  if (d->H % d->Hkv != 0) return FAB_ERR_INVALID;
  const int64_t lim = kMaxElems;
  if (d->B > lim / d->H || d->B * d->H > lim / d->N || d->B * d->H * d->N > lim / (d->DK > d->DV ? d->DK : d->DV))
    return FAB_ERR_INVALID;
  if (d->B > lim / d->Hkv || d->B * d->Hkv > lim / d->M ||
      d->B * d->Hkv * d->M > lim / (d->DK > d->DV ? d->DK : d->DV))
    return FAB_ERR_INVALID;
  return FAB_OK;
}

void layout(const fab_dims* d, size_t* off_k, size_t* off_v, size_t* end) {
  const int64_t elem_q = d->DK * d->N * d->H * d->B;
  const int64_t elem_k = d->DK * d->M * d->Hkv * d->B;
  const int64_t elem_v = d->DV * d->M * d->Hkv * d->B;
  const int64_t ok = pad16(elem_q * 4);
  const int64_t ov = ok + pad16(elem_k * 4);
  *off_k = (size_t)ok;
  *off_v = (size_t)ov;
  *end = (size_t)(ov + pad16(elem_v * 4));
}

size_t di_bytes(const fab_dims* d) {
  const size_t b = (size_t)(d->B * d->H * d->N) * sizeof(float);
  return (b + 255) / 256 * 256;
}

// After D_i: the mask's live-tile maps (a byte per 128 x 128 tile, by query
// tile rows and by key tile rows), which let the tensor-core passes skip
// tiles whose mask entries are all -inf.  Optional: a workspace without room
// for them skips nothing.
size_t live_map_bytes(const fab_dims* d) {
  const int64_t qt = (d->N + 127) / 128, kt = (d->M + 127) / 128;
  const size_t b = (size_t)(qt * live_stride(kt) + kt * live_stride(qt));
  return (b + 255) / 256 * 256;
}
size_t aux_bytes(const fab_dims* d) { return di_bytes(d) + live_map_bytes(d); }

// The forward output O [DV,H,N,B] and the row LSE [N,H,B] that fab_backward
// keeps in its workspace, after D_i and the live-tile maps, when the caller passes
// neither.
size_t o_bytes(const fab_dims* d, int dtype) {
  const size_t b = (size_t)(d->B * d->H * d->N * d->DV) * (dtype == FAB_F32 ? 4u : 2u);
  return (b + 255) / 256 * 256;
}
size_t recompute_bytes(const fab_dims* d, int dtype) { return aux_bytes(d) + o_bytes(d, dtype) + di_bytes(d); }

// Points p's live-tile maps into the workspace when there is a mask and room.
void set_live_maps(Problem* p, const fab_dims* d, const void* workspace, size_t workspace_bytes) {
  p->kt_live = p->qt_live = nullptr;
  // (the scan's grid holds up to 65535 query tiles)
  if (p->mask == nullptr || workspace_bytes < aux_bytes(d) || (d->N + 127) / 128 > 65535) return;
  uint8_t* ws = static_cast<uint8_t*>(const_cast<void*>(workspace));
  p->kt_live = ws + di_bytes(d);
  p->qt_live = p->kt_live + (d->N + 127) / 128 * live_stride((d->M + 127) / 128);
}

// The live-tile maps the tensor-core passes read, written on the stream before them.
cudaError_t scan_live_tiles(const Problem& p, cudaStream_t s) {
  return p.kt_live != nullptr ? launch_mask_scan(p, s) : cudaSuccess;
}

Problem make_problem(const fab_dims* d, int dtype, float scale, int causal) {
  Problem p{};
  p.B = d->B;
  p.H = d->H;
  p.Hkv = d->Hkv;
  p.N = d->N;
  p.M = d->M;
  p.DK = d->DK;
  p.DV = d->DV;
  p.scale = scale;
  p.causal = causal ? 1 : 0;
  p.dtype = dtype;
  layout(d, &p.off_k, &p.off_v, &p.end);
  return p;
}

bool dtype_ok(int dtype) { return dtype == FAB_F32 || dtype == FAB_BF16 || dtype == FAB_F16; }

bool widths_supported(const fab_dims* d) { return d->DK <= kMaxWidth && d->DV <= kMaxWidth; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? FAB_OK : FAB_ERR_CUDA; }

// Common checks of the backward entry points.  `need_*` select which pointers
// the entry point reads.
int check_backward(const fab_dims* dims, int dtype, const void* const* ptrs, int nptrs, const uint16_t* mask,
                   const void* workspace, size_t workspace_bytes, const float* packed) {
  int rc = check_dims(dims);
  if (rc != FAB_OK) return rc;
  if (!dtype_ok(dtype)) return FAB_ERR_INVALID;
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return FAB_ERR_INVALID;
  if (mask && !aligned16(mask)) return FAB_ERR_INVALID;
  if (!packed || !aligned16(packed)) return FAB_ERR_INVALID;
  if (!workspace || !aligned16(workspace) || workspace_bytes < di_bytes(dims)) return FAB_ERR_WORKSPACE;
  if (!widths_supported(dims)) return FAB_ERR_UNSUPPORTED;
  return FAB_OK;
}

}  // namespace
}  // namespace fab

using namespace fab;

FAB_API int fab_version(void) { return 100; }

FAB_API const char* fab_status_string(int status) {
  switch (status) {
    case FAB_OK:
      return "ok";
    case FAB_ERR_INVALID:
      return "invalid argument (null or misaligned pointer, bad dims, H % Hkv != 0)";
    case FAB_ERR_UNSUPPORTED:
      return "unsupported dims or dtype for the GPU kernels";
    case FAB_ERR_WORKSPACE:
      return "workspace missing, misaligned or too small";
    case FAB_ERR_CUDA:
      return "CUDA runtime error";
    case FAB_ERR_TIMEOUT:
      return "a device-side wait ran out; the kernel's outputs are invalid";
    default:
      return "unknown status";
  }
}

FAB_API int fab_packed_offsets(const fab_dims* dims, size_t* off_k, size_t* off_v, size_t* end) {
  const int rc = check_dims(dims);
  if (rc != FAB_OK) return rc;
  size_t a, b, c;
  layout(dims, &a, &b, &c);
  if (off_k) *off_k = a;
  if (off_v) *off_v = b;
  if (end) *end = c;
  return FAB_OK;
}

FAB_API size_t fab_packed_bytes(const fab_dims* dims) {
  size_t end = 0;
  if (fab_packed_offsets(dims, nullptr, nullptr, &end) != FAB_OK) return 0;
  return end;
}

FAB_API size_t fab_backward_workspace_bytes(const fab_dims* dims, int dtype) {
  if (check_dims(dims) != FAB_OK || !dtype_ok(dtype)) return 0;
  return aux_bytes(dims);
}

FAB_API size_t fab_backward_recompute_workspace_bytes(const fab_dims* dims, int dtype) {
  if (check_dims(dims) != FAB_OK || !dtype_ok(dtype)) return 0;
  return recompute_bytes(dims, dtype);
}

namespace {

// fab_forward_lse; live: the mask's live-tile maps (scanned on the stream
// before), which let the tensor-core forward skip all -inf tiles, or null.
int forward_lse(const void* q, const void* k, const void* v, const uint16_t* mask, int causal, float scale,
                int dtype, const fab_dims* dims, void* o, float* lse, const Problem* live, fab_stream stream) {
  int rc = check_dims(dims);
  if (rc != FAB_OK) return rc;
  if (!dtype_ok(dtype)) return FAB_ERR_INVALID;
  const void* ptrs[5] = {q, k, v, o, lse};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FAB_ERR_INVALID;
  if (mask && !aligned16(mask)) return FAB_ERR_INVALID;
  if (!widths_supported(dims)) return FAB_ERR_UNSUPPORTED;
  Problem p = make_problem(dims, dtype, scale, causal);
  p.q = q;
  p.k = k;
  p.v = v;
  p.mask = mask;
  if (live != nullptr && mask != nullptr) {
    p.kt_live = live->kt_live;
    p.qt_live = live->qt_live;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (forward_tc_supported(p)) {
    if (!encode_tiled_fn()) return FAB_ERR_CUDA;
    return from_cuda(launch_forward_tc(p, o, lse, s));
  }
  return from_cuda(launch_forward_simt(p, o, lse, s));
}

}  // namespace

FAB_API int fab_forward_lse(const void* q, const void* k, const void* v, const uint16_t* mask, int causal,
                            float scale, int dtype, const fab_dims* dims, void* o, float* lse, fab_stream stream) {
  return forward_lse(q, k, v, mask, causal, scale, dtype, dims, o, lse, nullptr, stream);
}

FAB_API int fab_backward_preprocess(const void* d, const void* o, int dtype, const fab_dims* dims, void* workspace,
                                    size_t workspace_bytes, float* packed_out, fab_stream stream) {
  const void* ptrs[2] = {d, o};
  int rc = check_backward(dims, dtype, ptrs, 2, nullptr, workspace, workspace_bytes, packed_out);
  if (rc != FAB_OK) return rc;
  Problem p = make_problem(dims, dtype, 1.f, 0);
  p.d = d;
  p.o = o;
  p.di = static_cast<float*>(workspace);
  p.packed = packed_out;
  return from_cuda(launch_preprocess(p, static_cast<cudaStream_t>(stream)));
}

FAB_API int fab_backward_main(const void* q, const void* k, const void* v, const void* d, const float* lse,
                              const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims,
                              const void* workspace, size_t workspace_bytes, float* packed_out, fab_stream stream) {
  const void* ptrs[5] = {q, k, v, d, lse};
  int rc = check_backward(dims, dtype, ptrs, 5, mask, workspace, workspace_bytes, packed_out);
  if (rc != FAB_OK) return rc;
  Problem p = make_problem(dims, dtype, scale, causal);
  p.q = q;
  p.k = k;
  p.v = v;
  p.d = d;
  p.lse = lse;
  p.mask = mask;
  p.di = static_cast<float*>(const_cast<void*>(workspace));
  p.packed = packed_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (backward_tc_supported(p)) {
    if (!encode_tiled_fn()) return FAB_ERR_CUDA;
    set_live_maps(&p, dims, workspace, workspace_bytes);
    rc = from_cuda(scan_live_tiles(p, s));
    if (rc != FAB_OK) return rc;
    // query pass (dQ), then key/value pass (dK, dV); they write disjoint slices
    rc = from_cuda(launch_dq_tc(p, false, s));
    if (rc != FAB_OK) return rc;
    return from_cuda(launch_backward_tc(p, s));
  }
  return from_cuda(launch_backward_simt(p, s));
}

namespace {

// The tensor-core problem of a validated backward call (fab_backward's
// arguments); false when the tensor-core kernels do not cover it.
bool tc_problem(const void* q, const void* k, const void* v, const void* d, const void* o, const float* lse,
                const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims, void* workspace,
                float* packed_out, Problem* out) {
  Problem p = make_problem(dims, dtype, scale, causal);
  if (!backward_tc_supported(p)) return false;
  p.q = q;
  p.k = k;
  p.v = v;
  p.d = d;
  p.o = o;
  p.lse = lse;
  p.mask = mask;
  p.di = static_cast<float*>(workspace);
  p.packed = packed_out;
  *out = p;
  return true;
}

}  // namespace

FAB_API int fab_backward_query_pass(const void* q, const void* k, const void* v, const void* d, const void* o,
                                    const float* lse, const uint16_t* mask, int causal, float scale, int dtype,
                                    const fab_dims* dims, void* workspace, size_t workspace_bytes, float* packed_out,
                                    fab_stream stream) {
  const void* ptrs[6] = {q, k, v, d, o, lse};
  int rc = check_backward(dims, dtype, ptrs, 6, mask, workspace, workspace_bytes, packed_out);
  if (rc != FAB_OK) return rc;
  Problem p;
  if (!tc_problem(q, k, v, d, o, lse, mask, causal, scale, dtype, dims, workspace, packed_out, &p))
    return FAB_ERR_UNSUPPORTED;
  if (!encode_tiled_fn()) return FAB_ERR_CUDA;
  set_live_maps(&p, dims, workspace, workspace_bytes);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = from_cuda(scan_live_tiles(p, s));
  if (rc != FAB_OK) return rc;
  return from_cuda(launch_dq_tc(p, true, s));
}

FAB_API int fab_backward_key_pass(const void* q, const void* k, const void* v, const void* d, const float* lse,
                                  const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims,
                                  const void* workspace, size_t workspace_bytes, float* packed_out,
                                  fab_stream stream) {
  const void* ptrs[5] = {q, k, v, d, lse};
  int rc = check_backward(dims, dtype, ptrs, 5, mask, workspace, workspace_bytes, packed_out);
  if (rc != FAB_OK) return rc;
  Problem p;
  if (!tc_problem(q, k, v, d, nullptr, lse, mask, causal, scale, dtype, dims, const_cast<void*>(workspace),
                  packed_out, &p))
    return FAB_ERR_UNSUPPORTED;
  if (!encode_tiled_fn()) return FAB_ERR_CUDA;
  set_live_maps(&p, dims, workspace, workspace_bytes);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = from_cuda(scan_live_tiles(p, s));
  if (rc != FAB_OK) return rc;
  return from_cuda(launch_backward_tc(p, s));
}

FAB_API int fab_backward(const void* q, const void* k, const void* v, const void* d, const void* o, const float* lse,
                         const uint16_t* mask, int causal, float scale, int dtype, const fab_dims* dims,
                         void* workspace, size_t workspace_bytes, float* packed_out, fab_stream stream) {
  bool scanned = false;  // the mask's live tiles already in the workspace
  if (o == nullptr || lse == nullptr) {
    // ggml_flash_attn_back's operands are q, k, v, the mask and d alone: with
    // neither o nor lse given, the forward is recomputed into the workspace
    // (after D_i) before the backward proper
    if (o != nullptr || lse != nullptr) return FAB_ERR_INVALID;
    const void* ptrs4[4] = {q, k, v, d};
    int rc0 = check_backward(dims, dtype, ptrs4, 4, mask, workspace, workspace_bytes, packed_out);
    if (rc0 != FAB_OK) return rc0;
    if (workspace_bytes < recompute_bytes(dims, dtype)) return FAB_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* o2 = ws + aux_bytes(dims);
    float* lse2 = reinterpret_cast<float*>(ws + aux_bytes(dims) + o_bytes(dims, dtype));
    // the mask's live tiles, scanned once for the forward and the backward
    Problem live = make_problem(dims, dtype, scale, causal);
    live.mask = mask;
    set_live_maps(&live, dims, workspace, workspace_bytes);
    rc0 = from_cuda(scan_live_tiles(live, static_cast<cudaStream_t>(stream)));
    if (rc0 != FAB_OK) return rc0;
    rc0 = forward_lse(q, k, v, mask, causal, scale, dtype, dims, o2, lse2, &live, stream);
    if (rc0 != FAB_OK) return rc0;
    o = o2;
    lse = lse2;
    scanned = true;
  }
  const void* ptrs[6] = {q, k, v, d, o, lse};
  int rc = check_backward(dims, dtype, ptrs, 6, mask, workspace, workspace_bytes, packed_out);
  if (rc != FAB_OK) return rc;
  Problem p;
  if (tc_problem(q, k, v, d, o, lse, mask, causal, scale, dtype, dims, workspace, packed_out, &p)) {
    // what fab_backward_query_pass then fab_backward_key_pass enqueue, with
    // the mask's live tiles scanned once: the query pass computes D_i itself
    // (and zeroes the padding), then the key/value pass reads it
    if (!encode_tiled_fn()) return FAB_ERR_CUDA;
    set_live_maps(&p, dims, workspace, workspace_bytes);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!scanned) {
      rc = from_cuda(scan_live_tiles(p, s));
      if (rc != FAB_OK) return rc;
    }
    rc = from_cuda(launch_dq_tc(p, true, s));
    if (rc != FAB_OK) return rc;
    return from_cuda(launch_backward_tc(p, s));
  }
  rc = fab_backward_preprocess(d, o, dtype, dims, workspace, workspace_bytes, packed_out, stream);
  if (rc != FAB_OK) return rc;
  return fab_backward_main(q, k, v, d, lse, mask, causal, scale, dtype, dims, workspace, workspace_bytes, packed_out,
                           stream);
}

FAB_API int fab_last_device_error(fab_stream stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FAB_ERR_CUDA;
  const uint32_t e = take_error_tc() | take_error_dq() | take_error_fwd();
  if (e & kErrSmemAlign) return FAB_ERR_CUDA;
  return (e & kErrTimeout) ? FAB_ERR_TIMEOUT : FAB_OK;
}
