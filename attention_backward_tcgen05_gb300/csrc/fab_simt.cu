// fab_simt.cu -- CUDA-core (SIMT) attention forward and backward for any
// dtype and any widths DK, DV <= 256.  These serve the f32 path, whose
// accuracy target a bf16 tensor-core contraction cannot meet, and widths the
// tensor-core kernel does not cover.  fp32 arithmetic throughout.
//
// Forward (ggmlR test-flash-attn-back.R, attn_ref; labml "Flash Attention",
// "Flash Attention Optimization"): one warp per query row walks the keys with
// an online softmax (running max, rescaled sum and output), skips
// non-finite scores, and writes o and the natural-log LSE (+inf for a row
// with no finite score).
//
// Backward (labml "Backward pass"): P is recomputed as exp(s - LSE);
// dP = dO . V, dS = P (dP - D).  Two kernels avoid atomics: one warp per
// query row accumulates dQ = scale sum dS K; one warp per key row of a
// key/value head accumulates dK = scale sum dS Q and dV = sum P dO over every
// query head of its GQA group.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "fab.h"
#include "fab_internal.h"

namespace fab {
namespace {

constexpr int kWarps = 8;  // warps per block

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ void from_f32(float& dst, float x) { dst = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16& dst, float x) { dst = __float2bfloat16_rn(x); }
__device__ __forceinline__ void from_f32(__half& dst, float x) { dst = __float2half_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float mask_at(const uint16_t* mask, int64_t M, int64_t m, int64_t n) {
  return __half2float(__ushort_as_half(mask[m + M * n]));
}

// Loads row[lane + 32 j] for j < R (0 beyond `len`).
template <typename T, int R>
__device__ __forceinline__ void load_row(const T* row, int len, int lane, float (&x)[R]) {
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = lane + 32 * j;
    x[j] = i < len ? to_f32(row[i]) : 0.f;
  }
}

template <typename T, int R>
__device__ __forceinline__ float dot_row(const float (&x)[R], const T* row, int len, int lane) {
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = lane + 32 * j;
    if (i < len) acc += x[j] * to_f32(row[i]);
  }
  return warp_sum(acc);
}

template <typename T, int R>
__global__ void __launch_bounds__(kWarps * 32) fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                               const T* __restrict__ v,
                                                               const uint16_t* __restrict__ mask, int causal,
                                                               float scale, int64_t B, int64_t H, int64_t Hkv,
                                                               int64_t N, int64_t M, int DK, int DV,
                                                               T* __restrict__ o, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);  // (b, h, n), n fastest
  if (row >= B * H * N) return;
  const int64_t n = row % N, bh = row / N, h = bh % H, b = bh / H;
  const int64_t hk = h / (H / Hkv);
  float qv[R], acc[R];
  load_row<T, R>(q + row * DK, DK, lane, qv);
#pragma unroll
  for (int j = 0; j < R; ++j) acc[j] = 0.f;
  float mx = -INFINITY, l = 0.f;
  const int64_t mend = causal ? (n + 1 < M ? n + 1 : M) : M;
  const T* kb = k + (b * Hkv + hk) * M * DK;
  const T* vb = v + (b * Hkv + hk) * M * DV;
  for (int64_t m = 0; m < mend; ++m) {
    float s = dot_row<T, R>(qv, kb + m * DK, DK, lane) * scale;
    if (mask) s += mask_at(mask, M, m, n);
    if (!isfinite(s)) continue;
    if (s > mx) {
      const float corr = expf(mx - s);  // exp(-inf) = 0 on the first finite score
      l *= corr;
#pragma unroll
      for (int j = 0; j < R; ++j) acc[j] *= corr;
      mx = s;
    }
    const float p = expf(s - mx);
    l += p;
    const T* vr = vb + m * DV;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int i = lane + 32 * j;
      if (i < DV) acc[j] += p * to_f32(vr[i]);
    }
  }
  T* orow = o + ((b * N + n) * H + h) * DV;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = lane + 32 * j;
    if (i < DV) from_f32(orow[i], acc[j] * inv);
  }
  if (lane == 0) lse[(b * H + h) * N + n] = l > 0.f ? mx + logf(l) : INFINITY;
}

template <typename T, int R>
__global__ void __launch_bounds__(kWarps * 32) dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                              const T* __restrict__ v, const T* __restrict__ d,
                                                              const float* __restrict__ lse,
                                                              const float* __restrict__ di,
                                                              const uint16_t* __restrict__ mask, int causal,
                                                              float scale, int64_t B, int64_t H, int64_t Hkv,
                                                              int64_t N, int64_t M, int DK, int DV,
                                                              float* __restrict__ dq) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);  // (b, h, n), n fastest
  if (row >= B * H * N) return;
  const int64_t n = row % N, bh = row / N, h = bh % H, b = bh / H;
  const int64_t hk = h / (H / Hkv);
  const float L = lse[row], Dn = di[row];
  float acc[R];
#pragma unroll
  for (int j = 0; j < R; ++j) acc[j] = 0.f;
  if (!isinf(L)) {
    float qv[R], dov[R];
    load_row<T, R>(q + row * DK, DK, lane, qv);
    load_row<T, R>(d + ((b * N + n) * H + h) * DV, DV, lane, dov);
    const int64_t mend = causal ? (n + 1 < M ? n + 1 : M) : M;
    const T* kb = k + (b * Hkv + hk) * M * DK;
    const T* vb = v + (b * Hkv + hk) * M * DV;
    for (int64_t m = 0; m < mend; ++m) {
      float s = dot_row<T, R>(qv, kb + m * DK, DK, lane) * scale;
      if (mask) s += mask_at(mask, M, m, n);
      if (!isfinite(s)) continue;
      const float p = expf(s - L);
      const float dp = dot_row<T, R>(dov, vb + m * DV, DV, lane);
      const float ds = p * (dp - Dn);
      const T* kr = kb + m * DK;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int i = lane + 32 * j;
        if (i < DK) acc[j] += ds * to_f32(kr[i]);
      }
    }
  }
  float* out = dq + row * DK;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = lane + 32 * j;
    if (i < DK) out[i] = scale * acc[j];
  }
}

template <typename T, int R>
__global__ void __launch_bounds__(kWarps * 32) dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                                const T* __restrict__ v, const T* __restrict__ d,
                                                                const float* __restrict__ lse,
                                                                const float* __restrict__ di,
                                                                const uint16_t* __restrict__ mask, int causal,
                                                                float scale, int64_t B, int64_t H, int64_t Hkv,
                                                                int64_t N, int64_t M, int DK, int DV,
                                                                float* __restrict__ dk, float* __restrict__ dv) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);  // (b, hk, m), m fastest
  if (row >= B * Hkv * M) return;
  const int64_t m = row % M, bhk = row / M, hk = bhk % Hkv, b = bhk / Hkv;
  const int64_t rk2 = H / Hkv;
  float kv[R], vv[R], adk[R], adv[R];
  load_row<T, R>(k + row * DK, DK, lane, kv);
  load_row<T, R>(v + row * DV, DV, lane, vv);
#pragma unroll
  for (int j = 0; j < R; ++j) adk[j] = adv[j] = 0.f;
  for (int64_t h = hk * rk2; h < (hk + 1) * rk2; ++h) {
    const T* qb = q + (b * H + h) * N * DK;
    const float* lb = lse + (b * H + h) * N;
    const float* db = di + (b * H + h) * N;
    for (int64_t n = causal ? m : 0; n < N; ++n) {
      const float L = lb[n];
      if (isinf(L)) continue;  // a row with no finite score contributes nothing
      float s = dot_row<T, R>(kv, qb + n * DK, DK, lane) * scale;
      if (mask) s += mask_at(mask, M, m, n);
      if (!isfinite(s)) continue;
      const float p = expf(s - L);
      const T* dor = d + ((b * N + n) * H + h) * DV;
      const float dp = dot_row<T, R>(vv, dor, DV, lane);
      const float ds = p * (dp - db[n]);
      const T* qr = qb + n * DK;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int i = lane + 32 * j;
        if (i < DK) adk[j] += ds * to_f32(qr[i]);
        if (i < DV) adv[j] += p * to_f32(dor[i]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = lane + 32 * j;
    if (i < DK) dk[row * DK + i] = scale * adk[j];
    if (i < DV) dv[row * DV + i] = adv[j];
  }
}

template <typename T, int R>
cudaError_t fwd_r(const Problem& p, void* o, float* lse, cudaStream_t s) {
  const int64_t rows = p.B * p.H * p.N;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  fwd_simt_kernel<T, R><<<grid, kWarps * 32, 0, s>>>(
      static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v), p.mask, p.causal,
      p.scale, p.B, p.H, p.Hkv, p.N, p.M, (int)p.DK, (int)p.DV, static_cast<T*>(o), lse);
  return cudaPeekAtLastError();
}

template <typename T, int R>
cudaError_t bwd_r(const Problem& p, cudaStream_t s) {
  const int64_t qrows = p.B * p.H * p.N, krows = p.B * p.Hkv * p.M;
  dq_simt_kernel<T, R><<<(unsigned)((qrows + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(
      static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v),
      static_cast<const T*>(p.d), p.lse, p.di, p.mask, p.causal, p.scale, p.B, p.H, p.Hkv, p.N, p.M, (int)p.DK,
      (int)p.DV, p.packed);
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  dkdv_simt_kernel<T, R><<<(unsigned)((krows + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(
      static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v),
      static_cast<const T*>(p.d), p.lse, p.di, p.mask, p.causal, p.scale, p.B, p.H, p.Hkv, p.N, p.M, (int)p.DK,
      (int)p.DV, p.packed + p.off_k / 4, p.packed + p.off_v / 4);
  return cudaPeekAtLastError();
}

int regs_per_lane(const Problem& p) {
  const int64_t w = p.DK > p.DV ? p.DK : p.DV;
  return (int)((w + 31) / 32);
}

// widths up to 32 R per lane
template <typename T>
cudaError_t fwd_t(const Problem& p, int r, void* o, float* lse, cudaStream_t s) {
  if (r <= 1) return fwd_r<T, 1>(p, o, lse, s);
  if (r <= 2) return fwd_r<T, 2>(p, o, lse, s);
  if (r <= 4) return fwd_r<T, 4>(p, o, lse, s);
  return fwd_r<T, 8>(p, o, lse, s);
}
template <typename T>
cudaError_t bwd_t(const Problem& p, int r, cudaStream_t s) {
  if (r <= 1) return bwd_r<T, 1>(p, s);
  if (r <= 2) return bwd_r<T, 2>(p, s);
  if (r <= 4) return bwd_r<T, 4>(p, s);
  return bwd_r<T, 8>(p, s);
}

}  // namespace

cudaError_t launch_forward_simt(const Problem& p, void* o, float* lse, cudaStream_t s) {
  const int r = regs_per_lane(p);
  if (p.dtype == FAB_BF16) return fwd_t<__nv_bfloat16>(p, r, o, lse, s);
  if (p.dtype == FAB_F16) return fwd_t<__half>(p, r, o, lse, s);
  return fwd_t<float>(p, r, o, lse, s);
}

cudaError_t launch_backward_simt(const Problem& p, cudaStream_t s) {
  const int r = regs_per_lane(p);
  if (p.dtype == FAB_BF16) return bwd_t<__nv_bfloat16>(p, r, s);
  if (p.dtype == FAB_F16) return bwd_t<__half>(p, r, s);
  return bwd_t<float>(p, r, s);
}

}  // namespace fab
