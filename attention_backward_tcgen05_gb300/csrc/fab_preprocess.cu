// fab_preprocess.cu -- the backward's memory-bound first step.
//
//   D_i = dO_i . O_i  (labml "Flash Attention", "Backward pass": the per-row
//   term sum_k P_ik dP_ik rewritten as the dot product of the output row and
//   its gradient), for every query row (b, h, n), into a f32 [N,H,B] buffer;
//   plus the zero fill of the packed result's padding (ggmlR packing test: the
//   whole buffer is zeroed and padding stays 0).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fab.h"
#include "fab_device.cuh"
#include "fab_internal.h"

namespace fab {
namespace {

template <typename T>
struct Vec;  // 16-byte vector loads
template <>
struct Vec<float> {
  static constexpr int kElems = 4;
  static __device__ __forceinline__ float dot(const uint4& a, const uint4& b) {
    return __uint_as_float(a.x) * __uint_as_float(b.x) + __uint_as_float(a.y) * __uint_as_float(b.y) +
           __uint_as_float(a.z) * __uint_as_float(b.z) + __uint_as_float(a.w) * __uint_as_float(b.w);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  static __device__ __forceinline__ float dot2(uint32_t a, uint32_t b) {
    const float a0 = __uint_as_float(a << 16), a1 = __uint_as_float(a & 0xffff0000u);
    const float b0 = __uint_as_float(b << 16), b1 = __uint_as_float(b & 0xffff0000u);
    return a0 * b0 + a1 * b1;
  }
  static __device__ __forceinline__ float dot(const uint4& a, const uint4& b) {
    return dot2(a.x, b.x) + dot2(a.y, b.y) + dot2(a.z, b.z) + dot2(a.w, b.w);
  }
};

template <>
struct Vec<__half> {
  static constexpr int kElems = 8;
  static __device__ __forceinline__ float dot2(uint32_t a, uint32_t b) {
    const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a));
    const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b));
    return fa.x * fb.x + fa.y * fb.y;
  }
  static __device__ __forceinline__ float dot(const uint4& a, const uint4& b) {
    return dot2(a.x, b.x) + dot2(a.y, b.y) + dot2(a.z, b.z) + dot2(a.w, b.w);
  }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

struct ZeroRange {
  float* ptr;
  int64_t n;  // floats
};

template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(const T* __restrict__ d, const T* __restrict__ o,
                                                         float* __restrict__ di, int64_t rows, int DV, int64_t H,
                                                         int64_t N, int lpr, ZeroRange pa, ZeroRange pb,
                                                         ZeroRange pc) {
  // `lpr` lanes (a power of two) share one row, so a warp covers 32 / lpr rows
  const int lane = threadIdx.x & 31;
  const int sub = lane & (lpr - 1);
  const int rpw = 32 / lpr;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool vec = (DV % Vec<T>::kElems) == 0;
  const int chunks = DV / Vec<T>::kElems;
  // Four row groups per pass: all loads are issued before any is reduced, so
  // each warp keeps several 16-byte requests per lane in flight.
  constexpr int U = 4;
  for (int64_t r0 = gw * rpw; r0 < rows; r0 += (int64_t)U * warps * rpw) {
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = 0.f;
    if (vec && chunks <= lpr) {  // one 16-byte chunk per lane and row
      uint4 dv[U], ov[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t r = r0 + (int64_t)u * warps * rpw + lane / lpr;
        if (r < rows && sub < chunks) {
          dv[u] = __ldg(reinterpret_cast<const uint4*>(d + r * DV) + sub);
          ov[u] = __ldg(reinterpret_cast<const uint4*>(o + r * DV) + sub);
        } else {
          dv[u] = make_uint4(0, 0, 0, 0);
          ov[u] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = Vec<T>::dot(dv[u], ov[u]);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t r = r0 + (int64_t)u * warps * rpw + lane / lpr;
        if (r >= rows) continue;
        const T* dr = d + r * DV;
        const T* orow = o + r * DV;
        if (vec) {
          const uint4* d4 = reinterpret_cast<const uint4*>(dr);
          const uint4* o4 = reinterpret_cast<const uint4*>(orow);
          for (int c = sub; c < chunks; c += lpr) acc[u] += Vec<T>::dot(__ldg(d4 + c), __ldg(o4 + c));
        } else {
          for (int i = sub; i < DV; i += lpr) acc[u] += to_f32(dr[i]) * to_f32(orow[i]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float a = acc[u];
      for (int off = lpr >> 1; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
      // r indexes rows of the [DV,H,N,B] layout: r = (b*N + n)*H + h
      const int64_t r = r0 + (int64_t)u * warps * rpw + lane / lpr;
      if (sub == 0 && r < rows) {
        const int64_t h = r % H;
        const int64_t bn = r / H;
        const int64_t n = bn % N, b = bn / N;
        di[(b * H + h) * N + n] = a;
      }
    }
  }
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid < pa.n) pa.ptr[tid] = 0.f;
  if (tid < pb.n) pb.ptr[tid] = 0.f;
  if (tid < pc.n) pc.ptr[tid] = 0.f;
}

}  // namespace

cudaError_t launch_preprocess(const Problem& p, cudaStream_t s) {
  const int64_t rows = p.B * p.N * p.H;
  const int64_t nq = p.DK * p.N * p.H * p.B, nk = p.DK * p.M * p.Hkv * p.B, nv = p.DV * p.M * p.Hkv * p.B;
  float* base = p.packed;
  ZeroRange pa{base + nq, (int64_t)(p.off_k / 4) - nq};
  ZeroRange pb{base + p.off_k / 4 + nk, (int64_t)((p.off_v - p.off_k) / 4) - nk};
  ZeroRange pc{base + p.off_v / 4 + nv, (int64_t)((p.end - p.off_v) / 4) - nv};
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // lanes per row: enough 16-byte chunks for every lane, at most a warp
  const int elems = p.dtype == FAB_F32 ? 4 : 8;
  int lpr = 32;
  if (p.DV % elems == 0) {
    const int64_t chunks = p.DV / elems;
    lpr = 1;
    while (lpr < 32 && lpr < chunks) lpr <<= 1;
  }
  // one wave: as many blocks as the SMs hold at once (a grid of 1.6 waves
  // left the last 0.6 of them running alone), fewer for a small problem
  int per_sm = 0;
  cudaError_t oe;
  if (p.dtype == FAB_BF16)
    oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, preprocess_kernel<__nv_bfloat16>, 256, 0);
  else if (p.dtype == FAB_F16)
    oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, preprocess_kernel<__half>, 256, 0);
  else
    oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, preprocess_kernel<float>, 256, 0);
  if (oe != cudaSuccess || per_sm < 1) per_sm = 1;
  int64_t blocks = (rows * lpr / 32 + 7) / 8 + 1;
  const int64_t cap = (int64_t)sms * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (p.dtype == FAB_BF16) {
    preprocess_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(p.d), static_cast<const __nv_bfloat16*>(p.o), p.di, rows, (int)p.DV, p.H,
        p.N, lpr, pa, pb, pc);
  } else if (p.dtype == FAB_F16) {
    preprocess_kernel<__half><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __half*>(p.d),
                                                               static_cast<const __half*>(p.o), p.di, rows, (int)p.DV,
                                                               p.H, p.N, lpr, pa, pb, pc);
  } else {
    preprocess_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const float*>(p.d),
                                                              static_cast<const float*>(p.o), p.di, rows, (int)p.DV,
                                                              p.H, p.N, lpr, pa, pb, pc);
  }
  return cudaPeekAtLastError();
}

namespace {

// One block per 128 x 128 (query tile, key tile) of the mask: does it hold an
// entry other than -inf (f16 0xfc00)?  Entries outside the matrix do not
// count.  Thread t reads 64 keys of row t / 2.  Every tile's byte is written
// in both maps, so nothing has to be cleared first.
__global__ void __launch_bounds__(256) mask_live_kernel(const uint16_t* __restrict__ mask, int64_t N, int64_t M,
                                                          uint8_t* kt_live, uint8_t* qt_live) {
  const int kt = (int)blockIdx.x, qt = (int)blockIdx.y;
  const int64_t k_tiles = gridDim.x, q_tiles = gridDim.y;
  const int64_t n = (int64_t)qt * 128 + (threadIdx.x >> 1);
  const int64_t mb = (int64_t)kt * 128 + (threadIdx.x & 1) * 64;
  bool live = false;
  if (n < N) {
    const uint16_t* row = mask + n * M;
    if ((M & 7) == 0 && mb + 64 <= M) {
      const uint4* src = reinterpret_cast<const uint4*>(row + mb);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = __ldg(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) live |= (w[i] & 0xffffu) != 0xfc00u || (w[i] >> 16) != 0xfc00u;
      }
    } else {
      for (int e = 0; e < 64 && mb + e < M; ++e) live |= __ldg(row + mb + e) != 0xfc00u;
    }
  }
  const uint8_t any = __syncthreads_or(live) ? 1 : 0;
  if (threadIdx.x == 0) {
    kt_live[qt * live_stride(k_tiles) + kt] = any;
    qt_live[kt * live_stride(q_tiles) + qt] = any;
  }
}

}  // namespace

cudaError_t launch_mask_scan(const Problem& p, cudaStream_t s) {
  const int64_t q_tiles = (p.N + 127) / 128, k_tiles = (p.M + 127) / 128;
  mask_live_kernel<<<dim3((unsigned)k_tiles, (unsigned)q_tiles), 256, 0, s>>>(p.mask, p.N, p.M, p.kt_live,
                                                                              p.qt_live);
  return cudaPeekAtLastError();
}

}  // namespace fab
