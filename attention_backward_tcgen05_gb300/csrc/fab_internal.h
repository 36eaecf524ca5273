// fab_internal.h -- declarations shared by the host layer and the kernel
// translation units of libfab.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fab {

// Error bits a kernel may OR into its translation unit's device error word.
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrSmemAlign = 2u;  // dynamic shared memory not 1024-byte aligned

// One validated call, in the units the kernels use.
struct Problem {
  int64_t B, H, Hkv, N, M, DK, DV;
  float scale;
  int causal;
  int dtype;  // FAB_F32, FAB_BF16 or FAB_F16
  const void* q;
  const void* k;
  const void* v;
  const void* d;  // upstream gradient, [DV,H,N,B]
  const void* o;  // forward output, [DV,H,N,B]
  const float* lse;
  const uint16_t* mask;  // f16 [M,N] or null
  float* di;             // workspace: D_i, f32 [N,H,B]
  // workspace, only with a mask: one byte per 128 x 128 tile of the mask,
  // nonzero when the tile holds an entry other than -inf, stored twice:
  // kt_live has a row per query tile over the key tiles, qt_live (right
  // after it) a row per key tile over the query tiles, each row
  // live_stride(tiles) bytes.  A pass skips the tiles before the first and
  // after the last live tile of its row.  Null: no skipping.
  uint8_t* kt_live;
  uint8_t* qt_live;
  float* packed;         // packed f32 result
  size_t off_k, off_v, end;  // bytes
};

// fab_preprocess.cu: D_i = rowsum(dO * O) into p.di; zero the padding of the
// packed result.
cudaError_t launch_preprocess(const Problem& p, cudaStream_t s);

// Bytes per row of a live-tile map over `tiles` tiles: padded to 16 so that
// rows can be read in 16-byte pieces.
__host__ __device__ inline int64_t live_stride(int64_t tiles) { return (tiles + 15) / 16 * 16; }

// fab_preprocess.cu: p.kt_live and p.qt_live from the mask (both non-null).
cudaError_t launch_mask_scan(const Problem& p, cudaStream_t s);

// fab_simt.cu: CUDA-core kernels for every dtype and width (DK, DV <= 256).
cudaError_t launch_forward_simt(const Problem& p, void* o, float* lse, cudaStream_t s);
cudaError_t launch_backward_simt(const Problem& p, cudaStream_t s);

// fab_fwd_tc.cu: the tcgen05 tensor-core forward with LSE (bf16 or f16, DK == DV in {64, 128}).
bool forward_tc_supported(const Problem& p);
cudaError_t launch_forward_tc(const Problem& p, void* o, float* lse, cudaStream_t s);

// fab_bwd_tc.cu: the tcgen05 tensor-core backward's key/value pass (dK, dV;
// bf16 or f16, DK == DV in {64, 128}).
bool backward_tc_supported(const Problem& p);
cudaError_t launch_backward_tc(const Problem& p, cudaStream_t s);

// fab_dq_tc.cu: the tcgen05 tensor-core backward's query pass (dQ), same
// problems as launch_backward_tc.  With fuse_d it also computes D_i from p.o
// into p.di and zeroes the packed result's padding (the preprocess's work);
// otherwise it reads D_i from p.di.
cudaError_t launch_dq_tc(const Problem& p, bool fuse_d, cudaStream_t s);

// fab_host.cu: cuTensorMapEncodeTiled from the driver, looked up once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Each kernel translation unit keeps a device error word; these read and
// clear it (host side, synchronous).
uint32_t take_error_tc();
uint32_t take_error_dq();
uint32_t take_error_fwd();

}  // namespace fab
