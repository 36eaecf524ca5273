// fab_fwd_tc.cu -- attention forward with the row log-sum-exp, on tcgen05.
// bf16 inputs, D = DK = DV in {64, 128}, f32 accumulation; writes O in bf16
// ([DV,H,N,B]) and LSE in f32 ([N,H,B], natural log, +inf for a row with no
// finite score).
//
// Math: labml "Flash Attention", "Forward pass" (S = scale Q K^T, P = e^S / L,
// O = P V) with the online softmax of "Flash Attention Optimization" (running
// max m, sum l, unnormalised O, per key block); ggmlR attn_ref for the
// additive mask (added after scaling) and for rows with no finite score.
//
// One CTA per (query tile of 128 rows, query head, batch).  Q stays in shared
// memory; key/value tiles of 128 keys stream through a two-stage TMA ring.
// S = Q K_j^T lands in one of two tensor-memory buffers, so the MMA for tile
// j+1 runs while the softmax warps turn tile j into P (bf16, written back over
// S) and the tensor core then accumulates O += P V_j in tensor memory.  The
// running max is only raised when a tile's max exceeds it by more than 8 (in
// log2 units); P is then bounded by 2^8 and O is rescaled in tensor memory
// only on those rare updates.  Using a stale max is exact: O and l share it.
//
// Warps: 0 = TMA producer, 1 = tensor-memory allocator and MMA issuer,
// 2-5 = softmax, rescale and epilogue (thread = query row).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fab.h"
#include "fab_device.cuh"
#include "fab_internal.h"

namespace fab {
namespace {

__device__ uint32_t g_err_fwd;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kThreads = 192;

template <int D>
struct FCfg {
  static constexpr int BQ = 128;  // queries per CTA (tensor-memory lanes)
  static constexpr int BK = 128;  // keys per tile
  static constexpr int STAGES = 2;
  static constexpr int ATOMS = D / 64;
  static constexpr uint32_t ATOM = 128 * 128;  // one 128-row x 128-byte swizzle atom column
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + ATOMS * ATOM;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * ATOMS * ATOM;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * ATOMS * ATOM;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 16 * 8;
  // at least 116 KB so one CTA owns an SM and its whole tensor memory
  static constexpr uint32_t SMEM_USED = OFF_MISC + 64 + 1024;
  static constexpr uint32_t SMEM = SMEM_USED > 118784 ? SMEM_USED : 118784;
  static constexpr uint32_t TM_S = 0;  // + 128 * buffer
  static constexpr uint32_t TM_O = 256;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, BK, false, false);
  static constexpr uint32_t ID_PV = idesc_bf16(128, D, false, true);
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum : int {
  F_Q = 0,
  F_FULL = 1,    // + stage
  F_EMPTY = 3,   // + stage
  F_S = 5,       // + buffer
  F_P = 7,       // + buffer
  F_PV = 9,      // + buffer
  F_FINAL = 11,
};

struct FParams {
  int64_t B, H, Hkv, N, M;
  float scale;
  int causal;
  const uint16_t* mask;
  __nv_bfloat16* o;
  float* lse;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FParams p) {
  using C = FCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 4);
  uint32_t* err = &g_err_fwd;

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();

  const int64_t q_tiles = (p.N + C::BQ - 1) / C::BQ;
  const int64_t qt = blockIdx.x % q_tiles;
  const int64_t bh = blockIdx.x / q_tiles;
  const int64_t h = bh % p.H, b = bh / p.H;
  const int64_t hkv = h / (p.H / p.Hkv);
  const int64_t n0 = qt * C::BQ;
  int64_t n_kv = (p.M + C::BK - 1) / C::BK;
  if (p.causal) {
    const int64_t last = (n0 + C::BQ - 1) / C::BK + 1;  // key tiles holding some m <= n
    if (last < n_kv) n_kv = last;
  }
  const int nkv = (int)n_kv;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar(F_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(F_FULL + s), 1);
      mbar_init(bar(F_EMPTY + s), 1);
      mbar_init(bar(F_S + s), 1);
      mbar_init(bar(F_P + s), 128);
      mbar_init(bar(F_PV + s), 1);
    }
    mbar_init(bar(F_FINAL), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_arrive_expect_tx(bar(F_Q), C::ATOMS * C::ATOM);
      for (int a = 0; a < C::ATOMS; ++a)
        tma_load_3d(sbase + C::OFF_Q + a * C::ATOM, &tmQ, bar(F_Q), a * 64, (int)n0, (int)(b * p.H + h));
      int issued = 0;
      const int kvrow = (int)(b * p.Hkv + hkv);
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(bar(F_EMPTY + s), ((j >> 1) & 1) ^ 1, abort_flag, err)) break;
        mbar_arrive_expect_tx(bar(F_FULL + s), 2 * C::ATOMS * C::ATOM);
        for (int a = 0; a < C::ATOMS; ++a) {
          tma_load_3d(sbase + C::OFF_K + (s * C::ATOMS + a) * C::ATOM, &tmK, bar(F_FULL + s), a * 64,
                      j * C::BK, kvrow);
          tma_load_3d(sbase + C::OFF_V + (s * C::ATOMS + a) * C::ATOM, &tmV, bar(F_FULL + s), a * 64,
                      j * C::BK, kvrow);
        }
        ++issued;
      }
      mbar_drain(bar(F_Q), 0);
      for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j) mbar_drain(bar(F_FULL + (j & 1)), (j >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this loop (descriptors stay warp-uniform); lane 0
    // issues the MMAs and commits
    {
      const uint32_t issue = lane == 0 ? 1u : 0u;
      auto wall = [&](int i, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, err));
      };
      const uint32_t sQ = sbase + C::OFF_Q;
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!wall(F_FULL + s, (j >> 1) & 1)) return false;
        // P(j-2) in this tensor-memory buffer must have been consumed
        if (j >= 2 && !wall(F_PV + s, ((j >> 1) - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sK = sbase + C::OFF_K + s * C::ATOMS * C::ATOM;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::ATOM + (kk & 3) * 32;
          mma_ss(tm + C::TM_S + s * 128, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), C::ID_S,
                 kk > 0, issue);
        }
        mma_commit(bar(F_S + s), issue);
        return true;
      };
      bool ok = wall(F_Q, 0) && issue_s(0);
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j & 1;
        if (j + 1 < nkv && !(ok = issue_s(j + 1))) break;
        if (!(ok = wall(F_P + s, (j >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t sV = sbase + C::OFF_V + s * C::ATOMS * C::ATOM;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)
          mma_ts(tm + C::TM_O, tm + C::TM_S + s * 128 + kk * 8, sdesc_sw128(sV + kk * 2048, C::ATOM, 1024), C::ID_PV,
                 (j > 0 || kk > 0) ? 1u : 0u, issue);
        mma_commit(bar(F_PV + s), issue);
        mma_commit(bar(F_EMPTY + s), issue);
      }
      mma_commit(bar(F_FINAL), issue);
      mbar_drain(bar(F_FINAL), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = (warp & 3) * 32 + lane;
    const int64_t n = n0 + r;
    const bool row_ok = n < p.N;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c1 = p.scale * kLog2e;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int s = j & 1;
      const int64_t m0 = (int64_t)j * C::BK;
      ok = mbar_wait(bar(F_S + s), (j >> 1) & 1, abort_flag, err);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t tS = tm + lane_off + C::TM_S + s * 128;
      // pass 1: the tile's row max (masked entries excluded)
      float tmax = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t ra[32];
        tmem_ld32(tS + c * 32, ra);
        tmem_ld_wait(ra);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int64_t m = m0 + c * 32 + e;
          float x = __uint_as_float(ra[e]) * c1;
          if (p.mask != nullptr && row_ok && m < p.M)
            x = fmaf(__half2float(__ushort_as_half(p.mask[m + p.M * n])), kLog2e, x);
          if ((p.causal && m > n) || m >= p.M || !row_ok) x = -INFINITY;
          tmax = fmaxf(tmax, x);
        }
      }
      float m_new = m_run, alpha = 1.f;
      if (tmax > m_run + kRescaleThreshold || (m_run == -INFINITY && tmax > -INFINITY)) {
        m_new = tmax;
        alpha = exp2f(m_run - m_new);  // 0 when m_run = -inf
      }
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // pass 2: P = exp2(x - m), packed bf16 over the consumed S columns
      float rsum = 0.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t ra[32];
        tmem_ld32(tS + c * 32, ra);
        tmem_ld_wait(ra);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pe[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int64_t m = m0 + c * 32 + e + t;
            float x = __uint_as_float(ra[e + t]) * c1;
            if (p.mask != nullptr && row_ok && m < p.M)
              x = fmaf(__half2float(__ushort_as_half(p.mask[m + p.M * n])), kLog2e, x);
            if ((p.causal && m > n) || m >= p.M || !row_ok) x = -INFINITY;
            pe[t] = ex2_approx(x - m_use);
          }
          const uint32_t packed = pack_bf16x2(pe[0], pe[1]);
          // sum what the tensor core will see (the bf16-rounded P)
          rsum += __uint_as_float(packed << 16) + __uint_as_float(packed & 0xffff0000u);
          pk[e >> 1] = packed;
        }
        tmem_st16(tS + c * 16, pk);
      }
      l = l * alpha + rsum;
      const bool need = (m_new != m_run) && (m_run != -INFINITY) && j > 0;
      if (__any_sync(0xffffffffu, need)) {
        // O holds sum_{j' < j} P V with the old max: rescale once PV(j-1) landed
        const bool done = mbar_wait(bar(F_PV + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, err);
        if (!__all_sync(0xffffffffu, done)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = need ? alpha : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ra[32];
          tmem_ld32(tm + lane_off + C::TM_O + c0, ra);
          tmem_ld_wait(ra);
#pragma unroll
          for (int e = 0; e < 32; ++e) ra[e] = __float_as_uint(__uint_as_float(ra[e]) * f);
          tmem_st32(tm + lane_off + C::TM_O + c0, ra);
        }
      }
      m_run = m_new;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(F_P + s));
    }
    // epilogue: O / l and the LSE
    if (ok && nkv > 0) {
      const bool done = mbar_wait(bar(F_PV + ((nkv - 1) & 1)), ((nkv - 1) >> 1) & 1, abort_flag, err);
      if (__all_sync(0xffffffffu, done && !*abort_flag)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.o + ((b * p.N + (row_ok ? n : 0)) * p.H + h) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ra[32];
          tmem_ld32(tm + lane_off + C::TM_O + c0, ra);
          tmem_ld_wait(ra);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(ra[e]) * inv, __uint_as_float(ra[e + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(ra[e + 2]) * inv, __uint_as_float(ra[e + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(ra[e + 4]) * inv, __uint_as_float(ra[e + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(ra[e + 6]) * inv, __uint_as_float(ra[e + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + c0 + e) = v;
            }
          }
        }
        if (row_ok) p.lse[(b * p.H + h) * p.N + n] = l > 0.f ? (m_run + log2f(l)) * kLn2 : INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, C::TM_COLS);
  }
}

bool make_map(CUtensorMap* map, const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const Problem& pr, void* o, float* lse, cudaStream_t s) {
  using C = FCfg<D>;
  CUtensorMap mq, mk, mv;
  const cuuint64_t e = 2;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.N, (cuuint64_t)(pr.H * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.N * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mq, pr.q, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.M, (cuuint64_t)(pr.Hkv * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.M * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BK, 1};
    if (!make_map(&mk, pr.k, dims, str, box)) return cudaErrorInvalidValue;
    if (!make_map(&mv, pr.v, dims, str, box)) return cudaErrorInvalidValue;
  }
  FParams p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.N = pr.N;
  p.M = pr.M;
  p.scale = pr.scale;
  p.causal = pr.causal;
  p.mask = pr.mask;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  const int64_t grid = ((pr.N + C::BQ - 1) / C::BQ) * pr.H * pr.B;
  cudaError_t err = cudaFuncSetAttribute(fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  fwd_tc_kernel<D><<<(unsigned)grid, kThreads, C::SMEM, s>>>(mq, mk, mv, p);
  return cudaPeekAtLastError();
}

}  // namespace

bool forward_tc_supported(const Problem& p) {
  if (p.dtype != FAB_BF16 || p.DK != p.DV) return false;
  if (p.DK != 64 && p.DK != 128) return false;
  if (p.N >= (1ll << 31) || p.M >= (1ll << 31) || p.H * p.B >= (1ll << 31)) return false;
  if (((p.N + 127) / 128) * p.H * p.B >= (1ll << 31)) return false;
  return true;
}

cudaError_t launch_forward_tc(const Problem& p, void* o, float* lse, cudaStream_t s) {
  return p.DK == 128 ? launch_d<128>(p, o, lse, s) : launch_d<64>(p, o, lse, s);
}

uint32_t take_error_fwd() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err_fwd, &z, sizeof(z));
  return v;
}

}  // namespace fab
