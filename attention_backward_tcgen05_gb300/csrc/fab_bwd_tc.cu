// fab_bwd_tc.cu -- the key/value pass of the attention backward on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory,
// operands staged by TMA in 128-byte-swizzled shared memory).  bf16 inputs,
// D = DK = DV in {64, 128}, f32 accumulation; writes the dK and dV slices of
// the packed f32 result.  The query pass (fab_dq_tc.cu) writes dQ.
//
// Math (labml "Flash Attention", "Backward pass"; ggmlR attn_ref for the mask
// and scale): with S = scale * Q K^T + mask, P = exp(S - LSE) (the saved row
// log-sum-exp), dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dQ = scale dS K,
// dK = scale dS^T Q.  D_i = dO_i . O_i comes from the preprocess kernel.
//
// Decomposition: one CTA per (key tile of BM = 128 keys, key/value head,
// batch).  The key/value tile stays in shared memory; the CTA walks every
// query head of the GQA group and every query tile of BQ = 64 queries
// (skipping tiles a top-left causal mask empties), so dK and dV of the group
// accumulate in tensor memory without atomics.
//
// Per query tile, all in the transposed ("key rows") orientation so that one
// thread owns one key row of every tensor-memory tile:
//   S^T  = K  Q^T     [BM x BQ]  A = K (smem, K-major),  B = Q (smem, K-major)
//   dP^T = V  dO^T    [BM x BQ]  A = V,                  B = dO
//   P^T  = exp2(S^T * scale*log2e + mask*log2e - LSE*log2e)  -> bf16, tmem
//          (written over the S^T columns it came from; the dV/dK products
//          address the two 32-query halves separately)
//   dV  += P^T dO     [BM x D]   A = P^T (tmem),         B = dO (smem, MN-major)
//   dS^T = P^T * (dP^T - D)      -> bf16, smem (128-byte swizzled, key rows)
//   dK  += dS^T Q     [BM x D]   A = dS^T (smem, K-major), B = Q (smem, MN-major)
//
// Warp roles (320 threads): warp 0 loads tiles with TMA (and the tile's LSE
// and D rows); warp 1 allocates tensor memory and one lane issues every MMA;
// warps 2-9 turn S and dP into P and dS (thread = key row; two warps share
// each tensor-memory lane quarter and split the BQ query columns) and write
// dK and dV at the end.  All hand-offs are mbarriers; every wait is bounded
// (see fab_device.cuh).
//
// Issue order per query tile i: dV(i) | dP^T(i+1), dK(i) | S^T(i+2).
// S^T has two tensor-memory buffers, so scores run two tiles ahead of the
// softmax warps; dP^T(i+1) is issued as soon as the softmax warps have read
// dP^T(i) (dS lives in shared memory, so no product reads the dP^T columns).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fab.h"
#include "fab_device.cuh"
#include "fab_internal.h"

namespace fab {
namespace {

__device__ uint32_t g_err_tc;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;

template <int D>
struct Cfg {
  static constexpr int BM = 128;  // keys per CTA (tensor-memory lanes)
  static constexpr int BQ = 64;   // queries per step
  static constexpr int STAGES = 4;
  static constexpr int ATOMS = D / 64;  // 128-byte swizzle atoms along D
  static constexpr uint32_t KV_ATOM = BM * 128;  // bytes of one atom column of a K/V tile
  static constexpr uint32_t Q_ATOM = BQ * 128;   // bytes of one atom column of a Q/dO tile
  static constexpr uint32_t DS_BYTES = BM * BQ * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + ATOMS * KV_ATOM;
  static constexpr uint32_t OFF_Q = OFF_V + ATOMS * KV_ATOM;
  static constexpr uint32_t OFF_DO = OFF_Q + STAGES * ATOMS * Q_ATOM;
  static constexpr uint32_t OFF_DS = OFF_DO + STAGES * ATOMS * Q_ATOM;
  static constexpr uint32_t OFF_LD = OFF_DS + 2 * DS_BYTES;  // per stage: lse2[BQ], D[BQ]
  static constexpr uint32_t OFF_BAR = OFF_LD + STAGES * 2 * BQ * 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
  static constexpr uint32_t SMEM = OFF_MISC + 64;
  // tensor-memory columns
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 64, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, BQ, false, false);
  static constexpr uint32_t ID_DVK = idesc_bf16(128, D, false, true);
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TM_DK + D <= TM_COLS, "tensor memory budget");
  static_assert(STAGES <= 4, "barrier slots hold up to four stages");
};

// barrier slots
enum : int {
  B_KV = 0,
  B_FULL = 1,   // + stage (up to 4)
  B_EMPTY = 5,  // + stage (up to 4)
  B_S = 9,      // + S buffer
  B_DP = 11,
  B_P = 12,     // + S buffer: per buffer, so warps one tile ahead cannot complete a phase early
  B_DS = 14,
  B_DV = 15,
  B_DK = 16,
  B_DSFREE = 17,  // + buffer
  B_FINAL = 19,
  B_COUNT = 20
};
static_assert(B_COUNT <= 32, "barrier area holds 32 slots");

struct Params {
  int64_t B, H, Hkv, N, M;
  float scale;
  int causal;
  const float* lse;
  const float* di;
  const uint16_t* mask;
  float* dk;
  float* dv;
  int kv_tiles;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023u) {  // swizzled tiles need a 1024-byte-aligned base
    if (threadIdx.x == 0) atomicOr(&g_err_tc, kErrSmemAlign);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 4);
  float* ld_smem = reinterpret_cast<float*>(smem + C::OFF_LD);

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();

  // tile coordinates: heavy (low) key tiles first so a causal grid drains evenly
  const int64_t units = p.Hkv * p.B;
  const int64_t j = blockIdx.x / units;
  const int64_t rem = blockIdx.x % units;
  const int64_t b = rem / p.Hkv, hkv = rem % p.Hkv;
  const int64_t m0 = j * C::BM;
  const int64_t rk2 = p.H / p.Hkv;
  const int64_t q_tiles = (p.N + C::BQ - 1) / C::BQ;
  int64_t qt0 = p.causal ? m0 / C::BQ : 0;
  if (qt0 > q_tiles) qt0 = q_tiles;
  const int64_t nqt = q_tiles - qt0;
  const int n_it = (int)(rk2 * nqt);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(B_FULL + s), 32);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    mbar_init(bar(B_S + 0), 1);
    mbar_init(bar(B_S + 1), 1);
    mbar_init(bar(B_DP), 1);
    mbar_init(bar(B_P + 0), kSoftmaxThreads);
    mbar_init(bar(B_P + 1), kSoftmaxThreads);
    mbar_init(bar(B_DS), kSoftmaxThreads);
    mbar_init(bar(B_DV), 1);
    mbar_init(bar(B_DK), 1);
    mbar_init(bar(B_DSFREE + 0), 1);
    mbar_init(bar(B_DSFREE + 1), 1);
    mbar_init(bar(B_FINAL), 1);
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
  uint32_t* err = &g_err_tc;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    if (n_it > 0) {
      if (lane == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmO);
        mbar_arrive_expect_tx(bar(B_KV), 2 * C::ATOMS * C::KV_ATOM);
        const int kvrow = (int)(b * p.Hkv + hkv);
        for (int a = 0; a < C::ATOMS; ++a) {
          tma_load_3d(sbase + C::OFF_K + a * C::KV_ATOM, &tmK, bar(B_KV), a * 64, (int)m0, kvrow);
          tma_load_3d(sbase + C::OFF_V + a * C::KV_ATOM, &tmV, bar(B_KV), a * 64, (int)m0, kvrow);
        }
      }
      for (int it = 0; it < n_it; ++it) {
        const int s = it % C::STAGES, u = it / C::STAGES;
        const bool ok = mbar_wait(bar(B_EMPTY + s), (u & 1) ^ 1, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int64_t h = hkv * rk2 + it / nqt;
        const int64_t n0 = (qt0 + it % nqt) * C::BQ;
        const int64_t rowbase = (b * p.H + h) * p.N;
        float* lds = ld_smem + s * 2 * C::BQ;
        // start the tile copies first; the LSE and D loads below overlap them
        if (lane == 0) {
          mbar_expect_tx(bar(B_FULL + s), 2 * C::ATOMS * C::Q_ATOM);
          const int qrow = (int)(b * p.H + h);
          for (int a = 0; a < C::ATOMS; ++a) {
            tma_load_3d(sbase + C::OFF_Q + (s * C::ATOMS + a) * C::Q_ATOM, &tmQ, bar(B_FULL + s), a * 64, (int)n0,
                        qrow);
            tma_load_4d(sbase + C::OFF_DO + (s * C::ATOMS + a) * C::Q_ATOM, &tmO, bar(B_FULL + s), a * 64, (int)h,
                        (int)n0, (int)b);
          }
        }
        for (int jj = lane; jj < C::BQ; jj += 32) {
          const int64_t n = n0 + jj;
          const bool in = n < p.N;
          lds[jj] = in ? p.lse[rowbase + n] * kLog2e : INFINITY;
          lds[C::BQ + jj] = in ? p.di[rowbase + n] : 0.f;
        }
        // one arrival per lane (count 32) publishes that lane's LSE/D stores
        mbar_arrive(bar(B_FULL + s));
        ++issued;
      }
      // let every load this warp started land before shared memory goes away
      if (lane == 0) {
        mbar_drain(bar(B_KV), 0);
        const int first = issued > C::STAGES ? issued - C::STAGES : 0;
        for (int it = first; it < issued; ++it) mbar_drain(bar(B_FULL + it % C::STAGES), (it / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this loop (descriptors stay warp-uniform); lane 0
    // issues the MMAs and commits
    if (n_it > 0) {
      const uint32_t issue = lane == 0 ? 1u : 0u;
      auto wall = [&](int i, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, err));
      };
      // Descriptors are built once; a K step only moves the start address,
      // whose 14-bit field (address >> 4, all addresses < 232 KB) never carries
      // into the neighbouring fields, so a step is one add.
      auto adv = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
      const uint64_t dK_km = sdesc_sw128(sbase + C::OFF_K, 16, 1024);               // K, K-major
      const uint64_t dV_km = sdesc_sw128(sbase + C::OFF_V, 16, 1024);               // V, K-major
      const uint64_t dQ_km = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);               // stage 0 Q, K-major
      const uint64_t dQ_mn = sdesc_sw128(sbase + C::OFF_Q, C::Q_ATOM, 1024);        // stage 0 Q, MN-major
      const uint64_t dO_km = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);
      const uint64_t dO_mn = sdesc_sw128(sbase + C::OFF_DO, C::Q_ATOM, 1024);
      const uint64_t dS_km = sdesc_sw128(sbase + C::OFF_DS, 16, 1024);              // dS^T buffer 0, K-major
      auto stage_off = [](int it) { return (uint32_t)((it % C::STAGES) * C::ATOMS * C::Q_ATOM); };
      auto s_buf = [&](int it) { return (it & 1) ? C::TM_S1 : C::TM_S0; };
      // packed bf16 P columns: queries 0-31 at +0..15, queries 32-63 at +32..47
      auto a_col = [](int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); };
      // byte offset of K step kk inside a K-major tile whose atom columns are `atom` bytes apart
      auto kstep = [](int kk, uint32_t atom) { return (uint32_t)((kk >> 2) * atom + (kk & 3) * 32); };
      // S^T(it) = K Q^T into its buffer
      auto issue_s = [&](int it) {
        const uint64_t q = adv(dQ_km, stage_off(it));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tm + s_buf(it), adv(dK_km, kstep(kk, C::KV_ATOM)), adv(q, kstep(kk, C::Q_ATOM)), C::ID_S, kk > 0, issue);
        mma_commit(bar(B_S + (it & 1)), issue);
      };
      // dP^T(it) = V dO^T
      auto issue_dp = [&](int it) {
        const uint64_t o = adv(dO_km, stage_off(it));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tm + C::TM_DP, adv(dV_km, kstep(kk, C::KV_ATOM)), adv(o, kstep(kk, C::Q_ATOM)), C::ID_S, kk > 0, issue);
        mma_commit(bar(B_DP), issue);
      };
      // prologue: S^T(0), dP^T(0), S^T(1)
      bool ok = wall(B_KV, 0) && wall(B_FULL, 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
        if (n_it > 1 && (ok = wall(B_FULL + 1, 0))) {
          tc_fence_after();
          issue_s(1);
        }
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % C::STAGES;
        const uint64_t o_mn = adv(dO_mn, stage_off(it)), q_mn = adv(dQ_mn, stage_off(it));
        const uint64_t ds_km = adv(dS_km, (it & 1) * C::DS_BYTES);
        // dV += P^T dO, P^T from this tile's score buffer
        if (!(ok = wall(B_P + (it & 1), (it >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          mma_ts(tm + C::TM_DV, tm + s_buf(it) + a_col(kk), adv(o_mn, kk * 2048), C::ID_DVK, (it > 0 || kk > 0) ? 1u : 0u, issue);
        mma_commit(bar(B_DV), issue);
        // dS^T(it) is in shared memory and dP^T(it) has been read: the next
        // tile's dP^T goes first so its dS work overlaps dK(it)
        if (!(ok = wall(B_DS, it & 1))) break;
        tc_fence_after();
        if (it + 1 < n_it) issue_dp(it + 1);
        // dK += dS^T Q, both from shared memory (dS^T K-major, Q MN-major)
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          mma_ss(tm + C::TM_DK, adv(ds_km, kk * 32), adv(q_mn, kk * 2048), C::ID_DVK, (it > 0 || kk > 0) ? 1u : 0u, issue);
        mma_commit(bar(B_EMPTY + s), issue);
        mma_commit(bar(B_DSFREE + (it & 1)), issue);
        if (it + 2 < n_it) {
          // S^T(it+2) overwrites P(it) in the same buffer: dV(it) must have read it
          if (!(ok = wall(B_FULL + (it + 2) % C::STAGES, ((it + 2) / C::STAGES) & 1)))
            break;
          if (!(ok = wall(B_DV, it & 1))) break;
          tc_fence_after();
          issue_s(it + 2);
        }
      }
      // every MMA issued above must finish before tensor memory is released
      mma_commit(bar(B_FINAL), issue);
      mbar_drain(bar(B_FINAL), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax / dS
    // warps 2-5 take query columns 0-31 of the tile, warps 6-9 columns 32-63
    const int hf = (warp - 2) >> 2;
    const int r = (warp & 3) * 32 + lane;  // key row within the tile
    const int64_t m = m0 + r;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c1 = p.scale * kLog2e;
    // masking only where the tile needs it: keys past M, or keys past some
    // query of the tile under the causal mask
    const bool tail_keys = m0 + C::BM > p.M;
    // additive mask: this thread's 32 values (its key row, its 32 query
    // columns) for the next tile are loaded one tile ahead, as f16 pairs, so
    // the L2 latency stays off the P computation.  Entries outside the matrix
    // read as 0; those rows or keys are masked through LSE = +inf or the key
    // bound anyway.
    const bool has_mask = p.mask != nullptr;
    const bool key_in = m < p.M;
    const uint16_t* mrow = p.mask + (key_in ? m : 0);
    uint32_t mk[16];
    auto load_mask = [&](int itx) {
      const int64_t nbx = (qt0 + itx % nqt) * C::BQ + hf * 32;
      const uint16_t* src = mrow + p.M * nbx;  // walks down the query rows
      if (key_in && nbx + 32 <= p.N) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t lo = __ldg(src);
          src += p.M;
          const uint32_t hi = __ldg(src);
          src += p.M;
          mk[c] = lo | (hi << 16);
        }
      } else {  // key past M or a ragged last query tile
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const bool in0 = key_in && nbx + 2 * c < p.N, in1 = key_in && nbx + 2 * c + 1 < p.N;
          const uint32_t lo = in0 ? __ldg(src) : 0u;
          src += p.M;
          const uint32_t hi = in1 ? __ldg(src) : 0u;
          src += p.M;
          mk[c] = lo | (hi << 16);
        }
      }
    };
    if (has_mask && n_it > 0) load_mask(0);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % C::STAGES, u = it / C::STAGES;
      const int64_t nb = (qt0 + it % nqt) * C::BQ + hf * 32;  // first query of this thread's columns
      ok = mbar_wait(bar(B_FULL + s), u & 1, abort_flag, err);
      ok = ok && mbar_wait(bar(B_S + (it & 1)), (it >> 1) & 1, abort_flag, err);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const float4* lse4 = reinterpret_cast<const float4*>(ld_smem + s * 2 * C::BQ + hf * 32);
      const float4* di4 = reinterpret_cast<const float4*>(ld_smem + s * 2 * C::BQ + C::BQ + hf * 32);
      const uint32_t sb = (it & 1) ? C::TM_S1 : C::TM_S0;
      uint32_t ra[32];
      tmem_ld32(tm + lane_off + sb + hf * 32, ra);
      tmem_ld_wait(ra);
      const bool need_causal = p.causal && (m0 + C::BM - 1 > nb);
      float pv[32];
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 l4 = lse4[q4];
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jj = q4 * 4 + e;
          float x = fmaf(__uint_as_float(ra[jj]), c1, -lv[e]);
          if (has_mask) {
            const uint32_t hbits = (jj & 1) ? (mk[jj >> 1] >> 16) : (mk[jj >> 1] & 0xffffu);
            x = fmaf(__half2float(__ushort_as_half((unsigned short)hbits)), kLog2e, x);
          }
          if (need_causal && m > nb + jj) x = -INFINITY;
          if (tail_keys && m >= p.M) x = -INFINITY;
          pv[jj] = ex2_approx(x);
        }
      }
      if (has_mask && it + 1 < n_it) load_mask(it + 1);
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
      // packed P goes over the first 16 of this warp's own 32 S columns: the
      // other warp of the lane quarter may still be reading its S columns
      tmem_st16(tm + lane_off + sb + hf * 32, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_P + (it & 1)));

      ok = mbar_wait(bar(B_DP), it & 1, abort_flag, err);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      tmem_ld32(tm + lane_off + C::TM_DP + hf * 32, ra);
      tmem_ld_wait(ra);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 d4 = di4[q4];
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jj = q4 * 4 + e;
          pv[jj] = pv[jj] * (__uint_as_float(ra[jj]) - dv[e]);
        }
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
      if (it >= 2) {
        ok = mbar_wait(bar(B_DSFREE + (it & 1)), ((it >> 1) - 1) & 1, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      // dS^T row r into the swizzled [BM x BQ] bf16 tile (16-byte chunk c of
      // row r lives at chunk c ^ (r % 8)); this thread owns chunks 4hf..4hf+3
      const uint32_t rowaddr = sbase + C::OFF_DS + (it & 1) * C::DS_BYTES + r * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(rowaddr + (((hf * 4 + c) ^ (r & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();  // the dP^T reads above are done before dP^T(it+1) may overwrite them
      mbar_arrive(bar(B_DS));
    }
    // epilogue: dV and dK (scaled) rows of this key tile, half of the
    // columns per warp.  The tensor-memory loads are warp collectives, so
    // every lane runs them and only the stores are per row.
    const bool row_ok = m < p.M;
    const int64_t row = (b * p.Hkv + hkv) * p.M + (row_ok ? m : 0);
    float* dst_v = p.dv + row * D + hf * (D / 2);
    float* dst_k = p.dk + row * D + hf * (D / 2);
    if (n_it == 0) {
      if (row_ok)
        for (int c = 0; c < D / 2; c += 4) {
          *reinterpret_cast<float4*>(dst_v + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(dst_k + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else {
      const bool done = mbar_wait(bar(B_FINAL), 0, abort_flag, err);
      if (__all_sync(0xffffffffu, done && !*abort_flag)) {
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          uint32_t rv[32], rk[32];
          tmem_ld32(tm + lane_off + C::TM_DV + hf * (D / 2) + c0, rv);
          tmem_ld32(tm + lane_off + C::TM_DK + hf * (D / 2) + c0, rk);
          tmem_ld_wait2(rv, rk);
          if (row_ok) {
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              *reinterpret_cast<float4*>(dst_v + c0 + c) =
                  make_float4(__uint_as_float(rv[c]), __uint_as_float(rv[c + 1]), __uint_as_float(rv[c + 2]),
                              __uint_as_float(rv[c + 3]));
              *reinterpret_cast<float4*>(dst_k + c0 + c) =
                  make_float4(p.scale * __uint_as_float(rk[c]), p.scale * __uint_as_float(rk[c + 1]),
                              p.scale * __uint_as_float(rk[c + 2]), p.scale * __uint_as_float(rk[c + 3]));
            }
          }
        }
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

bool make_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const Problem& pr, cudaStream_t s) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv, mo;
  const cuuint64_t e = 2;  // bytes per bf16
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.N, (cuuint64_t)(pr.H * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.N * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mq, pr.q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.M, (cuuint64_t)(pr.Hkv * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.M * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BM, 1};
    if (!make_map(&mk, pr.k, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!make_map(&mv, pr.v, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // d [DV,H,N,B]: rows n of one head are H*DV elements apart
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)pr.H, (cuuint64_t)pr.N, (cuuint64_t)pr.B};
    const cuuint64_t str[3] = {D * e, (cuuint64_t)pr.H * D * e, (cuuint64_t)pr.N * pr.H * D * e};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mo, pr.d, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  Params p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.N = pr.N;
  p.M = pr.M;
  p.scale = pr.scale;
  p.causal = pr.causal;
  p.lse = pr.lse;
  p.di = pr.di;
  p.mask = pr.mask;
  p.dk = pr.packed + pr.off_k / 4;
  p.dv = pr.packed + pr.off_v / 4;
  p.kv_tiles = (int)((pr.M + C::BM - 1) / C::BM);
  const int64_t grid = (int64_t)p.kv_tiles * pr.Hkv * pr.B;
  cudaError_t err = cudaFuncSetAttribute(bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  bwd_tc_kernel<D><<<(unsigned)grid, kThreads, C::SMEM, s>>>(mq, mk, mv, mo, p);
  return cudaPeekAtLastError();
}

}  // namespace

bool backward_tc_supported(const Problem& p) {
  if (p.dtype != FAB_BF16 || p.DK != p.DV) return false;
  if (p.DK != 64 && p.DK != 128) return false;
  // TMA coordinates are 32-bit; grid.x must fit as well
  if (p.N >= (1ll << 31) || p.M >= (1ll << 31) || p.H * p.B >= (1ll << 31)) return false;
  if (((p.N + 127) / 128) * p.H * p.B >= (1ll << 31)) return false;  // query-pass grid
  return true;
}

cudaError_t launch_backward_tc(const Problem& p, cudaStream_t s) {
  return p.DK == 128 ? launch_d<128>(p, s) : launch_d<64>(p, s);
}

uint32_t take_error_tc() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err_tc, &z, sizeof(z));
  return v;
}

}  // namespace fab
