// fab_fwd_tc.cu -- attention forward with the row log-sum-exp, on tcgen05.
// bf16 or f16 inputs (template parameter F16), D = DK = DV in {64, 128}, f32
// accumulation; writes O in the input type
// ([DV,H,N,B]) and LSE in f32 ([N,H,B], natural log, +inf for a row with no
// finite score).
//
// Math: labml "Flash Attention", "Forward pass" (S = scale Q K^T, P = e^S / L,
// O = P V) with the online softmax of "Flash Attention Optimization" (running
// max m, sum l, unnormalised O, per key block); ggmlR attn_ref for the
// additive mask (added after scaling) and for rows with no finite score.
//
// Work units of (query tile of 128 rows, query head, batch), heavy causal
// tiles first; persistent CTAs, one per SM, walk them.  A unit's Q stays in
// shared memory (the next unit's Q loads once the unit's last S MMA has read
// it); key/value tiles of 128 keys stream through a three-stage TMA ring, and
// ring stages, tensor-memory buffers and barrier phases count tiles across
// units.  S = Q K_j^T lands in one of three
// tensor-memory buffers, so the MMAs for the next tiles run while the softmax
// warps turn tile j into P (input type, written back over S) and the tensor core
// then accumulates O += P V_j in tensor memory.  The running max is only
// raised when a tile's max exceeds it by more than 8 (in log2 units); P is
// then bounded by 2^8 and O is rescaled in tensor memory only on those rare
// updates.  Using a stale max is exact: O and l share it.
//
// Warps (384 threads): 0 = TMA producer (Q, key tiles); 11 = value-tile
// producer; 1 = tensor-memory allocator and S
// issuer; 10 = PV issuer (lane 0 of an issuer warp issues); 2-9 = softmax,
// rescale and epilogue (thread = query row; two warps per tensor-memory lane
// quarter, each taking 64 of a tile's 128 keys).  Causal and key-bound tests
// run only on the tiles that have such keys.
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
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;

template <int D, bool F16 = false>
struct FCfg {
  static constexpr int BQ = 128;  // queries per CTA (tensor-memory lanes)
  static constexpr int BK = 128;  // keys per tile
  static constexpr int STAGES = 3;
  static constexpr int ATOMS = D / 64;
  static constexpr uint32_t ATOM = 128 * 128;  // one 128-row x 128-byte swizzle atom column
  static constexpr uint32_t TILE = ATOMS * ATOM;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KV = OFF_Q + TILE;  // stage s: K at + 2 s TILE, V at + (2 s + 1) TILE
  static constexpr uint32_t OFF_BAR = OFF_KV + STAGES * 2 * TILE;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
  static constexpr uint32_t OFF_MX = OFF_MISC + 64;  // [2 slots][2 halves][BQ] floats
  // the swizzled tiles need a 1024-byte-aligned base, checked at run time
  // (no room for alignment slack at D = 128); at least 116 KB so one CTA
  // owns an SM and its whole tensor memory
  // the mask's key-tile spans of a CTA's first SPAN_CAP units
  static constexpr int SPAN_CAP = 160;
  static constexpr uint32_t OFF_SPAN = OFF_MX + 2 * 2 * BQ * 4;
  static constexpr uint32_t SMEM_USED = OFF_SPAN + SPAN_CAP * 4;
  static constexpr uint32_t SMEM = SMEM_USED > 118784 ? SMEM_USED : 118784;
  static constexpr uint32_t TM_S = 0;  // + 128 * buffer, buffers 0..2
  static constexpr uint32_t TM_O = 384;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t ID_S = idesc_16(128, BK, false, false, F16);
  static constexpr uint32_t ID_PV = idesc_16(128, D, false, true, F16);
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TM_O + D <= TM_COLS, "tensor memory budget");
};

enum : int {
  F_Q = 0,       // phase k: unit k's Q landed
  F_FULL = 1,    // + g % 3: K_g landed
  F_S = 4,       // + g % 3: S(g) landed
  F_P = 7,       // + g % 3: softmax warps wrote P(g) (and rescaled O if they had to)
  F_PV = 10,     // + g % 3: PV(g) finished (its stage, S buffer free; O holds the unit's tiles <= g)
  F_FIN_S = 13,  // every S MMA finished
  F_FIN_O = 14,  // every PV MMA finished
  F_QE = 15,     // phase k: unit k's S MMAs finished (Q free)
  F_OE = 16,     // phase k: unit k's epilogue read O from tensor memory
  F_STG = 17,    // phase k: unit k's O is staged in shared memory
  F_VF = 18,     // + g % 3: V_g landed
  F_COUNT = 21
};

struct FParams {
  int64_t B, H, Hkv, N, M;
  float scale;
  int causal;
  const uint16_t* mask;
  void* o;
  float* lse;
  const uint8_t* kt_live;  // per query tile, a byte per key tile: mask not all -inf there; or null
};

template <int D, bool MASK, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmOut,
                  const FParams p) {
  using C = FCfg<D, F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023u) {  // swizzled tiles need a 1024-byte-aligned base
    if (threadIdx.x == 0) atomicOr(&g_err_fwd, kErrSmemAlign);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 4);
  float* mx = reinterpret_cast<float*>(smem + C::OFF_MX);
  // units whose staged O the bulk stores have read (the staging is the key
  // tile of the unit's last stage)
  uint32_t* o_cnt = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 8);
  uint32_t* err = &g_err_fwd;

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();

  // work units: (query tile, head, batch), heavy (late) query tiles first
  // under a causal mask.  Round k of the G CTAs takes units k G .. k G + G - 1,
  // CTA c the c-th of them on even rounds and the (G-1-c)-th on odd rounds.
  // (32-bit index arithmetic: the host guarantees units, N, M < 2^31.)
  const int q_tiles = (int)((p.N + C::BQ - 1) / C::BQ);
  const int hb = (int)(p.H * p.B);
  const int n_units = q_tiles * hb;
  const int H = (int)p.H, rk2 = (int)(p.H / p.Hkv), m_tiles = (int)((p.M + C::BK - 1) / C::BK);
  uint32_t* span_s = reinterpret_cast<uint32_t*>(smem + C::OFF_SPAN);
  const bool span_tab = MASK && p.kt_live != nullptr && m_tiles < 65536;
  const int64_t live_ks = live_stride(m_tiles);
  struct Unit {
    int h, b, hkv, n0, j0, nkv;  // key tiles j0 .. j0 + nkv - 1
  };
  auto unit_at = [&](int kk) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    return G * kk + ((kk & 1) ? G - 1 - c : c);
  };
  // the query tile of unit u
  auto tile_of = [&](int u) {
    const int qi = u / hb;
    return p.causal ? q_tiles - 1 - qi : qi;
  };
  // the live spans of this CTA's first units' query tiles, found once here
  // (made visible by the block sync below): {first live key tile, one past
  // the last} as 16-bit halves
  if (span_tab)
    for (int i = (int)threadIdx.x; i < C::SPAN_CAP && unit_at(i) < n_units; i += kThreads) {
      int s0, s1;
      live_span(p.kt_live + tile_of(unit_at(i)) * live_ks, m_tiles, s0, s1);
      span_s[i] = (uint32_t)s0 | ((uint32_t)s1 << 16);
    }
  // the unit this CTA takes in round kk
  auto unit_of = [&](int kk) {
    Unit x;
    const int u = unit_at(kk);
    const int qi = u / hb, rem = u - qi * hb;
    x.b = rem / H;
    x.h = rem - x.b * H;
    x.hkv = x.h / rk2;
    const int qt = p.causal ? q_tiles - 1 - qi : qi;
    x.n0 = qt * C::BQ;
    int j0 = 0, j1 = m_tiles;
    if (p.causal) {
      const int last = (x.n0 + C::BQ - 1) / C::BK + 1;  // key tiles holding some m <= n
      if (last < j1) j1 = last;
    }
    if (MASK && span_tab && kk < C::SPAN_CAP) {
      // key tiles before the first and after the last live one are all -inf
      // in the mask: they leave the running max, the row sum and O as they
      // are (a CTA's later rounds, if any, skip nothing)
      const uint32_t v = span_s[kk];
      const int s0 = (int)(v & 0xffffu), s1 = (int)(v >> 16);
      if (s0 > j0) j0 = s0;
      if (s1 < j1) j1 = s1;
      if (j1 <= j0) j0 = 0, j1 = 1;  // nothing live: one tile, as without skipping
    }
    x.j0 = j0;
    x.nkv = j1 - j0;  // >= 1: key tile 0 holds m = 0 <= n
    return x;
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *o_cnt = 0u;
    mbar_init(bar(F_Q), 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(bar(F_FULL + s), 1);
      mbar_init(bar(F_VF + s), 1);
      mbar_init(bar(F_S + s), 1);
      mbar_init(bar(F_P + s), kSoftmaxThreads);
      mbar_init(bar(F_PV + s), 1);
    }
    mbar_init(bar(F_FIN_S), 1);
    mbar_init(bar(F_FIN_O), 1);
    mbar_init(bar(F_QE), 1);
    mbar_init(bar(F_OE), kSoftmaxThreads);
    mbar_init(bar(F_STG), kSoftmaxThreads);
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
    // Per unit: K_g of its first tile, its Q (once the previous unit's S
    // MMAs are done with theirs), then the other tiles' keys.  K_g goes into
    // the key half of stage g % 3 once S(g-3) is done with it (the value
    // tiles have a producer warp of their own, so a key load never waits
    // behind a value tile's PV); g counts tiles across units.  A unit's
    // epilogue stages O in the key tile of its last stage G % 3, so K_{G+3}
    // also waits for that unit's bulk stores to read it.
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmOut);
      int g = 0, k = 0, issued = 0, q_issued = 0;
      int stG[3] = {-8, -8, -8}, stK[3] = {0, 0, 0};  // last tile and index of the latest units
      bool ok = true;
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const Unit x = unit_of(k);
        const int kvrow = x.b * (int)p.Hkv + x.hkv;
        for (int j = 0; j < x.nkv; ++j, ++g) {
          const int s = g % 3;
          if (g >= 3 && !(ok = mbar_wait(bar(F_S + s), ((g / 3) - 1) & 1, abort_flag, err))) break;
#pragma unroll
          for (int i = 0; i < 3; ++i)
            if (ok && stG[i] + 3 == g) ok = counter_wait(o_cnt, (uint32_t)(stK[i] + 1), abort_flag, err);
          if (!ok) break;
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar(F_FULL + s), C::TILE);
          const uint32_t sk = sbase + C::OFF_KV + 2 * s * C::TILE;
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(sk + a * C::ATOM, &tmK, bar(F_FULL + s), a * 64, (x.j0 + j) * C::BK, kvrow);
          ++issued;
          if (j == 0) {
            if (k > 0 && !(ok = mbar_wait(bar(F_QE), (k - 1) & 1, abort_flag, err))) break;
            mbar_arrive_expect_tx(bar(F_Q), C::TILE);
            for (int a = 0; a < C::ATOMS; ++a)
              tma_load_3d(sbase + C::OFF_Q + a * C::ATOM, &tmQ, bar(F_Q), a * 64, x.n0, x.b * H + x.h);
            ++q_issued;
          }
        }
        stG[k % 3] = g - 1;
        stK[k % 3] = k;
      }
      if (q_issued > 0) mbar_drain(bar(F_Q), (q_issued - 1) & 1);
      for (int j = issued > 3 ? issued - 3 : 0; j < issued; ++j) mbar_drain(bar(F_FULL + j % 3), (j / 3) & 1);
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------ value producer
    // V_g into the value half of stage g % 3 once PV(g-3) is done with it
    if (lane == 0) {
      int g = 0, k = 0, issued = 0;
      bool ok = true;
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const Unit x = unit_of(k);
        const int kvrow = x.b * (int)p.Hkv + x.hkv;
        for (int j = 0; j < x.nkv; ++j, ++g) {
          const int s = g % 3;
          if (g >= 3 && !(ok = mbar_wait(bar(F_PV + s), ((g / 3) - 1) & 1, abort_flag, err))) break;
          mbar_arrive_expect_tx(bar(F_VF + s), C::TILE);
          const uint32_t sv = sbase + C::OFF_KV + (2 * s + 1) * C::TILE;
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(sv + a * C::ATOM, &tmV, bar(F_VF + s), a * 64, (x.j0 + j) * C::BK, kvrow);
          ++issued;
        }
      }
      for (int j = issued > 3 ? issued - 3 : 0; j < issued; ++j) mbar_drain(bar(F_VF + j % 3), (j / 3) & 1);
    }
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // each issuer warp runs its loop convergently (descriptors stay
    // warp-uniform); lane 0 issues the MMAs and commits
    const uint32_t issue = lane == 0 ? 1u : 0u;
    auto wall = [&](int i, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, err));
    };
    bool ok = true;
    if (warp == 1) {
      // S(g) = Q K_g^T into buffer g % 3 once K_g landed and PV(g-3) is done
      // with the buffer's P; after a unit's last S, its Q is free.  A unit's
      // second S also waits for the previous unit's last PV, which the
      // softmax warps' epilogue waits for: issued behind the next unit's
      // first two S products, that PV came ~500 cycles later
      const uint32_t sQ = sbase + C::OFF_Q;
      int g = 0, k = 0;
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const int nkv = unit_of(k).nkv;
        if (!(ok = wall(F_Q, k & 1))) break;
        for (int j = 0; j < nkv; ++j, ++g) {
          const int s = g % 3;
          if (!(ok = wall(F_FULL + s, (g / 3) & 1))) break;
          if (g >= 3 && !(ok = wall(F_PV + s, ((g / 3) - 1) & 1))) break;
          if (j == 1 && k > 0 && !(ok = wall(F_PV + (g - 2) % 3, ((g - 2) / 3) & 1))) break;
          tc_fence_after();
          const uint32_t sK = sbase + C::OFF_KV + 2 * s * C::TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::ATOM + (kk & 3) * 32;
            mma_ss(tm + C::TM_S + s * 128, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                   C::ID_S, kk > 0, issue);
          }
          mma_commit(bar(F_S + s), issue);
        }
        mma_commit(bar(F_QE), issue);
      }
      mma_commit(bar(F_FIN_S), issue);
      mbar_drain(bar(F_FIN_S), 0);
    } else {
      // O += P(g) V_g once the softmax warps wrote P(g): packed 16-bit, key e
      // at column e / 2 of buffer g % 3; a unit's first product waits for
      // the previous unit's epilogue to have read O.  After a unit's last
      // product, once the softmax warps staged O/l, this warp writes it out
      // with bulk tensor stores and releases the staging once they read it.
      int g = 0, k = 0;
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const Unit x = unit_of(k);
        const int nkv = x.nkv;
        for (int j = 0; j < nkv; ++j, ++g) {
          const int s = g % 3;
          if (!(ok = wall(F_P + s, (g / 3) & 1))) break;
          if (!(ok = wall(F_VF + s, (g / 3) & 1))) break;
          if (j == 0 && k > 0 && !(ok = wall(F_OE, (k - 1) & 1))) break;
          tc_fence_after();
          const uint32_t sV = sbase + C::OFF_KV + (2 * s + 1) * C::TILE;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            mma_ts(tm + C::TM_O, tm + C::TM_S + s * 128 + kk * 8, sdesc_sw128(sV + kk * 2048, C::ATOM, 1024),
                   C::ID_PV, (j > 0 || kk > 0) ? 1u : 0u, issue);
          mma_commit(bar(F_PV + s), issue);
        }
        if (!ok) break;
        if (!(ok = wall(F_STG, k & 1))) break;
        if (lane == 0) {
          const uint32_t st = sbase + C::OFF_KV + 2 * ((g - 1) % 3) * C::TILE;  // key tile of the last stage
          for (int a = 0; a < C::ATOMS; ++a) tma_store_4d(&tmOut, st + a * C::ATOM, a * 64, x.h, x.n0, x.b);
          bulk_commit_group();
          bulk_wait_read_all();
          counter_bump(o_cnt);
        }
        __syncwarp();
      }
      if (lane == 0) bulk_wait_read_all();  // (every group was waited for above; kept for an early exit)
      mma_commit(bar(F_FIN_O), issue);
      mbar_drain(bar(F_FIN_O), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // warps 2-5 take keys 0-63 of a tile, warps 6-9 keys 64-127; thread =
    // query row.  The two halves of a row trade their maxima through shared
    // memory once per tile: warps w and w + 4 (the same rows) meet at named
    // barrier 1 + w % 4, OR-reducing an error flag so both leave their loop
    // at the same tile; the other pairs run on.
    const int hf = (warp - 2) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c1 = p.scale * kLog2e;
    const bool mvec = (p.M & 7) == 0;  // mask rows start 16-byte aligned
    uint32_t mk[MASK ? 32 : 1];
    bool ok = true;
    int g = 0, k = 0;
    for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
      const Unit x = unit_of(k);
      const int64_t n = (int64_t)x.n0 + r;
      const bool row_ok = n < p.N;
      const uint16_t* mrow = p.mask + p.M * (row_ok ? n : 0);
      float m_run = -INFINITY, l = 0.f;  // l: this half's share of the row sum
      for (int j = 0; j < x.nkv; ++j, ++g) {
        const int s = g % 3;
        const int64_t m0 = (int64_t)(x.j0 + j) * C::BK;
        const int64_t mb = m0 + hf * 64;  // first key of this thread's columns
        if (MASK) {
          // this thread's 64 mask values (f16 pairs); entries past M read as 0
          if (!row_ok) {
#pragma unroll
            for (int c = 0; c < 32; ++c) mk[c] = 0u;
          } else if (mvec && mb + 64 <= p.M) {
            const uint4* src = reinterpret_cast<const uint4*>(mrow + mb);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = __ldg(src + c);
              mk[4 * c] = v.x;
              mk[4 * c + 1] = v.y;
              mk[4 * c + 2] = v.z;
              mk[4 * c + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const uint32_t lo = (mb + 2 * c < p.M) ? (uint32_t)__ldg(mrow + mb + 2 * c) : 0u;
              const uint32_t hi = (mb + 2 * c + 1 < p.M) ? (uint32_t)__ldg(mrow + mb + 2 * c + 1) : 0u;
              mk[c] = lo | (hi << 16);
            }
          }
        }
        const uint32_t tS = tm + lane_off + C::TM_S + s * 128;
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar(F_S + s), (g / 3) & 1, abort_flag, err));
        float sv[64];
        float hmax = -INFINITY;
        if (got) {
          tc_fence_after();
          uint32_t ra[32], rb[32];
          tmem_ld32(tS + hf * 64, ra);
          tmem_ld32(tS + hf * 64 + 32, rb);
          tmem_ld_wait2(ra, rb);
#pragma unroll
          for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(e < 32 ? ra[e] : rb[e - 32]) * c1;
          if (MASK) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&mk[c]));
              sv[2 * c] = fmaf(mf.x, kLog2e, sv[2 * c]);
              sv[2 * c + 1] = fmaf(mf.y, kLog2e, sv[2 * c + 1]);
            }
          }
          // keys past the causal diagonal (top-left: key m > query n) or past
          // M, and rows past N; only the diagonal tile and a ragged last tile
          // (or query tile) have any
          if ((p.causal && m0 + C::BK - 1 > x.n0) || m0 + C::BK > p.M || !row_ok) {
            int64_t lim = 63;                              // last allowed column e (key mb + e)
            if (p.causal && n - mb < lim) lim = n - mb;    // m <= n
            if (p.M - 1 - mb < lim) lim = p.M - 1 - mb;    // m < M
            if (!row_ok) lim = -1;
            const int li = lim < -1 ? -1 : (int)lim;
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (e > li) sv[e] = -INFINITY;
          }
#pragma unroll
          for (int e = 0; e < 64; ++e) hmax = fmaxf(hmax, sv[e]);
        }
        mx[((g & 1) * 2 + hf) * C::BQ + r] = hmax;
        if (named_bar_or(1 + (warp & 3), 64, !(got && ok))) {
          ok = false;
          break;
        }
        // (S(g) is in registers on both halves: P may now go over its columns)
        const float tmax = fmaxf(hmax, mx[((g & 1) * 2 + (hf ^ 1)) * C::BQ + r]);
        float m_new = m_run, alpha = 1.f;
        if (tmax > m_run + kRescaleThreshold || (m_run == -INFINITY && tmax > -INFINITY)) {
          m_new = tmax;
          alpha = exp2f(m_run - m_new);  // 0 when m_run = -inf
        }
        const bool need = (m_new != m_run) && (m_run != -INFINITY) && j > 0;
        if (__any_sync(0xffffffffu, need)) {
          // O holds the unit's sum_{j' < j} P V with the old max: rescale this
          // half's columns once PV(g-1) landed
          const bool done = __all_sync(
              0xffffffffu, mbar_wait(bar(F_PV + (g - 1) % 3), ((g - 1) / 3) & 1, abort_flag, err));
          if (done) {
            tc_fence_after();
            const float f = need ? alpha : 1.f;
#pragma unroll 1
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
              uint32_t ra[32];
              tmem_ld32(tm + lane_off + C::TM_O + hf * (D / 2) + c0, ra);
              tmem_ld_wait(ra);
#pragma unroll
              for (int e = 0; e < 32; ++e) ra[e] = __float_as_uint(__uint_as_float(ra[e]) * f);
              tmem_st32(tm + lane_off + C::TM_O + hf * (D / 2) + c0, ra);
            }
          } else {
            ok = false;
          }
        }
        m_run = m_new;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        // P = exp2(x - m), packed 16-bit: key hf * 64 + e at column hf * 32 + e / 2
        float rsum = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint32_t packed = pack2<F16>(ex2_approx(sv[2 * c] - m_use), ex2_approx(sv[2 * c + 1] - m_use));
          // sum what the tensor core will see (P rounded to the input type)
          const float2 pr = unpack2<F16>(packed);
          rsum += pr.x + pr.y;
          pk[c] = packed;
        }
        tmem_st32(tS + hf * 32, pk);
        l = l * alpha + rsum;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(F_P + s));
      }
      // epilogue: O / l (this half's columns) and the LSE.  The halves' shares
      // of l meet in the last tile's shared slot: the first barrier below
      // lets both halves finish reading the maxima there, the second
      // publishes l.  Then O has been read: the next unit's first PV may
      // overwrite it.  (A warp whose wait failed reaches the first barrier
      // too, so both warps of the pair leave together.)
      const int G = g - 1;  // the unit's last tile
      const bool done =
          ok && __all_sync(0xffffffffu, mbar_wait(bar(F_PV + G % 3), (G / 3) & 1, abort_flag, err));
      if (named_bar_or(1 + (warp & 3), 64, !done || *abort_flag != 0u)) {
        ok = false;
        break;
      }
      mx[((G & 1) * 2 + hf) * C::BQ + r] = l;
      named_bar_sync(1 + (warp & 3), 64);
      tc_fence_after();
      const float lt = l + mx[((G & 1) * 2 + (hf ^ 1)) * C::BQ + r];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      // O / l in the input type, staged in the key tile of the last stage as 64-column
      // atoms of 128-byte swizzled rows (that stage's products are done; the
      // producer holds K_{G+3} until the stores have read it); the PV issuer
      // writes it out, clipping rows past N
      const uint32_t st = sbase + C::OFF_KV + 2 * (G % 3) * C::TILE;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t ra[32];
        tmem_ld32(tm + lane_off + C::TM_O + hf * (D / 2) + c0, ra);
        tmem_ld_wait(ra);
        const int col = hf * (D / 2) + c0;  // first of these 32 columns
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const int ch = ((col + e) % 64) / 8;  // 16-byte chunk within the 128-byte row
          st_shared_v4(st + (uint32_t)((col + e) / 64) * C::ATOM + r * 128 + ((ch ^ (r & 7)) << 4),
                       pack2<F16>(__uint_as_float(ra[e]) * inv, __uint_as_float(ra[e + 1]) * inv),
                       pack2<F16>(__uint_as_float(ra[e + 2]) * inv, __uint_as_float(ra[e + 3]) * inv),
                       pack2<F16>(__uint_as_float(ra[e + 4]) * inv, __uint_as_float(ra[e + 5]) * inv),
                       pack2<F16>(__uint_as_float(ra[e + 6]) * inv, __uint_as_float(ra[e + 7]) * inv));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(F_OE));
      mbar_arrive(bar(F_STG));
      if (row_ok && hf == 0)
        p.lse[((int64_t)x.b * p.H + x.h) * p.N + n] = lt > 0.f ? (m_run + log2f(lt)) * kLn2 : INFINITY;
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
              const cuuint32_t* box, CUtensorMapDataType dt) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map4(CUtensorMap* map, const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box, CUtensorMapDataType dt) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool MASK, bool F16>
cudaError_t launch_d(const Problem& pr, void* o, float* lse, cudaStream_t s) {
  using C = FCfg<D, F16>;
  const CUtensorMapDataType dt = F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap mq, mk, mv, mo;
  const cuuint64_t e = 2;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.N, (cuuint64_t)(pr.H * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.N * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mq, pr.q, dims, str, box, dt)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.M, (cuuint64_t)(pr.Hkv * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.M * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BK, 1};
    if (!make_map(&mk, pr.k, dims, str, box, dt)) return cudaErrorInvalidValue;
    if (!make_map(&mv, pr.v, dims, str, box, dt)) return cudaErrorInvalidValue;
  }
  {
    // O [DV,H,N,B]: rows n of one head are H*DV elements apart; stored in
    // 64-column boxes of 128 rows
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)pr.H, (cuuint64_t)pr.N, (cuuint64_t)pr.B};
    const cuuint64_t str[3] = {D * e, (cuuint64_t)pr.H * D * e, (cuuint64_t)pr.N * pr.H * D * e};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)C::BQ, 1};
    if (!make_map4(&mo, o, dims, str, box, dt)) return cudaErrorInvalidValue;
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
  p.o = o;
  p.lse = lse;
  p.kt_live = pr.kt_live;
  // persistent: one CTA per SM (each owns the SM's tensor memory), walking units
  const int64_t units = ((pr.N + C::BQ - 1) / C::BQ) * pr.H * pr.B;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int64_t grid = units < sms ? units : sms;
  cudaError_t err =
      cudaFuncSetAttribute(fwd_tc_kernel<D, MASK, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  fwd_tc_kernel<D, MASK, F16><<<(unsigned)grid, kThreads, C::SMEM, s>>>(mq, mk, mv, mo, p);
  return cudaPeekAtLastError();
}

}  // namespace

bool forward_tc_supported(const Problem& p) {
  if ((p.dtype != FAB_BF16 && p.dtype != FAB_F16) || p.DK != p.DV) return false;
  if (p.DK != 64 && p.DK != 128) return false;
  if (p.N >= (1ll << 31) || p.M >= (1ll << 31) || p.H * p.B >= (1ll << 31)) return false;
  if (((p.N + 127) / 128) * p.H * p.B >= (1ll << 31)) return false;
  return true;
}

cudaError_t launch_forward_tc(const Problem& p, void* o, float* lse, cudaStream_t s) {
  const bool m = p.mask != nullptr;
  if (p.dtype == FAB_F16) {
    if (p.DK == 128) return m ? launch_d<128, true, true>(p, o, lse, s) : launch_d<128, false, true>(p, o, lse, s);
    return m ? launch_d<64, true, true>(p, o, lse, s) : launch_d<64, false, true>(p, o, lse, s);
  }
  if (p.DK == 128) return m ? launch_d<128, true, false>(p, o, lse, s) : launch_d<128, false, false>(p, o, lse, s);
  return m ? launch_d<64, true, false>(p, o, lse, s) : launch_d<64, false, false>(p, o, lse, s);
}

uint32_t take_error_fwd() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err_fwd, &z, sizeof(z));
  return v;
}

}  // namespace fab
