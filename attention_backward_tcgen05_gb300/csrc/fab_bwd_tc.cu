// fab_bwd_tc.cu -- the key/value pass of the attention backward on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory,
// operands staged by TMA in 128-byte-swizzled shared memory).  bf16 or f16
// inputs (template parameter F16; P and dS are rounded to the same type),
// D = DK = DV in {64, 128}, f32 accumulation; writes the dK and dV slices of
// the packed f32 result.  The query pass (fab_dq_tc.cu) writes dQ.
//
// Math (labml "Flash Attention", "Backward pass"; ggmlR attn_ref for the mask
// and scale): with S = scale * Q K^T + mask, P = exp(S - LSE) (the saved row
// log-sum-exp), dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dK = scale dS^T Q.
// D_i = dO_i . O_i comes from the preprocess kernel.
//
// Decomposition: work units of (key tile of BM = 128 keys, key/value head,
// batch); persistent CTAs, one per SM, walk them.  A unit's key/value tile
// stays in shared memory; the unit walks every query tile of BQ = 128
// queries (skipping tiles a top-left causal mask empties) and, for each,
// every query head of the GQA group, so dK and dV of the group accumulate in
// tensor memory without atomics and the additive mask tile (shared by all
// heads) is read once per query tile.
//
// Per query tile, in the transposed ("key rows") orientation so that one
// thread owns one key row of every tensor-memory tile:
//   S^T  = K  Q^T     [BM x BQ]  A = K (smem, K-major),  B = Q (smem, K-major)
//   dP^T = V  dO^T    [BM x BQ]  A = V,                  B = dO
//   P^T  = exp2(S^T * scale*log2e + mask*log2e - LSE*log2e)
//   dS^T = P^T * (dP^T - D)
//   dV  += P^T dO     [BM x D]   A = P^T (tmem),  B = dO (smem, MN-major)
//   dK  += dS^T Q     [BM x D]   A = dS^T (tmem), B = Q (smem, MN-major)
// Every product is an M = 128, N = 128 (or D) MMA: an N = 64 product costs
// the tensor pipe as long as an N = 128 one.
//
// Tensor memory (512 columns): two tile buffers X0 at 0 and X1 at 128, dV at
// 256, dK at 256 + D.  Query tile i lives in X(i % 2) from start to end:
// S^T(i) lands there; the softmax warps read it into registers (P stays in
// registers), then dP^T(i) lands in the same columns; a warp reads its 64
// dP^T columns in two halves of 32 queries and writes each half's P^T and
// dS^T (packed 16-bit, 16 columns each) over the 32 columns it just read;
// dV(i) and dK(i) read them from there.  So dP^T(i) waits only for the
// softmax warps to read S^T(i), and S^T(i+1) only for dV(i-1), dK(i-1) to
// finish with the other buffer, while tile i is being worked on.
//
// Q and dO stream through separate rings: Q_i is needed first (S^T(i) is
// issued as soon as the other tile buffer is free), dO_i about a tile later
// (dP^T(i) after the softmax warps read S^T(i)), so the Q ring is one stage
// deeper and every load has about a tile to land.  The LSE and D rows of a
// tile travel with its dO stage.
//
// The products are issued by two warps, each waiting only on its own inputs.
// One issues dP^T(i) once S^T(i) was read, then S^T(i+1) once Q_{i+1} landed
// and dV(i-1), dK(i-1) are done.  The other issues dV(i) + dK(i) once P^T(i),
// dS^T(i) are written.  (Holding dV(i), dK(i) back until dP^T(i+1) is issued
// was measured slower: it delays the buffer S^T(i+2) needs.)  A single issuing thread stalls the tensor pipe for
// one to two hundred cycles at every commit and barrier wait; with two
// streams those stalls overlap the other stream's MMAs.
//
// Unit switch: a unit's key and value tiles are released as soon as its last
// S^T and dP^T finish, so the next unit's are loaded while the unit's last
// dV/dK products and its epilogue run.  The softmax warps write dV and dK
// themselves (through shared memory, whole rows to global memory), which
// leaves the TMA unit to the loads: bulk tensor stores of the 128 KB ahead
// of the next key tile held that load back by some 3,000 cycles.
//
// Warps (352 threads): 0 = TMA producer (and the tile's LSE and D rows);
// 1 = tensor-memory allocator and S^T/dP^T issuer; 10 = dV/dK issuer (lane 0
// of an issuer warp issues); 2-9 = softmax/dS and the epilogue (thread = key
// row; two warps per tensor-memory lane quarter, each taking 64 of the tile's
// 128 queries).  All hand-offs are mbarriers; every wait is bounded (see
// fab_device.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fab.h"
#include "fab_device.cuh"
#include "fab_internal.h"

namespace fab {
namespace {

__device__ uint32_t g_err_tc;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;

template <int D, bool F16 = false>
struct Cfg {
  static constexpr int BM = 128;  // keys per CTA (tensor-memory lanes)
  static constexpr int BQ = 128;  // queries per step
  static constexpr int QST = D == 128 ? 3 : 4;  // Q ring
  static constexpr int OST = D == 128 ? 2 : 4;  // dO ring (with the LSE and D rows)
  static constexpr int ATOMS = D / 64;             // 128-byte swizzle atoms along D
  static constexpr uint32_t ATOM = 128 * 128;      // one 128-row x 128-byte atom column
  static constexpr uint32_t TILE = ATOMS * ATOM;   // one 128 x D tile of 16-bit elements
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TILE;
  static constexpr uint32_t OFF_Q = OFF_V + TILE;           // + stage * TILE
  static constexpr uint32_t OFF_DO = OFF_Q + QST * TILE;    // + stage * TILE
  static constexpr uint32_t OFF_LD = OFF_DO + OST * TILE;   // per dO stage: lse2[BQ], D[BQ]
  static constexpr uint32_t OFF_BAR = OFF_LD + OST * 2 * BQ * 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
  // the swizzled tiles need a 1024-byte-aligned base, checked at run time
  // (no room for alignment slack at D = 128); at least 116 KB so one CTA
  // owns an SM and its whole tensor memory
  // the mask's query-tile spans of a CTA's first SPAN_CAP units
  static constexpr int SPAN_CAP = 160;
  static constexpr uint32_t OFF_SPAN = OFF_MISC + 64;
  static constexpr uint32_t SMEM_USED = OFF_SPAN + SPAN_CAP * 4;
  static constexpr uint32_t SMEM = SMEM_USED > 118784 ? SMEM_USED : 118784;
  // tensor-memory columns: tile buffer b at 128 b (b = 0, 1)
  static constexpr uint32_t TM_X = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t ID_S = idesc_16(128, BQ, false, false, F16);
  static constexpr uint32_t ID_DVK = idesc_16(128, D, false, true, F16);
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TM_DK + D <= TM_COLS, "tensor memory budget");
  // epilogue staging: one slot of 32 key rows x D/2 f32 columns per softmax
  // warp, four to a Q or dO stage
  static_assert(4 * 32 * (D / 2) * 4 == TILE, "four epilogue slots fill one ring stage");
  static_assert(QST <= 4 && OST <= QST, "barrier slots hold up to four stages; the dO ring is not deeper");
};

// barrier slots
enum : int {
  B_KV = 0,       // phase k: unit k's key tile landed
  B_FQ = 1,       // + i % QST: Q_i landed
  B_FO = 5,       // + i % OST: dO_i, LSE and D rows of tile i landed
  B_XF = 9,       // + i % QST: dV(i), dK(i) finished (Q and dO stages of i, buffer i % 2 free)
  B_S = 13,       // + i % 2: S^T(i) landed
  B_SF = 15,      // + i % 2: softmax warps read S^T(i)
  B_DP = 17,      // + i % 2: dP^T(i) landed
  B_DS = 19,      // + i % 2: softmax warps wrote P^T(i) and dS^T(i)
  B_FINAL = 21,   // phase k: unit k's dV/dK MMAs finished
  B_FIN_S = 22,   // every S^T and dP^T MMA finished
  B_FIN_X = 23,   // every dV/dK MMA finished
  B_DF = 24,      // phase k: unit k's epilogue read dV, dK from tensor memory
  B_KVF = 25,     // phase k: unit k's S^T and dP^T MMAs finished (its key and value tiles are free)
  B_V = 26,       // phase k: unit k's value tile landed
  B_COUNT = 27
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
  const uint8_t* qt_live;  // per key tile, a byte per query tile: mask not all -inf there; or null
};

template <int D, bool MASK, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const Params p) {
  using C = Cfg<D, F16>;
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
  // epilogue slots released: one count per softmax warp per unit
  uint32_t* r_cnt = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);
  float* ld_smem = reinterpret_cast<float*>(smem + C::OFF_LD);
  uint32_t* err = &g_err_tc;

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();

  // work units: (key tile, key/value head, batch), heavy (low) key tiles
  // first under a causal mask.  Round k of the G CTAs takes units k G ..
  // k G + G - 1, CTA c the c-th of them on even rounds and the (G-1-c)-th on
  // odd rounds.  (32-bit index arithmetic: the host guarantees units, N,
  // M < 2^31.)  A unit with no query at or after its keys (causal, M > N)
  // has n_it = 0: its dK, dV rows are zero.
  const int hb = (int)(p.Hkv * p.B);
  const int m_tiles = (int)((p.M + C::BM - 1) / C::BM);
  const int n_units = m_tiles * hb;
  const int rk2 = (int)(p.H / p.Hkv);
  const int q_tiles = (int)((p.N + C::BQ - 1) / C::BQ);
  uint32_t* span_s = reinterpret_cast<uint32_t*>(smem + C::OFF_SPAN);
  const bool span_tab = MASK && p.qt_live != nullptr && q_tiles < 65536;
  const int64_t live_qs = live_stride(q_tiles);
  struct Unit {
    int b, hkv, m0, qt0, n_it;
  };
  auto unit_at = [&](int kk) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    return G * kk + ((kk & 1) ? G - 1 - c : c);
  };
  // the live spans of this CTA's first units' key tiles, found once here
  // (made visible by the block sync below) instead of at every unit switch
  // of every role: {first live query tile, one past the last} as 16-bit halves
  if (span_tab)
    for (int i = (int)threadIdx.x; i < C::SPAN_CAP && unit_at(i) < n_units; i += kThreads) {
      int s0, s1;
      live_span(p.qt_live + (unit_at(i) / hb) * live_qs, q_tiles, s0, s1);
      span_s[i] = (uint32_t)s0 | ((uint32_t)s1 << 16);
    }
  // the unit this CTA takes in round kk; tab: its span from the shared table
  // (filled before the block sync), else from the map itself
  auto unit_of = [&](int kk, bool tab = true) {
    Unit x;
    const int u = unit_at(kk);
    const int jt = u / hb, rem = u - jt * hb;
    x.b = rem / (int)p.Hkv;
    x.hkv = rem - x.b * (int)p.Hkv;
    x.m0 = jt * C::BM;
    int qt0 = p.causal ? x.m0 / C::BQ : 0;  // first query tile holding some n >= m0
    if (qt0 > q_tiles) qt0 = q_tiles;
    int qt1 = q_tiles;  // one past the last query tile to visit
    if constexpr (MASK) {
      // query tiles before the first and after the last live one are all
      // -inf in the mask: their P is 0
      // (a CTA's rounds past the table, if any, skip nothing)
      if (span_tab && kk < C::SPAN_CAP) {
        int s0, s1;
        if (tab) {
          const uint32_t v = span_s[kk];
          s0 = (int)(v & 0xffffu);
          s1 = (int)(v >> 16);
        } else {
          live_span(p.qt_live + jt * live_qs, q_tiles, s0, s1);
        }
        if (s0 > qt0) qt0 = s0;
        if (s1 < qt1) qt1 = s1;
      }
    }
    x.qt0 = qt0;
    x.n_it = qt1 > qt0 ? rk2 * (qt1 - qt0) : 0;
    return x;
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *r_cnt = 0u;
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_V), 1);
    for (int s = 0; s < C::QST; ++s) {
      mbar_init(bar(B_FQ + s), 1);
      mbar_init(bar(B_XF + s), 1);
    }
    for (int s = 0; s < C::OST; ++s) mbar_init(bar(B_FO + s), 32);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(B_S + x), 1);
      mbar_init(bar(B_SF + x), kSoftmaxThreads);
      mbar_init(bar(B_DP + x), 1);
      mbar_init(bar(B_DS + x), kSoftmaxThreads);
    }
    mbar_init(bar(B_FINAL), 1);
    mbar_init(bar(B_FIN_S), 1);
    mbar_init(bar(B_FIN_X), 1);
    mbar_init(bar(B_DF), kSoftmaxThreads);
    mbar_init(bar(B_KVF), 1);
    fence_mbar_init();
    // this thread is the producer's issuing lane: start the first unit's
    // key/value tile copies before the tensor-memory allocation and block
    // sync below
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmO);
    for (int kk = 0; unit_at(kk) < n_units; ++kk) {
      const Unit x = unit_of(kk, false);
      if (x.n_it == 0) continue;
      mbar_arrive_expect_tx(bar(B_KV), C::TILE);
      mbar_arrive_expect_tx(bar(B_V), C::TILE);
      const int kvrow = x.b * (int)p.Hkv + x.hkv;
      for (int a = 0; a < C::ATOMS; ++a) {
        tma_load_3d(sbase + C::OFF_K + a * C::ATOM, &tmK, bar(B_KV), a * 64, x.m0, kvrow);
        tma_load_3d(sbase + C::OFF_V + a * C::ATOM, &tmV, bar(B_V), a * 64, x.m0, kvrow);
      }
      break;
    }
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
    // Per unit: an L2 prefetch of the next unit's key/value tiles, Q_g and
    // dO_g (with the tile's LSE and D rows) for every tile g, the key/value
    // tiles after the first tile's, as soon as the previous unit's last S^T
    // and dP^T are done with theirs.  Stages and barrier phases count tiles g
    // across units.  A unit's epilogue passes dV and dK through the Q and dO
    // stages of its last tile G, so Q_{G+QST} and dO_{G+OST} also wait for
    // the softmax warps to have released them.
    int g = 0, ku = 0, q_issued = 0, o_issued = 0;
    int kv_issued = 0;  // the first unit's copies were started at barrier initialisation
    for (int kk = 0; kv_issued == 0 && unit_at(kk) < n_units; ++kk)
      if (unit_of(kk).n_it > 0) kv_issued = 1;
    int stG[3] = {-64, -64, -64}, stK[3] = {0, 0, 0};  // last tile and index of the latest units
    bool ok = true;
    // a load into the stage tile gg - dist left: wait for the staging of the
    // unit (if any) whose last tile that was
    auto staged_wait = [&](int gg, int dist) {
#pragma unroll
      for (int i = 0; i < 3; ++i)
        if (stG[i] + dist == gg)
          return counter_wait(r_cnt, (uint32_t)(kSoftmaxThreads / 32) * (uint32_t)(stK[i] + 1), abort_flag, err);
      return true;
    };
    for (int kk = 0; ok && unit_at(kk) < n_units; ++kk) {
      const Unit x = unit_of(kk);
      if (x.n_it == 0) continue;
      if (lane == 0)
        for (int k2 = kk + 1; unit_at(k2) < n_units; ++k2) {
          const Unit y = unit_of(k2);
          if (y.n_it == 0) continue;
          for (int a = 0; a < C::ATOMS; ++a) {
            tma_prefetch_3d(&tmK, a * 64, y.m0, y.b * (int)p.Hkv + y.hkv);
            tma_prefetch_3d(&tmV, a * 64, y.m0, y.b * (int)p.Hkv + y.hkv);
          }
          break;
        }
      for (int it = 0; it < x.n_it; ++it, ++g) {
        const int qs = g % C::QST, os = g % C::OST;
        const int h = x.hkv * rk2 + it % rk2;
        const int n0 = (x.qt0 + it / rk2) * C::BQ;
        const int64_t rowbase = ((int64_t)x.b * p.H + h) * p.N;
        const int qrow = x.b * (int)p.H + h;
        // Q stage qs held tile g - QST: free once its dV and dK finished
        ok = (g < C::QST || mbar_wait(bar(B_XF + qs), ((g / C::QST) - 1) & 1, abort_flag, err)) &&
             staged_wait(g, C::QST);
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_proxy_async_smem();
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_FQ + qs), C::TILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(sbase + C::OFF_Q + qs * C::TILE + a * C::ATOM, &tmQ, bar(B_FQ + qs), a * 64, n0, qrow);
        }
        ++q_issued;
        // the tile's LSE and D rows, into registers first: their latency
        // overlaps the wait for the dO stage below
        float lv[C::BQ / 32], dv[C::BQ / 32];
#pragma unroll
        for (int k = 0; k < C::BQ / 32; ++k) {
          const int64_t n = n0 + lane + 32 * k;
          const bool in = n < p.N;
          lv[k] = in ? __ldg(p.lse + rowbase + n) * kLog2e : INFINITY;
          dv[k] = in ? __ldg(p.di + rowbase + n) : 0.f;
        }
        // dO stage os held tile g - OST: free once its dV and dK finished
        ok = (g < C::OST ||
              mbar_wait(bar(B_XF + (g - C::OST) % C::QST), ((g - C::OST) / C::QST) & 1, abort_flag, err)) &&
             staged_wait(g, C::OST);
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_proxy_async_smem();
        if (lane == 0) {
          mbar_expect_tx(bar(B_FO + os), C::TILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_4d(sbase + C::OFF_DO + os * C::TILE + a * C::ATOM, &tmO, bar(B_FO + os), a * 64, h, n0, x.b);
        }
        float* lds = ld_smem + os * 2 * C::BQ;
#pragma unroll
        for (int k = 0; k < C::BQ / 32; ++k) {
          lds[lane + 32 * k] = lv[k];
          lds[C::BQ + lane + 32 * k] = dv[k];
        }
        // one arrival per lane (count 32) publishes that lane's LSE/D stores
        mbar_arrive(bar(B_FO + os));
        ++o_issued;
        if (it == 0 && ku > 0) {
          // the unit's key and value tiles (the first unit's were started at
          // barrier initialisation), once the previous unit's last S^T and
          // dP^T products are done with theirs
          const int kvrow = x.b * (int)p.Hkv + x.hkv;
          ok = mbar_wait(bar(B_KVF), (ku - 1) & 1, abort_flag, err);
          if (!__all_sync(0xffffffffu, ok)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_KV), C::TILE);
            mbar_arrive_expect_tx(bar(B_V), C::TILE);
            for (int a = 0; a < C::ATOMS; ++a) {
              tma_load_3d(sbase + C::OFF_K + a * C::ATOM, &tmK, bar(B_KV), a * 64, x.m0, kvrow);
              tma_load_3d(sbase + C::OFF_V + a * C::ATOM, &tmV, bar(B_V), a * 64, x.m0, kvrow);
            }
          }
          ++kv_issued;
        }
      }
      stG[ku % 3] = g - 1;
      stK[ku % 3] = ku;
      ++ku;
    }
    // let every load this warp started land before shared memory goes away
    if (lane == 0) {
      if (kv_issued > 0) {
        mbar_drain(bar(B_KV), (kv_issued - 1) & 1);
        mbar_drain(bar(B_V), (kv_issued - 1) & 1);
      }
      for (int i = q_issued > C::QST ? q_issued - C::QST : 0; i < q_issued; ++i)
        mbar_drain(bar(B_FQ + i % C::QST), (i / C::QST) & 1);
      for (int i = o_issued > C::OST ? o_issued - C::OST : 0; i < o_issued; ++i)
        mbar_drain(bar(B_FO + i % C::OST), (i / C::OST) & 1);
    }
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // each issuer warp runs its loop convergently (descriptors stay
    // warp-uniform); lane 0 issues the MMAs and commits
    const uint32_t issue = lane == 0 ? 1u : 0u;
    auto wall = [&](int i, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, err));
    };
    // a K step only moves the descriptor's start address (address >> 4 in
    // the low 14 bits, all addresses < 232 KB), so a step is one add
    auto adv = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
    auto kstep = [](int kk) { return (uint32_t)((kk >> 2) * C::ATOM + (kk & 3) * 32); };
    bool ok = true;
    int g = 0, ku = 0;
    if (warp == 1) {
      // dP^T(g) = V dO_g^T into X(g % 2) once S^T(g) there was read; then
      // S^T(g+1) = K Q_{g+1}^T into X((g+1) % 2) once Q_{g+1} landed and
      // dV(g-1), dK(g-1) are done with that buffer.  A unit's first S^T also
      // waits for the unit's key tile, its first dP^T for the value tile.
      const uint64_t dK_km = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dV_km = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      const uint64_t dQ_km = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);   // stage 0
      const uint64_t dO_km = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);  // stage 0
      auto issue_s = [&](int gg) {
        const uint64_t q = adv(dQ_km, (gg % C::QST) * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tm + (gg & 1) * C::TM_X, adv(dK_km, kstep(kk)), adv(q, kstep(kk)), C::ID_S, kk > 0, issue);
        mma_commit(bar(B_S + (gg & 1)), issue);
      };
      for (int kk = 0; ok && unit_at(kk) < n_units; ++kk) {
        const int n_it = unit_of(kk).n_it;
        if (n_it == 0) continue;
        if (!(ok = wall(B_KV, ku & 1))) break;
        if (!(ok = wall(B_FQ + g % C::QST, (g / C::QST) & 1))) break;
        if (g >= 2 && !(ok = wall(B_XF + (g - 2) % C::QST, ((g - 2) / C::QST) & 1))) break;
        tc_fence_after();
        issue_s(g);
        for (int it = 0; it < n_it; ++it, ++g) {
          if (!(ok = wall(B_SF + (g & 1), (g >> 1) & 1))) break;
          if (!(ok = wall(B_FO + g % C::OST, (g / C::OST) & 1))) break;
          if (it == 0 && !(ok = wall(B_V, ku & 1))) break;
          tc_fence_after();
          const uint64_t o = adv(dO_km, (g % C::OST) * C::TILE);
#pragma unroll
          for (int kk2 = 0; kk2 < D / 16; ++kk2)
            mma_ss(tm + (g & 1) * C::TM_X, adv(dV_km, kstep(kk2)), adv(o, kstep(kk2)), C::ID_S, kk2 > 0, issue);
          mma_commit(bar(B_DP + (g & 1)), issue);
          if (it + 1 < n_it) {
            if (!(ok = wall(B_FQ + (g + 1) % C::QST, ((g + 1) / C::QST) & 1))) break;
            if (g >= 1 && !(ok = wall(B_XF + (g - 1) % C::QST, ((g - 1) / C::QST) & 1))) break;
            tc_fence_after();
            issue_s(g + 1);
          }
        }
        // the unit's key and value tiles are free once these products finish
        mma_commit(bar(B_KVF), issue);
        ++ku;
      }
      mma_commit(bar(B_FIN_S), issue);
      mbar_drain(bar(B_FIN_S), 0);
    } else {
      // dV += P^T dO_g and dK += dS^T Q_g once the softmax warps wrote
      // P^T(g), dS^T(g) into X: packed 16-bit, queries 32 c .. 32 c + 31 at
      // columns 32 c + 0..15 (P) and 32 c + 16..31 (dS).  A unit's first
      // products wait for the previous unit's epilogue to have read dV, dK.
      const uint64_t dO_mn = sdesc_sw128(sbase + C::OFF_DO, C::ATOM, 1024);  // stage 0, MN-major
      const uint64_t dQ_mn = sdesc_sw128(sbase + C::OFF_Q, C::ATOM, 1024);
      auto p_col = [](int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); };
      for (int kk = 0; ok && unit_at(kk) < n_units; ++kk) {
        const Unit x = unit_of(kk);
        if (x.n_it == 0) continue;
        for (int it = 0; it < x.n_it; ++it, ++g) {
          if (!(ok = wall(B_DS + (g & 1), (g >> 1) & 1))) break;
          if (it == 0 && ku > 0 && !(ok = wall(B_DF, (ku - 1) & 1))) break;
          tc_fence_after();
          const uint64_t o = adv(dO_mn, (g % C::OST) * C::TILE), q = adv(dQ_mn, (g % C::QST) * C::TILE);
          const uint32_t xb = tm + (g & 1) * C::TM_X;
#pragma unroll
          for (int kk2 = 0; kk2 < C::BQ / 16; ++kk2)
            mma_ts(tm + C::TM_DV, xb + p_col(kk2), adv(o, kk2 * 2048), C::ID_DVK, (it > 0 || kk2 > 0) ? 1u : 0u,
                   issue);
#pragma unroll
          for (int kk2 = 0; kk2 < C::BQ / 16; ++kk2)
            mma_ts(tm + C::TM_DK, xb + 16 + p_col(kk2), adv(q, kk2 * 2048), C::ID_DVK, (it > 0 || kk2 > 0) ? 1u : 0u,
                   issue);
          mma_commit(bar(B_XF + g % C::QST), issue);
        }
        // the unit's dV, dK (the last product depends on every S^T and dP^T
        // MMA of the unit) are complete for the epilogue
        mma_commit(bar(B_FINAL), issue);
        if (!ok) break;
        ++ku;
      }
      mma_commit(bar(B_FIN_X), issue);
      mbar_drain(bar(B_FIN_X), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax / dS
    // warps 2-5 take query columns 0-63 of the tile, warps 6-9 columns 64-127
    const int hf = (warp - 2) >> 2;
    const int r = (warp & 3) * 32 + lane;  // key row within the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c1 = p.scale * kLog2e;
    uint32_t mk[MASK ? 32 : 1];
    int g = 0, ku = 0;
    for (int kk = 0; unit_at(kk) < n_units; ++kk) {
      const Unit x = unit_of(kk);
      const int m = x.m0 + r;  // this thread's key (< 2^31)
      const bool key_in = m < p.M;
      if (x.n_it == 0) {
        // no query reaches these keys: dK = dV = 0
        if (key_in) {
          const int64_t row = ((int64_t)x.b * p.Hkv + x.hkv) * p.M + m;
          float* dst_v = p.dv + row * D + hf * (D / 2);
          float* dst_k = p.dk + row * D + hf * (D / 2);
          for (int c = 0; c < D / 2; c += 4) {
            *reinterpret_cast<float4*>(dst_v + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(dst_k + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        continue;
      }
      // additive mask: this thread's 64 values (its key row, its 64 query
      // columns), as f16 pairs, loaded once per query tile (the first head of
      // the group) and kept for the others.  Entries outside the matrix read
      // as 0; those rows or keys are masked through LSE = +inf or the key
      // bound anyway.
      auto load_mask = [&](int nbx) {  // nbx = the first of the thread's 64 queries
        if (!MASK) return;
        const uint16_t* src = p.mask + (key_in ? m : 0) + p.M * nbx;  // walks down the query rows
        if (key_in && nbx + 64 <= p.N) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t lo = __ldg(src);
            src += p.M;
            const uint32_t hi = __ldg(src);
            src += p.M;
            mk[c] = lo | (hi << 16);
          }
        } else {  // key past M or a ragged last query tile
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const bool in0 = key_in && nbx + 2 * c < p.N, in1 = key_in && nbx + 2 * c + 1 < p.N;
            const uint32_t lo = in0 ? __ldg(src) : 0u;
            src += p.M;
            const uint32_t hi = in1 ? __ldg(src) : 0u;
            src += p.M;
            mk[c] = lo | (hi << 16);
          }
        }
      };
      bool ok = true;
      // tiles walk query tile by query tile, each for every head of the group
      int nb = x.qt0 * C::BQ + hf * 64;  // first query of this thread's columns
      int hc = 0;                        // head within the group
      for (int left = x.n_it; left > 0; --left, ++g) {
        const int os = g % C::OST;
        if (MASK && hc == 0) load_mask(nb);
        ok = mbar_wait(bar(B_FO + os), (g / C::OST) & 1, abort_flag, err);
        const uint32_t xb = (uint32_t)(g & 1) * C::TM_X;
        const uint32_t ph = (uint32_t)(g >> 1) & 1u;
        ok = ok && mbar_wait(bar(B_S + (g & 1)), ph, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        uint32_t ra[32], rb[32];
        tmem_ld32(tm + lane_off + xb + hf * 64, ra);
        tmem_ld32(tm + lane_off + xb + hf * 64 + 32, rb);
        tmem_ld_wait2(ra, rb);
        // S^T(g) is in registers: the buffer may take dP^T(g)
        tc_fence_before();
        mbar_arrive(bar(B_SF + (g & 1)));
        const float4* lse4 = reinterpret_cast<const float4*>(ld_smem + os * 2 * C::BQ + hf * 64);
        const float4* di4 = reinterpret_cast<const float4*>(ld_smem + os * 2 * C::BQ + C::BQ + hf * 64);
        float pv[64];
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 l4 = lse4[q4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int jj = q4 * 4 + e;
            pv[jj] = fmaf(__uint_as_float(jj < 32 ? ra[jj] : rb[jj - 32]), c1, -lv[e]);
          }
        }
        if (MASK) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&mk[c]));
            pv[2 * c] = fmaf(mf.x, kLog2e, pv[2 * c]);
            pv[2 * c + 1] = fmaf(mf.y, kLog2e, pv[2 * c + 1]);
          }
        }
        // queries before the causal diagonal (top-left: key m > query n) and
        // keys past M; only diagonal tiles and the last key tile have any
        if ((p.causal && m - r + C::BM - 1 > nb) || m - r + C::BM > p.M) {
          int lo = 0;  // first allowed column e (query nb + e)
          if (p.causal && m - nb > lo) lo = m - nb;
          if (!key_in) lo = 64;
          const int li = lo > 64 ? 64 : lo;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e < li) pv[e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < 64; ++e) pv[e] = ex2_approx(pv[e]);

        ok = mbar_wait(bar(B_DP + (g & 1)), ph, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // queries 32 hh .. 32 hh + 31 of this warp's 64: read dP^T, then
          // write [P^T | dS^T] (16 + 16 packed columns) over the same 32 columns
          const uint32_t xcol = tm + lane_off + xb + hf * 64 + hh * 32;
          tmem_ld32(xcol, ra);
          tmem_ld_wait(ra);
          uint32_t pk[32];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 d4 = di4[hh * 8 + q4];
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const int jj = q4 * 4 + e;  // column within the half
              const float p0 = pv[hh * 32 + jj], p1 = pv[hh * 32 + jj + 1];
              pk[jj >> 1] = pack2<F16>(p0, p1);
              pk[16 + (jj >> 1)] = pack2<F16>(p0 * (__uint_as_float(ra[jj]) - dv[e]),
                                               p1 * (__uint_as_float(ra[jj + 1]) - dv[e + 1]));
            }
          }
          tmem_st32(xcol, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_DS + (g & 1)));
        if (++hc == rk2) {
          hc = 0;
          nb += C::BQ;
        }
      }
      if (!ok) break;
      // epilogue: dV and dK (scaled) of this key tile.  Each warp writes its
      // 32 key rows x D/2 columns, dV first, then dK, through its own slot in
      // the Q stage (warps 2-5) or the dO stage (warps 6-9) of the unit's
      // last tile G (every product reading them is done): tensor memory ->
      // registers -> the slot, a row per thread, its 16-byte chunks rotated
      // by the row so that neither these writes nor the column-wise reads
      // below conflict on banks -> global memory, each 16 lanes one half row
      // of whole 128-byte lines.  Rows past M are skipped.  The producer
      // holds the next loads into those stages until every warp has
      // released its slot; the key and value tiles were released when the
      // unit's last S^T and dP^T finished, so the next unit's are on their
      // way.  The tensor-memory loads are warp collectives, so every lane
      // runs them.
      const int G = g - 1;
      const bool done = mbar_wait(bar(B_FINAL), ku & 1, abort_flag, err);
      const bool write = __all_sync(0xffffffffu, done && !*abort_flag);
      if (!write) break;
      tc_fence_after();
      constexpr int CH = D / 8;      // 16-byte chunks in a slot row (D/2 f32)
      constexpr int ROWB = CH * 16;  // slot row bytes
      constexpr int RPI = 32 / CH;   // slot rows per read instruction
      const uint32_t slot = (hf == 0 ? sbase + C::OFF_Q + (uint32_t)(G % C::QST) * C::TILE
                                     : sbase + C::OFF_DO + (uint32_t)(G % C::OST) * C::TILE) +
                            (uint32_t)(warp & 3) * (32u * ROWB);
      const int mw = x.m0 + (warp & 3) * 32;  // this warp's first key
      const int64_t kvrow0 = ((int64_t)x.b * p.Hkv + x.hkv) * p.M;
      auto stage = [&](uint32_t tcol, float mul) {
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          uint32_t rv[32];
          tmem_ld32(tm + lane_off + tcol + hf * (D / 2) + c0, rv);
          tmem_ld_wait(rv);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = c0 / 4 + k;
            st_shared_v4(slot + (uint32_t)lane * ROWB + ((uint32_t)(c ^ (lane & 7)) << 4),
                         __float_as_uint(mul * __uint_as_float(rv[4 * k])),
                         __float_as_uint(mul * __uint_as_float(rv[4 * k + 1])),
                         __float_as_uint(mul * __uint_as_float(rv[4 * k + 2])),
                         __float_as_uint(mul * __uint_as_float(rv[4 * k + 3])));
          }
        }
        __syncwarp();
      };
      auto drain = [&](float* dst) {
#pragma unroll 4
        for (int i = 0; i < CH; ++i) {
          const int rr = i * RPI + lane / CH, cl = lane % CH;
          const uint4 v = ld_shared_v4(slot + (uint32_t)rr * ROWB + ((uint32_t)(cl ^ (rr & 7)) << 4));
          if (mw + rr < p.M)
            __stcs(reinterpret_cast<float4*>(dst + (kvrow0 + mw + rr) * D + hf * (D / 2) + cl * 4),
                   make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                               __uint_as_float(v.w)));
        }
        __syncwarp();
      };
      stage(C::TM_DV, 1.f);
      drain(p.dv);
      stage(C::TM_DK, p.scale);
      // dV, dK have been read: the next unit's first products may overwrite them
      tc_fence_before();
      mbar_arrive(bar(B_DF));
      drain(p.dk);
      if (lane == 0) counter_bump(r_cnt);
      ++ku;
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
              const cuuint32_t* box, CUtensorMapDataType dt) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, dt, (cuuint32_t)rank,
                   const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool MASK, bool F16>
cudaError_t launch_d(const Problem& pr, cudaStream_t s) {
  using C = Cfg<D, F16>;
  const CUtensorMapDataType dt = F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap mq, mk, mv, mo;
  const cuuint64_t e = 2;  // bytes per 16-bit element
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.N, (cuuint64_t)(pr.H * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.N * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mq, pr.q, 3, dims, str, box, dt)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.M, (cuuint64_t)(pr.Hkv * pr.B)};
    const cuuint64_t str[2] = {D * e, (cuuint64_t)pr.M * D * e};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BM, 1};
    if (!make_map(&mk, pr.k, 3, dims, str, box, dt)) return cudaErrorInvalidValue;
    if (!make_map(&mv, pr.v, 3, dims, str, box, dt)) return cudaErrorInvalidValue;
  }
  {
    // d [DV,H,N,B]: rows n of one head are H*DV elements apart
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)pr.H, (cuuint64_t)pr.N, (cuuint64_t)pr.B};
    const cuuint64_t str[3] = {D * e, (cuuint64_t)pr.H * D * e, (cuuint64_t)pr.N * pr.H * D * e};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mo, pr.d, 4, dims, str, box, dt)) return cudaErrorInvalidValue;
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
  p.qt_live = pr.qt_live;
  // persistent: one CTA per SM (each owns the SM's tensor memory), walking units
  const int64_t units = ((pr.M + C::BM - 1) / C::BM) * pr.Hkv * pr.B;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int64_t grid = units < sms ? units : sms;
  cudaError_t err =
      cudaFuncSetAttribute(bwd_tc_kernel<D, MASK, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  bwd_tc_kernel<D, MASK, F16><<<(unsigned)grid, kThreads, C::SMEM, s>>>(mq, mk, mv, mo, p);
  return cudaPeekAtLastError();
}

}  // namespace

bool backward_tc_supported(const Problem& p) {
  if ((p.dtype != FAB_BF16 && p.dtype != FAB_F16) || p.DK != p.DV) return false;
  if (p.DK != 64 && p.DK != 128) return false;
  // TMA coordinates are 32-bit; grid.x must fit as well
  if (p.N >= (1ll << 31) || p.M >= (1ll << 31) || p.H * p.B >= (1ll << 31)) return false;
  if (((p.N + 127) / 128) * p.H * p.B >= (1ll << 31)) return false;  // query-pass units
  if (((p.M + 127) / 128) * p.Hkv * p.B >= (1ll << 31)) return false;  // key-pass units
  return true;
}

cudaError_t launch_backward_tc(const Problem& p, cudaStream_t s) {
  const bool m = p.mask != nullptr;
  if (p.dtype == FAB_F16) {
    if (p.DK == 128) return m ? launch_d<128, true, true>(p, s) : launch_d<128, false, true>(p, s);
    return m ? launch_d<64, true, true>(p, s) : launch_d<64, false, true>(p, s);
  }
  if (p.DK == 128) return m ? launch_d<128, true, false>(p, s) : launch_d<128, false, false>(p, s);
  return m ? launch_d<64, true, false>(p, s) : launch_d<64, false, false>(p, s);
}

uint32_t take_error_tc() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err_tc, &z, sizeof(z));
  return v;
}

}  // namespace fab
