// fab_dq_tc.cu -- the query-gradient pass of the attention backward on the
// fifth-generation tensor cores.  bf16 or f16 inputs (template parameter
// F16; P and dS are rounded to the same type), D = DK = DV in {64, 128}, f32
// accumulation; writes the dQ slice of the packed f32 result.
//
// Math (labml "Flash Attention", "Backward pass"; ggmlR attn_ref for the mask
// and scale): P = exp(scale * Q K^T + mask - LSE), dP = dO V^T,
// dS = P * (dP - D), dQ = scale * dS K; LSE from the forward.  D_i = dO_i .
// O_i either comes from the preprocess kernel or, when the kernel is built
// with FUSE_D, is computed here (each row's dO is in shared memory anyway)
// and written out for the key/value pass, which then runs after this one.
//
// Decomposition: one CTA per (query tile of 128 rows, query head, batch).  Q
// and dO stay in shared memory; key tiles stream through a three-stage TMA
// ring and value tiles through a two-stage one.  dQ accumulates in tensor
// memory over every key tile and is written once, so this pass needs no
// atomics and no zero fill.  The key/value pass (fab_bwd_tc.cu) recomputes
// the same S and dP in the transposed orientation; the two passes write
// disjoint slices.
//
// Per key tile j (thread = query row, 128 tensor-memory lanes):
//   S    = Q  K_j^T   [128 x 128]  A = Q (smem, K-major),   B = K_j (K-major)
//   dP   = dO V_j^T   [128 x 128]  A = dO (smem, K-major),  B = V_j (K-major)
//   dS   = exp2(S*scale*log2e + mask*log2e - LSE*log2e) * (dP - D) -> 16-bit,
//          written over the S columns it came from
//   dQ  += dS K_j     [128 x D]    A = dS (tmem),           B = K_j (MN-major)
// Three 128-column tensor-memory buffers rotate: tile j's S lands in buffer
// j % 3, its dP (and then dS, written over dP) in buffer (j + 2) % 3.  P stays
// in registers, so S(j)'s buffer is free as soon as the softmax warps have
// read it and dP(j+1) may go there; S(j+2) takes the buffer dQ(j) has
// finished reading.
//
// The three products are issued by three warps, one stream each, every one
// waiting only on its own inputs: S(j) once K_j landed and dQ(j-2) freed its
// buffer, dP(j) once V_j landed and the softmax warps read S(j-1), dQ(j) once
// they wrote dS(j).  A single issuing thread stalls the tensor pipe for one
// to two hundred cycles at every commit and barrier wait; with three streams
// those stalls overlap other streams' MMAs.  Each group of eight MMAs ends in
// one commit, which the producer also uses to recycle key and value stages.
//
// Warps (384 threads): 0 = TMA producer; 1 = tensor-memory allocator and S
// issuer; 10 = dP issuer; 11 = dQ issuer (lane 0 of an issuer warp issues);
// 2-9 = softmax/dS and the epilogue (two warps per tensor-memory lane
// quarter, each taking 64 of the tile's 128 keys).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fab.h"
#include "fab_device.cuh"
#include "fab_internal.h"

namespace fab {
namespace {

__device__ uint32_t g_err_dq;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;

template <int D, bool F16 = false>
struct QCfg {
  static constexpr int BQ = 128;  // queries per CTA (tensor-memory lanes)
  static constexpr int BK = 128;  // keys per tile
  static constexpr int KST = 3;   // key ring stages
  static constexpr int VST = 2;   // value ring stages
  static constexpr int ATOMS = D / 64;
  static constexpr uint32_t ATOM = 128 * 128;  // one 128-row x 128-byte swizzle atom column
  static constexpr uint32_t TILE = ATOMS * ATOM;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = OFF_Q + TILE;
  static constexpr uint32_t OFF_K = OFF_DO + TILE;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + VST * TILE;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
  // +1024 to align the dynamic base; at least 116 KB so one CTA owns an SM
  // and its whole tensor memory
  static constexpr uint32_t OFF_DPART = OFF_MISC + 64;  // D_i partial sums, 2 x BQ floats
  // the mask's key-tile spans of a CTA's first SPAN_CAP units
  static constexpr int SPAN_CAP = 160;
  static constexpr uint32_t OFF_SPAN = OFF_DPART + 2 * BQ * 4;
  static constexpr uint32_t SMEM_USED = OFF_SPAN + SPAN_CAP * 4 + 1024;
  static constexpr uint32_t SMEM = SMEM_USED > 118784 ? SMEM_USED : 118784;
  // tensor-memory columns
  static constexpr uint32_t TM_BUF = 128;  // buffer b at columns 128 b, b = 0, 1, 2
  static constexpr uint32_t TM_DQ = 384;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t ID_S = idesc_16(128, BK, false, false, F16);
  static constexpr uint32_t ID_DQ = idesc_16(128, D, false, true, F16);
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TM_DQ + D <= TM_COLS, "tensor memory budget");
  static_assert(D * 128 * 4 == 2 * TILE, "dQ staging: one key stage per half of the columns");
};

enum : int {
  Q_QF = 0,      // Q and dO landed
  Q_KF = 1,      // + key stage (3)
  Q_KE = 4,      // + j % 3: dQ(j) finished (buffer (j + 2) % 3 and key stage j % 3 free)
  Q_VF = 7,      // + value stage (2)
  Q_S = 11,       // + j % 3: S(j) landed
  Q_DP = 14,      // + j % 3: dP(j) landed (value stage j % 2 free)
  Q_PD = 17,      // + j % 3: softmax warps read S(j) (its buffer is free)
  Q_DS = 20,      // + j % 3: softmax warps wrote dS(j)
  Q_FINAL = 23,   // phase k: unit k's dQ MMAs finished
  Q_FIN_S = 24,   // every S MMA finished
  Q_FIN_P = 25,   // every dP MMA finished
  Q_FIN_Q = 26,   // every dQ MMA finished
  Q_QOE = 27,     // phase k: unit k's S and dP MMAs finished and its D_i read dO (Q, dO free)
  Q_DF = 28,      // phase k: unit k's epilogue read dQ from tensor memory
  Q_STG = 29,     // phase k: unit k's dQ is staged in shared memory
  Q_DQI = 30,     // phase k: unit k's last dQ products have been issued
  Q_COUNT = 31
};
static_assert(Q_COUNT <= 32, "barrier area holds 32 slots");

struct QParams {
  int64_t B, H, Hkv, N, M;
  float scale;
  int causal;
  const float* lse;
  float* di;  // read, or written with FUSE_D
  const uint16_t* mask;
  float* dq;
  const uint16_t* o;  // forward output [D,H,N,B] (16-bit input type), read with FUSE_D
  float* pad[3];           // the packed result's padding after each slice, zeroed with FUSE_D
  int pad_n[3];
  const uint8_t* kt_live;  // per query tile, a byte per key tile: mask not all -inf there; or null
};

template <int D, bool FUSE_D, bool F16, bool MASK>
__global__ void __launch_bounds__(kThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                 const __grid_constant__ CUtensorMap tmDQ, const QParams p) {
  using C = QCfg<D, F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 4);
  // staging stages released by the bulk stores: two per unit, stage
  // (G + 2) % 3 first, then G % 3 (G = the unit's last tile)
  uint32_t* epi_cnt = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 8);
  uint32_t* err = &g_err_dq;

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();

  // work units: (query tile, head, batch), heavy (late) query tiles first
  // under a causal mask; heads of one GQA group are adjacent so their
  // key/value tiles are shared through L2.  Round k of the G CTAs takes units
  // k G .. k G + G - 1, CTA c the c-th of them on even rounds and the
  // (G-1-c)-th on odd rounds, which evens out the per-CTA totals.
  // (32-bit index arithmetic: the host guarantees units, N, M < 2^31)
  const int q_tiles = (int)((p.N + C::BQ - 1) / C::BQ);
  const int hb = (int)(p.H * p.B);
  const int n_units = q_tiles * hb;
  const int H = (int)p.H, rk2 = (int)(p.H / p.Hkv), m_tiles = (int)((p.M + C::BK - 1) / C::BK);
  uint32_t* span_s = reinterpret_cast<uint32_t*>(smem + C::OFF_SPAN);
  const bool span_tab = MASK && p.kt_live != nullptr && m_tiles < 65536;
  const int64_t live_ks = live_stride(m_tiles);
  struct Unit {
    int h, b, hkv, n0, j0, nkv;  // key tiles j0 .. j0 + nkv - 1; 32-bit, products that can exceed 2^31 widen first
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
  // the unit this CTA takes in round kk
  auto unit_of = [&](int kk) {
    Unit x;
    const int u = unit_at(kk);
    const int qi = u / hb, rem = u - qi * hb;
    const int b = rem / H, h = rem - b * H;
    x.h = h;
    x.b = b;
    x.hkv = h / rk2;
    const int qt = p.causal ? q_tiles - 1 - qi : qi;
    x.n0 = qt * C::BQ;
    int j0 = 0, j1 = m_tiles;
    if (p.causal) {
      const int last = (qt * C::BQ + C::BQ - 1) / C::BK + 1;  // key tiles holding some m <= n
      if (last < j1) j1 = last;
    }
    if (MASK && span_tab && kk < C::SPAN_CAP) {
      // key tiles before the first and after the last live one are all -inf
      // in the mask: their P is 0 (a CTA's later rounds, if any, skip nothing)
      const uint32_t v = span_s[kk];
      const int s0 = (int)(v & 0xffffu), s1 = (int)(v >> 16);
      if (s0 > j0) j0 = s0;
      if (s1 < j1) j1 = s1;
      if (j1 <= j0) j0 = 0, j1 = 1;  // nothing live: one tile (all P = 0), as without skipping
    }
    x.j0 = j0;
    x.nkv = j1 - j0;  // >= 1: key tile 0 holds m = 0 <= n
    return x;
  };

  // the live spans of this CTA's first units' query tiles, found once here
  // (made visible by the block sync below) instead of at every unit switch
  // of every role: {first live key tile, one past the last} as 16-bit halves
  if (span_tab)
    for (int i = (int)threadIdx.x; i < C::SPAN_CAP && unit_at(i) < n_units; i += kThreads) {
      int s0, s1;
      live_span(p.kt_live + tile_of(unit_at(i)) * live_ks, m_tiles, s0, s1);
      span_s[i] = (uint32_t)s0 | ((uint32_t)s1 << 16);
    }
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *epi_cnt = 0u;
    mbar_init(bar(Q_QF), 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bar(Q_KF + s), 1);
      mbar_init(bar(Q_KE + s), 1);
    }
    for (int s = 0; s < C::VST; ++s) mbar_init(bar(Q_VF + s), 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(bar(Q_S + s), 1);
      mbar_init(bar(Q_DP + s), 1);
      mbar_init(bar(Q_PD + s), kSoftmaxThreads);
      mbar_init(bar(Q_DS + s), kSoftmaxThreads);
    }
    mbar_init(bar(Q_FINAL), 1);
    mbar_init(bar(Q_FIN_S), 1);
    mbar_init(bar(Q_FIN_P), 1);
    mbar_init(bar(Q_FIN_Q), 1);
    mbar_init(bar(Q_QOE), 2 + kSoftmaxThreads);
    mbar_init(bar(Q_DF), kSoftmaxThreads);
    mbar_init(bar(Q_STG), kSoftmaxThreads);
    mbar_init(bar(Q_DQI), 1);
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
    // Per unit: V_0, K_0, then Q and dO (as soon as the previous unit's S and
    // dP products and its D_i no longer need theirs), then V_j, K_j.  Stages
    // and barrier phases count tiles g across units.  A unit's epilogue
    // stages dQ in the key stages of its last two tiles G - 1 and G (the
    // stages K(G+2) and K(G+3) would take), so those two loads also wait
    // for that unit's stores to have read them.
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmO);
      static_assert(C::KST == 3 && C::VST == 2, "stage recycling follows the three score buffers");
      int g = 0, k = 0, k_issued = 0, v_issued = 0, qo_issued = 0;
      int stG[3] = {-8, -8, -8}, stK[3] = {0, 0, 0};  // last tile and index of the latest units
      bool ok = true;
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const Unit x = unit_of(k);
        const int kvrow = (int)(x.b * p.Hkv + x.hkv);
        auto load_qo = [&]() {
          if (k > 0 && !(ok = mbar_wait(bar(Q_QOE), (k - 1) & 1, abort_flag, err))) return;
          mbar_arrive_expect_tx(bar(Q_QF), 2 * C::TILE);
          for (int a = 0; a < C::ATOMS; ++a) {
            tma_load_3d(sbase + C::OFF_Q + a * C::ATOM, &tmQ, bar(Q_QF), a * 64, (int)x.n0, (int)(x.b * p.H + x.h));
            tma_load_4d(sbase + C::OFF_DO + a * C::ATOM, &tmO, bar(Q_QF), a * 64, (int)x.h, (int)x.n0, (int)x.b);
          }
          ++qo_issued;
        };
        bool qo = false;
        for (int j = 0; j < x.nkv; ++j, ++g) {
          if (j == 1) {
            load_qo();
            qo = true;
            if (!ok) break;
          }
          // value stage g % 2 held V(g-2): free once dP(g-2) finished
          if (g >= 2 && !(ok = mbar_wait(bar(Q_DP + (g - 2) % 3), ((g - 2) / 3) & 1, abort_flag, err))) break;
          const int vs = g % C::VST;
          mbar_arrive_expect_tx(bar(Q_VF + vs), C::TILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(sbase + C::OFF_V + vs * C::TILE + a * C::ATOM, &tmV, bar(Q_VF + vs), a * 64,
                        (x.j0 + j) * C::BK, kvrow);
          ++v_issued;
          // key stage g % 3 held K(g-3): free once dQ(g-3) finished, and
          // once any epilogue staging there has been stored
          if (g >= 3 && !(ok = mbar_wait(bar(Q_KE + g % 3), ((g - 3) / 3) & 1, abort_flag, err))) break;
          int need = 0;  // releases of staging stages this load must see
#pragma unroll
          for (int i = 0; i < 3; ++i)
            if (stG[i] + 2 <= g && g <= stG[i] + 3) {
              const int r2 = 2 * stK[i] + (g - stG[i] - 1);  // 2k+1 for K(G+2), 2k+2 for K(G+3)
              if (r2 > need) need = r2;
            }
          if (need > 0) {
            if (!(ok = counter_wait(epi_cnt, (uint32_t)need, abort_flag, err))) break;
            fence_proxy_async_smem();
          }
          const int ks = g % C::KST;
          mbar_arrive_expect_tx(bar(Q_KF + ks), C::TILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(sbase + C::OFF_K + ks * C::TILE + a * C::ATOM, &tmK, bar(Q_KF + ks), a * 64,
                        (x.j0 + j) * C::BK, kvrow);
          ++k_issued;
        }
        if (ok && !qo) load_qo();
        stG[k % 3] = g - 1;
        stK[k % 3] = k;
      }
      // let every load started above land before shared memory goes away
      if (qo_issued > 0) mbar_drain(bar(Q_QF), (qo_issued - 1) & 1);
      for (int j = k_issued > C::KST ? k_issued - C::KST : 0; j < k_issued; ++j)
        mbar_drain(bar(Q_KF + j % C::KST), (j / C::KST) & 1);
      for (int j = v_issued > C::VST ? v_issued - C::VST : 0; j < v_issued; ++j)
        mbar_drain(bar(Q_VF + j % C::VST), (j / C::VST) & 1);
    }
  } else if (warp == 1 || warp >= 10) {
    // ------------------------------------------------------------ MMA issuers
    // each issuer warp runs its loops convergently (descriptors stay
    // warp-uniform); lane 0 issues the MMAs and commits
    const uint32_t issue = lane == 0 ? 1u : 0u;
    auto wall = [&](int i, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, abort_flag, err));
    };
    // a K step only moves the descriptor's start address (address >> 4 in
    // the low 14 bits, all addresses < 232 KB), so a step is one add
    auto adv = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
    auto kstep = [](int kk) { return (uint32_t)((kk >> 2) * C::ATOM + (kk & 3) * 32); };
    auto buf = [](int x) { return (uint32_t)(x % 3) * C::TM_BUF; };
    bool ok = true;
    int g = 0, k = 0;
    if (warp == 1) {
      // S(g) = Q K^T into buffer g, which held dS(g-2)
      const uint64_t dQ_km = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dK_km = sdesc_sw128(sbase + C::OFF_K, 16, 1024);  // key stage 0, K-major
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const int nkv = unit_of(k).nkv;
        if (!(ok = wall(Q_QF, k & 1))) break;
        // the previous unit's last dQ products go into the tensor pipe
        // before this unit's first scores: its epilogue waits for them
        if (k > 0 && !(ok = wall(Q_DQI, (k - 1) & 1))) break;
        for (int j = 0; j < nkv; ++j, ++g) {
          if (g >= 2 && !(ok = wall(Q_KE + (g - 2) % 3, ((g - 2) / 3) & 1))) break;
          if (!(ok = wall(Q_KF + g % C::KST, (g / C::KST) & 1))) break;
          tc_fence_after();
          const uint64_t kd = adv(dK_km, (g % C::KST) * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tm + buf(g), adv(dQ_km, kstep(kk)), adv(kd, kstep(kk)), C::ID_S, kk > 0, issue);
          mma_commit(bar(Q_S + g % 3), issue);
        }
        mma_commit(bar(Q_QOE), issue);  // the unit's S products are done with Q
      }
      mma_commit(bar(Q_FIN_S), issue);
      mbar_drain(bar(Q_FIN_S), 0);
    } else if (warp == 10) {
      // dP(g) = dO V^T into buffer g + 2, which held S(g-1)
      const uint64_t dO_km = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);
      const uint64_t dV_km = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const int nkv = unit_of(k).nkv;
        if (!(ok = wall(Q_QF, k & 1))) break;
        if (k > 0 && !(ok = wall(Q_DQI, (k - 1) & 1))) break;  // as for the scores
        for (int j = 0; j < nkv; ++j, ++g) {
          if (g >= 1 && !(ok = wall(Q_PD + (g - 1) % 3, ((g - 1) / 3) & 1))) break;
          if (!(ok = wall(Q_VF + g % C::VST, (g / C::VST) & 1))) break;
          tc_fence_after();
          const uint64_t vd = adv(dV_km, (g % C::VST) * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tm + buf(g + 2), adv(dO_km, kstep(kk)), adv(vd, kstep(kk)), C::ID_S, kk > 0, issue);
          mma_commit(bar(Q_DP + g % 3), issue);
        }
        mma_commit(bar(Q_QOE), issue);  // the unit's dP products are done with dO
      }
      mma_commit(bar(Q_FIN_P), issue);
      mbar_drain(bar(Q_FIN_P), 0);
    } else if (warp == 11) {
      // dQ += dS(g) K, dS(g) in buffer g + 2 (packed 16-bit: keys 0-63 at
      // +0..31, keys 64-127 at +64..95), K MN-major; a unit's first product
      // waits for the previous unit's epilogue to have read dQ
      const uint64_t dK_mn = sdesc_sw128(sbase + C::OFF_K, C::ATOM, 1024);
      auto a_col = [](int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); };
      for (int u = unit_at(0); ok && u < n_units; u = unit_at(++k)) {
        const int nkv = unit_of(k).nkv;
        for (int j = 0; j < nkv; ++j, ++g) {
          if (!(ok = wall(Q_DS + g % 3, (g / 3) & 1))) break;
          if (j == 0 && k > 0 && !(ok = wall(Q_DF, (k - 1) & 1))) break;
          tc_fence_after();
          const uint64_t kmn = adv(dK_mn, (g % C::KST) * C::TILE);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            mma_ts(tm + C::TM_DQ, tm + buf(g + 2) + a_col(kk), adv(kmn, kk * 2048), C::ID_DQ,
                   (j > 0 || kk > 0) ? 1u : 0u, issue);
          mma_commit(bar(Q_KE + g % 3), issue);
        }
        // the unit's dQ (its last product depends on every S and dP MMA of
        // the unit) is complete for the epilogue
        mma_commit(bar(Q_FINAL), issue);
        if (lane == 0) mbar_arrive(bar(Q_DQI));
        if (!ok) break;
        // the epilogue's bulk stores: once the softmax warps staged dQ, write
        // it out and release the two staging stages as each has been read
        if (!(ok = wall(Q_STG, k & 1))) break;
        if (lane == 0) {
          const Unit x = unit_of(k);
          const int G = g - 1;
          const uint32_t st0 = sbase + C::OFF_K + (uint32_t)((G + 2) % 3) * C::TILE;  // columns 0 .. D/2-1
          const uint32_t st1 = sbase + C::OFF_K + (uint32_t)(G % 3) * C::TILE;        // columns D/2 .. D-1
          for (int a = 0; a < D / 64; ++a)
            tma_store_3d(&tmDQ, st0 + a * C::ATOM, a * 32, (int)x.n0, (int)(x.b * p.H + x.h));
          bulk_commit_group();
          for (int a = 0; a < D / 64; ++a)
            tma_store_3d(&tmDQ, st1 + a * C::ATOM, D / 2 + a * 32, (int)x.n0, (int)(x.b * p.H + x.h));
          bulk_commit_group();
          bulk_wait_read_1();
          counter_bump(epi_cnt);
          bulk_wait_read_all();
          counter_bump(epi_cnt);
        }
        __syncwarp();
      }
      if (lane == 0) bulk_wait_read_all();  // (every group was waited for above; kept for an early exit)
      mma_commit(bar(Q_FIN_Q), issue);
      mbar_drain(bar(Q_FIN_Q), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax / dS
    const int hf = (warp - 2) >> 2;        // warps 2-5: keys 0-63 of a tile, warps 6-9: keys 64-127
    const int r = (warp & 3) * 32 + lane;  // query row within the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c1 = p.scale * kLog2e;
    constexpr bool has_mask = MASK;
    const bool mvec = (p.M & 7) == 0;  // mask rows start 16-byte aligned
    float* dpart = reinterpret_cast<float*>(smem + C::OFF_DPART);
    if (FUSE_D && blockIdx.x == 0 && warp == 2 && lane == 0)
#pragma unroll
      for (int k = 0; k < 3; ++k)
        for (int i = 0; i < p.pad_n[k]; ++i) p.pad[k][i] = 0.f;
    // A unit's first global reads (this thread's LSE, half of its share of
    // O for D_i, its first mask chunk) are issued before the previous unit's
    // epilogue, so their latency hides behind it; the other half of O is
    // read at the unit's start (all of it would not stay in registers).
    constexpr int CPH = D / 16;      // 16-byte chunks per half row
    constexpr int RPI = 32 / CPH;    // rows per load instruction
    uint4 ov[CPH];
    float lse_next = 0.f, di_next = 0.f;
    uint32_t mk[32];
    // (loads only, from a valid row: nothing here consumes a loaded value,
    // so the loads stay in flight; a row past N is masked where the values
    // are used)
    auto fetch = [&](int kk) {
      const Unit y = unit_of(kk);
      const int64_t ny = y.n0 + r < p.N ? y.n0 + r : p.N - 1;
      lse_next = ld_global_nc_f32(p.lse + (y.b * p.H + y.h) * p.N + ny);
      if (!FUSE_D) di_next = p.di[(y.b * p.H + y.h) * p.N + ny];
      if (FUSE_D) {
        // whole half rows per instruction: instruction i, lane l reads chunk
        // l % CPH of (this warp's) row i * RPI + l / CPH, so a row is full
        // cache lines rather than one sector per thread
#pragma unroll
        for (int i = 0; i < CPH / 2; ++i) {
          const int64_t nr = (int64_t)y.n0 + (warp & 3) * 32 + i * RPI + lane / CPH;
          const int64_t nc = nr < p.N ? nr : p.N - 1;
          ov[i] = ld_global_nc_v4(reinterpret_cast<const uint4*>(p.o + ((y.b * p.N + nc) * p.H + y.h) * D +
                                                                 hf * (D / 2) + (lane % CPH) * 8));
        }
      }
    };
    int g = 0, k = 0;
    if (unit_at(0) < n_units) fetch(0);
    for (int u = unit_at(0); u < n_units; u = unit_at(++k)) {
      const Unit x = unit_of(k);
      const int64_t n = x.n0 + r;
      const bool row_ok = n < p.N;
      const int64_t rowidx = (x.b * p.H + x.h) * p.N + (row_ok ? n : 0);
      // a row past N (zero-filled Q, dO) gets LSE = +inf, hence P = 0 and dS = 0
      const float lse2 = row_ok ? lse_next * kLog2e : INFINITY;
      float di;
      if (FUSE_D) {
        // D_i = dO_i . O_i: this thread takes columns hf * D/2 .. hf * D/2 + D/2 - 1
        // of its row (O fetched above, dO from the swizzled tile in shared
        // memory); the two halves meet in shared memory, the two warps of
        // the rows (w and w + 4) at named barrier 1 + w % 4
#pragma unroll
        for (int i = CPH / 2; i < CPH; ++i) {
          const int64_t nr = (int64_t)x.n0 + (warp & 3) * 32 + i * RPI + lane / CPH;
          const int64_t nc = nr < p.N ? nr : p.N - 1;
          ov[i] = ld_global_nc_v4(reinterpret_cast<const uint4*>(p.o + ((x.b * p.N + nc) * p.H + x.h) * D +
                                                                 hf * (D / 2) + (lane % CPH) * 8));
        }
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar(Q_QF), k & 1, abort_flag, err));
        float part = 0.f;
        if (got) {
          auto dot2 = [](uint32_t a, uint32_t b) {
            const float2 fa = unpack2<F16>(a), fb = unpack2<F16>(b);
            return fa.x * fb.x + fa.y * fb.y;
          };
          // chunk l % CPH of row i * RPI + l / CPH (as loaded), against the
          // same chunk of dO from the swizzled tile; the CPH lanes of a row
          // sum by shuffles, then each thread takes its own row's sum
          const int c = lane % CPH;
          const int e = hf * (D / 2) + 8 * c;  // first column of the 16-byte chunk
#pragma unroll
          for (int i = 0; i < CPH; ++i) {
            const int rr = (warp & 3) * 32 + i * RPI + lane / CPH;
            const uint4 dv = ld_shared_v4(sbase + C::OFF_DO + (uint32_t)(e / 64) * C::ATOM + rr * 128 +
                                          ((((e % 64) / 8) ^ (rr & 7)) << 4));
            float q = dot2(dv.x, ov[i].x) + dot2(dv.y, ov[i].y) + dot2(dv.z, ov[i].z) + dot2(dv.w, ov[i].w);
#pragma unroll
            for (int o = CPH / 2; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
            const float mine = __shfl_sync(0xffffffffu, q, (lane % RPI) * CPH);
            if (i == lane / RPI) part = mine;
          }
        }
        dpart[hf * C::BQ + r] = row_ok ? part : 0.f;
        named_bar_sync(1 + (warp & 3), 64);
        di = dpart[r] + dpart[C::BQ + r];
        if (hf == 0 && row_ok) p.di[rowidx] = di;
      } else {
        di = row_ok ? di_next : 0.f;
      }
      mbar_arrive(bar(Q_QOE));  // dO has been read for D_i
      // additive mask: this thread's 64 values (its query row, its 64 keys) of
      // the next tile are loaded one tile ahead, as f16 pairs.  Entries past M
      // read as 0; those keys are masked by the key bound anyway.
      const uint16_t* mrow = p.mask + p.M * (row_ok ? n : 0);
      auto load_mask = [&](int jx) {
        const int64_t mb = (int64_t)jx * C::BK + hf * 64;
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
      };
      if (has_mask && k == 0) load_mask(x.j0);  // later units: fetched with the previous unit's tail
      bool ok = true;
      int j = x.j0;
      for (; j < x.j0 + x.nkv; ++j, ++g) {
        const uint32_t sb = (uint32_t)(g % 3) * C::TM_BUF, db = (uint32_t)((g + 2) % 3) * C::TM_BUF;
        const uint32_t ph = (uint32_t)(g / 3) & 1u;
        const int64_t m0 = (int64_t)j * C::BK;
        const int64_t mb = m0 + hf * 64;  // first key of this thread's columns
        ok = mbar_wait(bar(Q_S + g % 3), ph, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        uint32_t ra[32], rb[32];
        tmem_ld32(tm + lane_off + sb + hf * 64, ra);
        tmem_ld32(tm + lane_off + sb + hf * 64 + 32, rb);
        tmem_ld_wait2(ra, rb);
        // S(g) is in registers: its buffer may take dP(g+1)
        tc_fence_before();
        mbar_arrive(bar(Q_PD + g % 3));
        float pv[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) pv[e] = fmaf(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]), c1, -lse2);
        if (has_mask) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&mk[c]));
            pv[2 * c] = fmaf(mf.x, kLog2e, pv[2 * c]);
            pv[2 * c + 1] = fmaf(mf.y, kLog2e, pv[2 * c + 1]);
          }
          if (j + 1 < x.j0 + x.nkv) load_mask(j + 1);
        }
        // keys past the causal diagonal (top-left: key m > query n) or past M;
        // only the diagonal tile and a ragged last tile have any
        if ((p.causal && m0 + C::BK - 1 > x.n0) || m0 + C::BK > p.M) {
          int64_t lim = 63;                              // last allowed column e (key mb + e)
          if (p.causal && n - mb < lim) lim = n - mb;    // m <= n
          if (p.M - 1 - mb < lim) lim = p.M - 1 - mb;    // m < M
          const int li = lim < -1 ? -1 : (int)lim;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e > li) pv[e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < 64; ++e) pv[e] = ex2_approx(pv[e]);
        ok = mbar_wait(bar(Q_DP + g % 3), ph, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        tmem_ld32(tm + lane_off + db + hf * 64, ra);
        tmem_ld32(tm + lane_off + db + hf * 64 + 32, rb);
        tmem_ld_wait2(ra, rb);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 2 * c;
          const float d0 = __uint_as_float(e < 32 ? ra[e] : rb[e - 32]);
          const float d1 = __uint_as_float(e + 1 < 32 ? ra[e + 1] : rb[e + 1 - 32]);
          pk[c] = pack2<F16>(pv[e] * (d0 - di), pv[e + 1] * (d1 - di));
        }
        // packed dS over the first 32 of this warp's own 64 dP columns (the
        // other warp of the lane quarter reads only its own columns)
        tmem_st32(tm + lane_off + db + hf * 64, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(Q_DS + g % 3));
      }
      g += x.j0 + x.nkv - j;  // keep the tile count in step after an early exit
      if (unit_at(k + 1) < n_units) {
        fetch(k + 1);
        if (has_mask) {
          const Unit y = unit_of(k + 1);
          const int64_t ny = y.n0 + r;
          const int64_t my = (int64_t)y.j0 * C::BK + hf * 64;  // first key of the next unit's first tile
          if (ny < p.N) {
            const uint16_t* src = p.mask + p.M * ny + my;
            if (mvec && my + 64 <= p.M) {
              const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint4 v = __ldg(s4 + c);
                mk[4 * c] = v.x;
                mk[4 * c + 1] = v.y;
                mk[4 * c + 2] = v.z;
                mk[4 * c + 3] = v.w;
              }
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const uint32_t lo = (my + 2 * c < p.M) ? (uint32_t)__ldg(src + 2 * c) : 0u;
                const uint32_t hi = (my + 2 * c + 1 < p.M) ? (uint32_t)__ldg(src + 2 * c + 1) : 0u;
                mk[c] = lo | (hi << 16);
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) mk[c] = 0u;
          }
        }
      }
      // epilogue: dQ of this query tile (scaled), half of the columns per
      // warp.  Staged in the key stages of the unit's last two tiles (their
      // products are done; the producer holds the next loads into them until
      // the dQ issuer's bulk stores have read them): columns 0 .. D/2-1 in
      // stage (G + 2) % 3, the rest in stage G % 3, as 32-column atoms of
      // 128-byte swizzled rows.  The stores clip rows past N.  The
      // tensor-memory loads are warp collectives, so every lane runs them.
      const int G = g - 1;  // the unit's last tile
      auto stage = [&](int half) {
        return sbase + C::OFF_K + (uint32_t)((half == 0 ? G + 2 : G) % 3) * C::TILE;
      };
      const bool done = mbar_wait(bar(Q_FINAL), k & 1, abort_flag, err);
      const bool write = __all_sync(0xffffffffu, done && !*abort_flag);
      if (write) {
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          uint32_t rv[32];
          tmem_ld32(tm + lane_off + C::TM_DQ + hf * (D / 2) + c0, rv);
          tmem_ld_wait(rv);
          const uint32_t row = stage(hf) + (uint32_t)(c0 / 32) * C::ATOM + r * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(row + ((q ^ (r & 7)) << 4), __float_as_uint(p.scale * __uint_as_float(rv[4 * q])),
                         __float_as_uint(p.scale * __uint_as_float(rv[4 * q + 1])),
                         __float_as_uint(p.scale * __uint_as_float(rv[4 * q + 2])),
                         __float_as_uint(p.scale * __uint_as_float(rv[4 * q + 3])));
        }
        fence_proxy_async_smem();
      }
      // dQ has been read: the next unit's first dQ product may overwrite it;
      // and it is staged: the dQ issuer writes it out
      tc_fence_before();
      mbar_arrive(bar(Q_DF));
      mbar_arrive(bar(Q_STG));
      // both warps of the rows (w and w + 4, named barrier 5 + w % 4) take
      // the same branch below, so the D_i barrier of the next unit pairs up
      if (named_bar_or(5 + (warp & 3), 64, !write || *abort_flag != 0u)) break;
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
  return enc(map, dt, (cuuint32_t)rank,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool FUSE_D, bool F16, bool MASK>
cudaError_t launch_d(const Problem& pr, cudaStream_t s) {
  using C = QCfg<D, F16>;
  const CUtensorMapDataType dt = F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap mq, mk, mv, mo, mdq;
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
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BK, 1};
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
  {
    // the packed f32 dQ slice [D,N,H,B], stored in 32-column (128-byte) boxes
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)pr.N, (cuuint64_t)(pr.H * pr.B)};
    const cuuint64_t str[2] = {D * 4, (cuuint64_t)pr.N * D * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)C::BQ, 1};
    if (!make_map(&mdq, pr.packed, 3, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) return cudaErrorInvalidValue;
  }
  QParams p;
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
  p.dq = pr.packed;
  p.o = static_cast<const uint16_t*>(pr.o);
  p.kt_live = pr.kt_live;
  {
    const int64_t nq = D * pr.N * pr.H * pr.B, nk = D * pr.M * pr.Hkv * pr.B;
    p.pad[0] = pr.packed + nq;
    p.pad_n[0] = (int)(pr.off_k / 4 - nq);
    p.pad[1] = pr.packed + pr.off_k / 4 + nk;
    p.pad_n[1] = (int)((pr.off_v - pr.off_k) / 4 - nk);
    p.pad[2] = pr.packed + pr.off_v / 4 + nk;
    p.pad_n[2] = (int)((pr.end - pr.off_v) / 4 - nk);
  }
  // persistent: one CTA per SM (each owns the SM's tensor memory), walking units
  const int64_t units = ((pr.N + C::BQ - 1) / C::BQ) * pr.H * pr.B;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int64_t grid = units < sms ? units : sms;
  cudaError_t err =
      cudaFuncSetAttribute(dq_tc_kernel<D, FUSE_D, F16, MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  dq_tc_kernel<D, FUSE_D, F16, MASK><<<(unsigned)grid, kThreads, C::SMEM, s>>>(mq, mk, mv, mo, mdq, p);
  return cudaPeekAtLastError();
}

// the instance with the additive mask's code, or without it
template <int D, bool FUSE_D, bool F16>
cudaError_t launch_m(const Problem& pr, cudaStream_t s) {
  return pr.mask != nullptr ? launch_d<D, FUSE_D, F16, true>(pr, s) : launch_d<D, FUSE_D, F16, false>(pr, s);
}

}  // namespace

cudaError_t launch_dq_tc(const Problem& p, bool fuse_d, cudaStream_t s) {
  if (p.dtype == FAB_F16) {
    if (fuse_d) return p.DK == 128 ? launch_m<128, true, true>(p, s) : launch_m<64, true, true>(p, s);
    return p.DK == 128 ? launch_m<128, false, true>(p, s) : launch_m<64, false, true>(p, s);
  }
  if (fuse_d) return p.DK == 128 ? launch_m<128, true, false>(p, s) : launch_m<64, true, false>(p, s);
  return p.DK == 128 ? launch_m<128, false, false>(p, s) : launch_m<64, false, false>(p, s);
}

uint32_t take_error_dq() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_dq, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err_dq, &z, sizeof(z));
  return v;
}

}  // namespace fab
