// bwd.cu -- tile-list-driven flash-attention backward for sm_103a.
//
// Gradients of L = sum(out * dO) through the softmax and the score mod
// (tutorial "FlexAttention in PyTorch", Pattern 3: both score mods are
// differentiable and the backward is fused):
//     P_ij  = exp(s_ij - LSE_i)                      (s = score_mod(scale q.k))
//     dP_ij = dO_i . v_j,   Delta_i = dO_i . out_i   (= sum_j P_ij dP_ij)
//     dS_ij = P_ij (dP_ij - Delta_i) * ds_ij/dx_ij
//     dv_j = sum_i P_ij dO_i,  dk_j = scale sum_i dS_ij q_i,  dq_i = scale sum_j dS_ij k_j
// over the visible pairs only, visiting for each key tile the query tiles of
// its column lists (FULL first, then PARTIAL with the mask per element).
//
// Kernels:
//  1. bwd_pre   -- Delta_i = dO_i . out_i (fp32) and LSE, laid out per query
//                  tile (the key-row warps copy a tile's values in per step),
//                  and a zeroed fp32 dq accumulator.
//  2. bwd_kernel -- persistent, one CTA per SM, each taking every gridDim.x-th
//     (b, h, key tile J) of the longest-first order:
//       warps 0-7    TMEM lane r = 32 (warp % 4) + lane = key row r, query columns
//                    [64 (warp / 4), +64): phase A, P^T into TMEM; phase B, dS^T
//                    into shared memory; LSE_I, Delta_I copied in per step
//       warps 8-11   dQ rows [32 (warp % 4), +32) out of TMEM, staged 32 x 32 at a
//                    time and TMA bulk reduce-added into the fp32 accumulator;
//                    after a key tile's last step, its dV and dK rows out of TMEM,
//                    staged the same way and TMA-stored
//       warp 12      TMA producer: V_J, then Q_I, dO_I per step, K_J with the first
//       warp 13      MMA issuer, five tcgen05 GEMMs per (I, J):
//                     once P^T is in:  dV  += P^T dO   (P^T bf16 read from TMEM [0,32), [64,96))
//                     once dS is in:   dQ   = dS K     (dS read MN-major; D = 128: TMEM [128,256),
//                                                       D = 64: two buffers [384,448), [448,512))
//                                      S^T  = K Q^T    (next step; TMEM [0,128))
//                                      dK  += dS^T Q   (dS read K-major)
//                                      dP^T = V dO^T   (next step; TMEM [128,256); with D = 128
//                                                       once dQ is read out of those columns)
//     dV runs while the key-row warps compute dS, and the next S^T before dK
//     (with D = 64, right after dV) so that phase A of the next step can start
//     early.  Registers are split per warpgroup (setmaxnreg): the dQ and
//     producer / MMA warpgroups give theirs up to the key-row warps, which hold
//     a row's 64 probabilities across the two phases.
//     dK and dV stay in TMEM for the whole key tile and are written once
//     (no atomics); dQ partial tiles are added into the fp32 accumulator.
//     Across key tiles the pipeline keeps going: the next tile's V loads once
//     its last dP^T is done, its K once its last dQ is, and the dK / dV write-out
//     of one key tile overlaps the first step of the next.
//  3. bwd_dq_convert -- dq = bf16(scale * accumulator).
#include <cfloat>
#include <cmath>

#include <algorithm>
#include <mutex>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int NC = D / 64;
  static constexpr uint32_t TILE = 128u * D * 2u;  // one 128 x D bf16 tile
  static constexpr int NQ = 2;                     // Q ring slots
  static constexpr int NDO = (D == 64) ? 2 : 1;    // dO ring slots
  static constexpr uint32_t DS_BYTES = 128u * 128u * 2u;
  static constexpr uint32_t BOX_BYTES = 32u * 32u * 4u;    // one fp32 dQ box: 32 rows x 32 columns
  static constexpr uint32_t STG_BYTES = 4u * 2u * BOX_BYTES;  // two boxes per dQ warp
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  // dQ buffers: with D = 128 dQ is computed over the dP^T columns (TMEM is full),
  // so the next dP^T waits until dQ has been read out; with D = 64 two buffers
  // of their own in the columns left over, so that it does not
  static constexpr int NDQ = (D == 64) ? 2 : 1;
  static constexpr uint32_t t_dq(int b) { return NDQ == 1 ? T_DP : 256u + 2u * D + 64u * (uint32_t)b; }
  static constexpr int KEY_THREADS = 256;  // warps 0-7: P^T / dS^T, epilogue
  static constexpr int DQ_WARP0 = 8;       // warps 8-11: dQ out of TMEM into the accumulator
  static constexpr int DQ_THREADS = 128;
  static constexpr int PRODUCER_WARP = 12, MMA_WARP = 13;  // (warps 14, 15 idle)
  static constexpr int THREADS = 512;
  // registers per thread of each warpgroup after setmaxnreg (launched at 128):
  // key-row warps, dQ warps, producer / MMA warpgroup
  static constexpr uint32_t KEY_REGS = (D == 128) ? 160 : 168, DQ_REGS = 104, PM_REGS = (D == 128) ? 88 : 72;
  static_assert(2 * KEY_REGS + DQ_REGS + PM_REGS == 4 * 128, "the split must add up to the launch's registers");
};

struct TileStats {  // per query tile, from the workspace
  float nlse[128];    // -LSE * log2(e) of the tile's query rows
  float ndelta[128];  // -Delta of the tile's query rows
};

// One work item: the key tile J of head (b, h), with the query tiles of its
// column lists (FULL first, then PARTIAL).
struct BwdItem {
  int J, bh, bm, h, n_full, n;
  int64_t list;  // offset of the column's lists
};

struct BwdCtl {
  alignas(16) TileStats stats;  // of the current step, copied in by the key-row warps
  uint64_t k_full, v_full, k_empty, v_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full[2], do_empty[2];
  uint64_t s_full, dp_full, pa_full, pb_full, acc_full, acc_free, fin;
  uint64_t dq_full[2], dq_free[2];
  // this CTA's items in the order the producer claimed them (see sched_get)
  uint64_t sched_full[4], sched_empty[4];
  int sched_k[4];
  BwdItem sched_it[4];  // and their descriptors, so that no role reloads them from global memory
  uint32_t tmem;
  int abort;
  int32_t arg[2][FA_MAX_MASK_NODES];  // mask program arguments of the current item, per key-row half
};

static_assert(BwdCfg<64>::NQ <= 2 && BwdCfg<64>::NDO <= 2 && BwdCfg<64>::NDQ <= 2 && BwdCfg<128>::NQ <= 2 &&
                  BwdCfg<128>::NDO <= 2 && BwdCfg<128>::NDQ <= 2,
              "BwdCtl holds two barriers per Q, dO and dQ buffer");

template <int D>
constexpr size_t bwd_smem_bytes() {
  using C = BwdCfg<D>;
  return 1024 + (size_t)C::TILE * (2 + C::NQ + C::NDO) + C::DS_BYTES + C::STG_BYTES + sizeof(BwdCtl);
}
static_assert(bwd_smem_bytes<128>() <= 227 * 1024, "backward shared memory");

#ifdef FA_TEST_HOOKS
__device__ int g_hook_skip_first_k;  // see test_hook_backward
#endif

__device__ __forceinline__ void fail(const AttnArgs& p, BwdCtl* ctl) {
  atomicOr(p.status, kStatusTimeout);
  ctl->abort = 1;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  const bool r = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, r);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Writes 32 bf16 values (16 packed words) of row r into a 128-byte-swizzled
// [chunks][128 rows][64] tile at columns [32 c, 32 c + 32).
__device__ __forceinline__ void store_row32(uint8_t* tile, int r, int c, const uint32_t (&w)[16]) {
  uint8_t* row = tile + (c / 2) * 16384 + r * 128;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const int piece = (c % 2) * 4 + q4;
    *reinterpret_cast<uint4*>(row + ((piece ^ (r & 7)) << 4)) =
        make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
  }
}


__device__ __forceinline__ BwdItem bwd_item(const AttnArgs& p, int k) {
  const int rep = (p.B / p.Bm) * (p.H / p.Hm);
  const int col = __ldg(p.col_order + k / rep);  // index into [Bm][Hm][nkv], longest first
  const int t = k % rep;
  BwdItem it;
  it.J = col % p.nkv;
  const int hm = (col / p.nkv) % p.Hm;
  it.bm = col / (p.nkv * p.Hm);
  const int b = (p.Bm == 1) ? t / (p.H / p.Hm) : it.bm;
  it.h = (p.Hm == 1) ? t % (p.H / p.Hm) : hm;
  it.bh = b * p.H + it.h;
  it.n_full = __ldg(p.full_q_num + col);
  it.n = it.n_full + __ldg(p.q_num + col);
  it.list = (int64_t)col * p.nq;
  return it;
}

__device__ __forceinline__ int tile_of(const AttnArgs& p, const BwdItem& it, int s) {
  return s < it.n_full ? __ldg(p.full_q_idx + it.list + s) : __ldg(p.q_idx + it.list + s - it.n_full);
}

// Dynamic schedule: the CTAs claim items from one counter in the longest-first
// order, so that each takes the next item when its last one is done (the
// greedy longest-processing-time rule: a few very long columns, such as the
// sink tokens' column that every query tile sees, no longer pile up on the
// CTAs that a static round robin gives them to).  Only items with at least one
// visible query tile are handed out; the key tiles of the others get zero dK /
// dV from bwd_pre.
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 4 + 8;  // MMA thread, dQ warps, key-row warps (one arrival per warp)

__device__ __forceinline__ int claim_live(const AttnArgs& p, uint32_t* sched, int items, BwdItem& it) {
  while (true) {
    const int k = (int)atomicAdd(sched, 1u);
    if (k >= items) return items;
    it = bwd_item(p, k);
    if (it.n > 0) return k;
  }
}

template <int D, int SCORE, bool PGRAD>
__global__ void __launch_bounds__(512, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
               const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ AttnArgs p,
               const float* __restrict__ stats_g, uint32_t* __restrict__ sched) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::TILE;
  uint8_t* sQ0 = sV + C::TILE;             // Q ring
  uint8_t* sDO0 = sQ0 + C::NQ * C::TILE;   // dO ring
  uint8_t* sDS = sDO0 + C::NDO * C::TILE;
  uint8_t* sSTG = sDS + C::DS_BYTES;       // dQ staging: per dQ warp two 32 x 32 fp32 boxes
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(sSTG + C::STG_BYTES);
  auto sQ = [&](int st) { return sQ0 + st * C::TILE; };
  auto sDO = [&](int st) { return sDO0 + st * C::TILE; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int items = p.B * p.H * p.nkv;  // below 2^31: checked at launch

  const uint32_t b_kf = smem_u32(&ctl->k_full), b_vf = smem_u32(&ctl->v_full), b_ke = smem_u32(&ctl->k_empty),
                 b_ve = smem_u32(&ctl->v_empty), b_s = smem_u32(&ctl->s_full), b_dp = smem_u32(&ctl->dp_full),
                 b_pa = smem_u32(&ctl->pa_full), b_pb = smem_u32(&ctl->pb_full), b_acc = smem_u32(&ctl->acc_full),
                 b_accf = smem_u32(&ctl->acc_free), b_fin = smem_u32(&ctl->fin);
  if (threadIdx.x == 0) {
    mbar_init(b_kf, 1);
    mbar_init(b_vf, 1);
    mbar_init(b_ke, 1);
    mbar_init(b_ve, 1);
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(smem_u32(&ctl->q_full[s2]), 1);
      mbar_init(smem_u32(&ctl->q_empty[s2]), 1);
      mbar_init(smem_u32(&ctl->do_full[s2]), 1);
      mbar_init(smem_u32(&ctl->do_empty[s2]), 1);
    }
    mbar_init(b_s, 1);
    mbar_init(b_dp, 1);
    mbar_init(b_pa, C::KEY_THREADS);
    mbar_init(b_pb, C::KEY_THREADS);
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(smem_u32(&ctl->dq_full[b2]), 1);
      mbar_init(smem_u32(&ctl->dq_free[b2]), C::DQ_THREADS);
    }
    mbar_init(b_acc, 1);
    mbar_init(b_accf, C::DQ_THREADS);
    mbar_init(b_fin, 1);
    for (int sl = 0; sl < kSchedSlots; ++sl) {
      mbar_init(smem_u32(&ctl->sched_full[sl]), 1);
      mbar_init(smem_u32(&ctl->sched_empty[sl]), kSchedConsumers);
    }
    ctl->abort = (*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == C::PRODUCER_WARP) {
    tmem_alloc(smem_u32(&ctl->tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const bool skip = ctl->abort != 0;

  // Item u of this CTA's sequence (u = 0, 1, ...; `items` ends it), as the
  // producer published it; false when the wait gave up.  Every consumer role
  // releases slot u once it is done with item u.
  auto sched_get = [&](int u, int& k, BwdItem& it) -> bool {
    const int sl = u % kSchedSlots;
    if (!mbar_wait(smem_u32(&ctl->sched_full[sl]), (u / kSchedSlots) & 1, &ctl->abort)) return false;
    k = *reinterpret_cast<volatile int*>(&ctl->sched_k[sl]);
    it = ctl->sched_it[sl];  // read after the wait (a memory clobber): the producer's values
    return true;
  };
  auto sched_get_warp = [&](int u, int& k, BwdItem& it) -> bool {
    const bool r = __all_sync(0xffffffffu, sched_get(u, k, it));
    return r;
  };
  auto sched_release = [&](int u) { mbar_arrive(smem_u32(&ctl->sched_empty[u % kSchedSlots])); };

  // teardown, at the end of every role: all threads past their last TMEM
  // access, then the allocating warp frees the columns
  auto teardown = [&]() {
    tc_fence_before();
    named_bar_sync(15, C::THREADS);
    if (warp == C::PRODUCER_WARP) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  };

  // The CTA stays resident and takes the items its producer claims; every role
  // walks that sequence through the item ring.  Steps (I, J) are numbered
  // across items (g) for the per-step barriers and the Q / dO rings; items are
  // numbered (u) for the ring, the K / V buffers and the dK / dV accumulators.
  //
  // Register budgets per warpgroup, set at the top of each warpgroup's branch
  // (launched with 128 per thread; BwdCfg): key-row warps 160 (D = 128) or 168,
  // dQ warps 104, producer / MMA warpgroup 88 or 72 (the item claims and the item
  // ring need more than the 48 it had before) -- 256 x 160 + 128 x 104 + 128 x 88
  // = 256 x 168 + 128 x 104 + 128 x 72 = 512 x 128.
  if (warp >= C::PRODUCER_WARP) {
    setmaxnreg_dec<C::PM_REGS>();
    if (warp == C::PRODUCER_WARP) {
      // ------------------------------------------------------------ producer
      // Per item: V once dP of the last item's last step is done with it, then
      // the step's Q and dO, and K once dQ of the last item's last step is.
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
      }
      int g = 0, q_issued = 0, do_issued = 0, v_issued = 0, k_issued = 0;
      int u = 0;
      bool ok = true;
      // claims the next live item (lane 0) and publishes it as item uu
      auto claim_publish = [&](int uu) -> int {
        int kc = items;
        BwdItem it{};
        if (lane == 0 && !skip) kc = claim_live(p, sched, items, it);
        kc = __shfl_sync(0xffffffffu, kc, 0);
        const int sl = uu % kSchedSlots;
        if (uu >= kSchedSlots &&
            !warp_wait(smem_u32(&ctl->sched_empty[sl]), (uu / kSchedSlots - 1) & 1, &ctl->abort))
          return -1;
        if (lane == 0) {
          ctl->sched_k[sl] = kc;
          ctl->sched_it[sl] = it;
          mbar_arrive(smem_u32(&ctl->sched_full[sl]));
        }
        return kc;
      };
      // Items are claimed two ahead: item u + 2 once item u's first loads are
      // issued, so that the claim's latency (an atomic, then the item's counts)
      // stays off the path to those loads; the consumers look one item ahead.
      int k = claim_publish(0);
      int kn = items;
      ok = k >= 0;
      if (ok && k < items) {
        kn = claim_publish(1);
        ok = kn >= 0;
      }
      while (ok && k < items) {
        __syncwarp();
        const BwdItem cur = ctl->sched_it[u % kSchedSlots];  // as lane 0 published it
        int kn2 = items;  // item u + 2
        if (u > 0 && !warp_wait(b_ve, (u - 1) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(b_vf, C::TILE);
          for (int c = 0; c < C::NC; ++c) tma_load_3d(smem_u32(sV + c * 16384), &tm_v, b_vf, c * 64, cur.J * 128, cur.bh);
        }
        v_issued = u + 1;
        for (int s = 0; s < cur.n; ++s, ++g) {
          const int I = tile_of(p, cur, s);
          // Q slot (freed by the MMA warp once dK, its last reader, is done)
          const int qs = g % C::NQ, quse = g / C::NQ;
          if (quse > 0 && !warp_wait(smem_u32(&ctl->q_empty[qs]), (quse - 1) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t qbar = smem_u32(&ctl->q_full[qs]);
            mbar_arrive_expect_tx(qbar, C::TILE);
            for (int c = 0; c < C::NC; ++c) tma_load_3d(smem_u32(sQ(qs) + c * 16384), &tm_q, qbar, c * 64, I * 128, cur.bh);
          }
          q_issued = g + 1;
          // dO slot (freed once dV, its last reader, is done)
          const int ds = g % C::NDO, duse = g / C::NDO;
          if (duse > 0 && !warp_wait(smem_u32(&ctl->do_empty[ds]), (duse - 1) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t dbar = smem_u32(&ctl->do_full[ds]);
            mbar_arrive_expect_tx(dbar, C::TILE);
            for (int c = 0; c < C::NC; ++c)
              tma_load_3d(smem_u32(sDO(ds) + c * 16384), &tm_do, dbar, c * 64, I * 128, cur.bh);
          }
          do_issued = g + 1;
          if (s == 0) {
            if (u > 0 && !warp_wait(b_ke, (u - 1) & 1, &ctl->abort)) {
              ok = false;
              break;
            }
#ifdef FA_TEST_HOOKS
            const bool hook_skip = g_hook_skip_first_k != 0 && blockIdx.x == 0 && u == 0;
#else
            constexpr bool hook_skip = false;
#endif
            if (lane == 0 && !hook_skip) {
              mbar_arrive_expect_tx(b_kf, C::TILE);
              for (int c = 0; c < C::NC; ++c)
                tma_load_3d(smem_u32(sK + c * 16384), &tm_k, b_kf, c * 64, cur.J * 128, cur.bh);
            }
            k_issued = u + 1;
            if (kn < items) {  // item u + 2 (after the end marker nothing more is read)
              kn2 = claim_publish(u + 2);
              if (kn2 < 0) {
                ok = false;
                break;
              }
            }
          }
        }
        k = kn;
        kn = kn2;
        ++u;
      }
      if (!ok && lane == 0) fail(p, ctl);
      // drain: every copy this CTA started lands before it exits (each buffer's
      // earlier loads were waited for before the last one was issued)
      if (lane == 0) {
        if (v_issued > 0) mbar_wait(b_vf, (v_issued - 1) & 1, nullptr);
        if (k_issued > 0) mbar_wait(b_kf, (k_issued - 1) & 1, nullptr);
        for (int s = max(0, q_issued - C::NQ); s < q_issued; ++s)
          mbar_wait(smem_u32(&ctl->q_full[s % C::NQ]), (s / C::NQ) & 1, nullptr);
        for (int s = max(0, do_issued - C::NDO); s < do_issued; ++s)
          mbar_wait(smem_u32(&ctl->do_full[s % C::NDO]), (s / C::NDO) & 1, nullptr);
      }
    } else if (warp == C::MMA_WARP) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t kIdKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t kIdKM = idesc_bf16(128, D, false, true);     // dV (A in TMEM), dK
        constexpr uint32_t kIdMM = idesc_bf16(128, D, true, true);      // dQ
        // Where the next step's S^T goes in the MMA order.  Each step's chain
        // runs dS -> dQ -> dQ read out of TMEM -> next dP^T -> next dS, with
        // phase A off it; with D = 128 the S^T MMA goes after dQ so as not to
        // delay that chain, with D = 64 (shorter MMAs) right after dV, so that
        // phase A of the next step can start as soon as dS is in (measured
        // faster each way on the packed-document workloads).
        constexpr bool kEarlyS = (D == 64);
        const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV), ds_base = smem_u32(sDS);
        // S^T = K Q^T of step g (step s of item u), into columns the dV MMA of
        // the step before has read
        auto issue_s = [&](int g, int s, int u) -> bool {
          const int qs = g % C::NQ;
          if (s == 0 && !mbar_wait(b_kf, u & 1, &ctl->abort)) return false;
          if (!mbar_wait(smem_u32(&ctl->q_full[qs]), (g / C::NQ) & 1, &ctl->abort)) return false;
          tc_fence_after();
          const uint64_t a0 = opaque(sdesc_sw128(k_base, 16, 1024)), b0 = opaque(sdesc_sw128(smem_u32(sQ(qs)), 16, 1024));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + C::T_S, kmajor_step(a0, kk), kmajor_step(b0, kk), kIdKK, kk > 0);
          mma_commit(b_s);
          return true;
        };
        // dP^T = V dO^T of step g; with one dQ buffer it goes into the columns dQ
        // of the step before was computed in, and waits until the dQ warps have
        // read that dQ out.  The item's last dP^T is the last reader of V.
        auto issue_dp = [&](int g, int s, int n, int u) -> bool {
          const int ds = g % C::NDO;
          if (s == 0 && !mbar_wait(b_vf, u & 1, &ctl->abort)) return false;
          if (!mbar_wait(smem_u32(&ctl->do_full[ds]), (g / C::NDO) & 1, &ctl->abort)) return false;
          if (C::NDQ == 1 && g > 0 && !mbar_wait(smem_u32(&ctl->dq_free[0]), (g - 1) & 1, &ctl->abort)) return false;
          tc_fence_after();
          const uint64_t a0 = opaque(sdesc_sw128(v_base, 16, 1024)), b0 = opaque(sdesc_sw128(smem_u32(sDO(ds)), 16, 1024));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + C::T_DP, kmajor_step(a0, kk), kmajor_step(b0, kk), kIdKK, kk > 0);
          mma_commit(b_dp);
          if (s == n - 1) mma_commit(b_ve);
          return true;
        };
        int g = 0, u = 0, k = items;
        BwdItem cur, nxt;
        bool ok = sched_get(0, k, cur);
        while (ok && k < items) {
          const int n = cur.n;
          if (!issue_s(g, 0, u) || !issue_dp(g, 0, n, u)) {
            ok = false;
            break;
          }
          int kn = items;
          if (!sched_get(u + 1, kn, nxt)) {
            ok = false;
            break;
          }
          for (int s = 0; s < n; ++s, ++g) {
            const int qs = g % C::NQ, ds = g % C::NDO;
            const uint32_t q_base = smem_u32(sQ(qs)), do_base = smem_u32(sDO(ds));
            if (!mbar_wait(b_pa, g & 1, &ctl->abort)) {
              ok = false;
              break;
            }
            // the dV / dK accumulators of the last item have been read out
            if (s == 0 && u > 0 && !mbar_wait(b_accf, (u - 1) & 1, &ctl->abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // dV += P^T dO; P^T of query columns [64 h, 64 h + 64) sits at TMEM columns [64 h, 64 h + 32).
            // It runs while the key-row warps compute dS.
            {
              const uint64_t b0 = opaque(sdesc_sw128(do_base, 16384, 1024));
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts(tmem + C::T_DV, tmem + C::T_S + (kk / 4) * 64 + (kk % 4) * 8, mnmajor_step(b0, kk), kIdKM,
                       (s > 0 || kk > 0));
            }
            mma_commit(smem_u32(&ctl->do_empty[ds]));
            if (kEarlyS && s + 1 < n && !issue_s(g + 1, s + 1, u)) {
              ok = false;
              break;
            }
            if (!mbar_wait(b_pb, g & 1, &ctl->abort)) {
              ok = false;
              break;
            }
            // with two dQ buffers, this step's has been read out two steps ago
            if (C::NDQ == 2 && g >= 2 &&
                !mbar_wait(smem_u32(&ctl->dq_free[g & 1]), ((g >> 1) - 1) & 1, &ctl->abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            {  // dQ = dS K (one buffer: over the dP^T columns the key-row warps have read)
              const uint64_t a0 = opaque(sdesc_sw128(ds_base, 16384, 1024)), b0 = opaque(sdesc_sw128(k_base, 16384, 1024));
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem + C::t_dq(g % C::NDQ), mnmajor_step(a0, kk), mnmajor_step(b0, kk), kIdMM, kk > 0);
            }
            mma_commit(smem_u32(&ctl->dq_full[g % C::NDQ]));
            if (!kEarlyS && s + 1 < n && !issue_s(g + 1, s + 1, u)) {
              ok = false;
              break;
            }
            if (s + 1 == n) mma_commit(b_ke);  // K read for the last time in this item
            {  // dK += dS^T Q
              const uint64_t a0 = opaque(sdesc_sw128(ds_base, 16, 1024)), b0 = opaque(sdesc_sw128(q_base, 16384, 1024));
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem + C::T_DK, kmajor_step(a0, kk), mnmajor_step(b0, kk), kIdKM, (s > 0 || kk > 0));
            }
            mma_commit(smem_u32(&ctl->q_empty[qs]));  // Q read for the last time
            if (s + 1 < n && !issue_dp(g + 1, s + 1, n, u)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          mma_commit(b_acc);  // dV, dK of the item complete
          sched_release(u);
          k = kn;
          cur = nxt;
          ++u;
        }
        if (!ok) fail(p, ctl);
        mma_commit(b_fin);
        mbar_wait(b_fin, 0, nullptr);
      }
    }
    __syncwarp();
    teardown();
  } else if (warp >= C::DQ_WARP0) {
    setmaxnreg_dec<C::DQ_REGS>();
    // ------------------------------------------------------------ dQ warps
    // Warp w drains dQ rows [32 (w % 4), +32) (its TMEM lanes) of each step:
    // 32 columns at a time into one of its two 128-byte-swizzled 32 x 32 fp32
    // boxes, which lane 0 TMA bulk reduce-adds into the fp32 accumulator.  A
    // box is rewritten only once the bulk copy issued from it two rounds before
    // has read it.  After an item's last step the same rows of dV and
    // scale * dK leave TMEM through the same boxes (as 32 x 64 bf16) by TMA
    // store.
    const int rw = (warp % 4) * 32;  // first dQ / key row of this warp
    const uint32_t t_lane = tmem + ((uint32_t)rw << 16);
    uint8_t* box0 = sSTG + (warp % 4) * (2 * C::BOX_BYTES);
    int round = 0, u = 0, g = 0, k = items;
    BwdItem cur;
    bool ok = sched_get_warp(0, k, cur);
    while (ok && k < items) {
      for (int s = 0; s < cur.n; ++s, ++g) {
        const int I = tile_of(p, cur, s);
        const int bq = g % C::NDQ;
        if (!warp_wait(smem_u32(&ctl->dq_full[bq]), (g / C::NDQ) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tq = t_lane + C::t_dq(bq);
#pragma unroll 1
        for (int h2 = 0; h2 < D / 64; ++h2) {
          float v[64];
          tmem_ld64f(tq + 64 * h2, v);
          if (h2 == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl->dq_free[bq]));  // TMEM columns free for the next dP^T / dQ
          }
#pragma unroll
          for (int bx = 0; bx < 2; ++bx, ++round) {
            uint8_t* box = box0 + (round & 1) * C::BOX_BYTES;
            if (lane == 0) bulk_wait_read1();  // the copy from this box two rounds ago has read it
            __syncwarp();
            uint8_t* rowp = box + lane * 128;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              *reinterpret_cast<float4*>(rowp + ((q4 ^ (lane & 7)) << 4)) =
                  make_float4(v[32 * bx + 4 * q4], v[32 * bx + 4 * q4 + 1], v[32 * bx + 4 * q4 + 2],
                              v[32 * bx + 4 * q4 + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d(&tm_dq, smem_u32(box), 64 * h2 + 32 * bx, I * 128 + rw, cur.bh);
              bulk_commit();
            }
          }
        }
      }
      if (!ok) break;
      // dV, then scale * dK, 64 columns at a time; the accumulators are free for
      // the next item once the last columns are read
      if (!warp_wait(b_acc, u & 1, &ctl->abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2 * (D / 64); ++c, ++round) {
        const bool is_k = c >= D / 64;
        const int h2 = is_k ? c - D / 64 : c;
        float a[64];
        tmem_ld64f(t_lane + (is_k ? C::T_DK : C::T_DV) + 64 * h2, a);
        if (c == 2 * (D / 64) - 1) {
          tc_fence_before();
          mbar_arrive(b_accf);
        }
        const float sc = is_k ? p.scale : 1.0f;
        uint8_t* box = box0 + (round & 1) * C::BOX_BYTES;
        if (lane == 0) bulk_wait_read1();
        __syncwarp();
        uint8_t* rowp = box + lane * 128;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<uint4*>(rowp + ((q4 ^ (lane & 7)) << 4)) =
              make_uint4(pack_bf16x2(a[8 * q4] * sc, a[8 * q4 + 1] * sc), pack_bf16x2(a[8 * q4 + 2] * sc, a[8 * q4 + 3] * sc),
                         pack_bf16x2(a[8 * q4 + 4] * sc, a[8 * q4 + 5] * sc), pack_bf16x2(a[8 * q4 + 6] * sc, a[8 * q4 + 7] * sc));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(is_k ? &tm_dk : &tm_dv, smem_u32(box), 64 * h2, cur.J * 128 + rw, cur.bh);
          bulk_commit();
        }
      }
      __syncwarp();
      if (lane == 0) sched_release(u);
      ++u;
      ok = sched_get_warp(u, k, cur);
    }
    if (!ok) fail(p, ctl);
    if (lane == 0) bulk_wait0();  // every reduce and store of this warp has completed
    __syncwarp();
    teardown();
  } else {
    setmaxnreg_inc<C::KEY_REGS>();
    // ------------------------------------------------------------ key-row warps
    // Thread (warp w, lane) owns TMEM lane r = 32 (w % 4) + lane = key row r, of
    // which it handles query columns [64 half, 64 half + 64) (half = w / 4).
    const int r = (warp % 4) * 32 + lane;
    const int half = warp / 4;
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S, tP = tmem + lane_off + C::T_DP;
    const uint64_t mask_ops = pack_ops(p.mask);
    const int qoff = (int)p.mask.q_off;  // query row i is position i + qoff (below 2^31: checked on the host)
    const float sc_l2 = p.scale * kLog2e;
    float cap_l2 = 0.f, sc_cap2 = 0.f;
    if constexpr (SCORE == FA_S_SOFTCAP) {
      const float cap = __ldg(p.score_param);
      cap_l2 = cap * kLog2e;
      sc_cap2 = (p.scale / cap) * (2.0f * kLog2e);  // S -> the exponent of e^{2 x / c}, base 2
    }
    // -LSE (log2 units) and -Delta of the query columns this half handles: one
    // value per thread of the half, copied into shared memory once per step;
    // the mask program's arguments (per mask batch), once per item
    const int st_idx = (r < 64) ? (64 * half + r) : (128 + 64 * half + r - 64);
    auto stat_of = [&](int bh, int I) { return __ldg(stats_g + ((int64_t)bh * p.nq + I) * 256 + st_idx); };
    int32_t* arg_s = ctl->arg[half];
    int k = items, I_next = 0;  // the query tile of the next step
    BwdItem cur, nxt;
    bool ok = sched_get_warp(0, k, cur), lok = true;
    if (ok && k < items) {
      const BwdItem& it0 = cur;
      I_next = tile_of(p, it0, 0);
      reinterpret_cast<float*>(&ctl->stats)[st_idx] = stat_of(it0.bh, I_next);
      if (r < p.mask.n) arg_s[r] = node_arg(p.mask, r, it0.bm);
    }
    int g = 0, u = 0;
    while (ok && k < items) {
      // of the next item only what the last step hands over: its first query
      // tile (for the stats), head and mask batch
      int kn = items, nxt_i0 = 0, nxt_bh = 0, nxt_bm = 0;
      if (!sched_get_warp(u + 1, kn, nxt)) {
        ok = false;
        break;
      }
      if (kn < items) {
        nxt_i0 = tile_of(p, nxt, 0);
        nxt_bh = nxt.bh;
        nxt_bm = nxt.bm;
      }
      const int n = cur.n, bh = cur.bh;
      const int j = cur.J * 128 + r;  // key row
      // this key's visible query rows as two intervals, when they are; the
      // document id and run of the key only where they are not, for the
      // per-word evaluation of the program
      const int4 seg = __ldg(p.row_segs + ((int64_t)cur.bm * 2 + 1) * p.seg_len + min(j, p.kv_len - 1));
      const int32_t* doc_row = p.mask.has_doc ? p.mask.doc + (int64_t)cur.bm * p.mask.doc_len : nullptr;
      int32_t doc_j = 0;
      int run_lo = 0, run_hi = 0;  // with sorted ids: doc[i] == doc[j] exactly for i in [run_lo, run_hi)
      bool use_run = false;
      if (seg.x < 0 && doc_row != nullptr) {
        doc_j = __ldg(doc_row + min(j, p.kv_len - 1));
        use_run = doc_run(p.mask, cur.bm, min(j, p.kv_len - 1), run_lo, run_hi);
      }
      float slope_l2 = 0.f;
      if constexpr (SCORE == FA_S_ALIBI) slope_l2 = __ldg(p.score_param + cur.h) * kLog2e;
      const float* bias_h = nullptr;  // RELBIAS: this head's table
      if constexpr (SCORE == FA_S_RELBIAS) bias_h = p.score_param + (int64_t)cur.h * p.bias_len;
      const bool row_ok = j < p.kv_len;
      float2 pacc = make_float2(0.f, 0.f);  // PGRAD: this thread's share of dL/dslope[h] in this item
      for (int s = 0; s < n; ++s, ++g) {
        // collective per half: this step's stats are in place, and every wait of
        // the last step succeeded for all of the half (a failed wait is acted on
        // here; until then the thread goes on with whatever TMEM holds, writing
        // only TMEM and shared memory)
        ok = named_bar_and(2 + half, 128, lok);
        if (!ok) break;
        const int I = I_next;
        float st_next = 0.f;
        if (s + 1 < n) {
          I_next = tile_of(p, cur, s + 1);
          st_next = stat_of(bh, I_next);
        } else if (kn < items) {
          I_next = nxt_i0;
          st_next = stat_of(nxt_bh, nxt_i0);
        }
        const bool partial = s >= cur.n_full;
        // visibility words of this thread's two 32-column chunks, built before S^T is waited for
        uint32_t wm0 = row_ok ? 0xffffffffu : 0u, wm1 = wm0;
        if (partial && row_ok && seg.x >= 0) {
          wm0 = seg_word(seg, I * 128 + 64 * half);
          wm1 = seg_word(seg, I * 128 + 64 * half + 32);
        } else if (partial && row_ok) {
#pragma unroll 1
          for (int c2 = 0; c2 < 2; ++c2) {
            const int i0 = I * 128 + 32 * (2 * half + c2);
            const int ip0 = i0 + qoff;  // the rows' positions (query row i is position i + q_off)
            auto eq = [&]() {
              if (use_run) return range_bits(run_lo, run_hi, ip0);
              uint32_t bits = 0;
              if (i0 + 32 <= p.q_len && p.mask.doc_vec_ok && (qoff & 3) == 0) {  // 16-byte aligned rows
                const int4* dv = reinterpret_cast<const int4*>(doc_row + ip0);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  const int4 d = __ldg(dv + q4);
                  bits |= (uint32_t)(d.x == doc_j) << (4 * q4) | (uint32_t)(d.y == doc_j) << (4 * q4 + 1) |
                          (uint32_t)(d.z == doc_j) << (4 * q4 + 2) | (uint32_t)(d.w == doc_j) << (4 * q4 + 3);
                }
              } else {
                const int in = min(i0 + 32, p.q_len);
                for (int i = i0; i < in; ++i)
                  bits |= (uint32_t)(__ldg(doc_row + i + qoff) == doc_j) << (uint32_t)(i - i0);
              }
              return bits;
            };
            const uint32_t w = mask_word_t_rolled(p.mask.n, mask_ops, arg_s, j, ip0, eq);
            wm0 = (c2 == 0) ? w : wm0;
            wm1 = (c2 == 1) ? w : wm1;
          }
        }
        const float* nlse_s = ctl->stats.nlse;
        const float* ndel_s = ctl->stats.ndelta;
        // -- phase A: P = exp2(s - LSE) over this thread's 64 query columns; P^T
        //    (bf16) over the S^T columns already read, for the dV MMA.  pg keeps
        //    P times the score mod's derivative (P itself unless soft-capped).
        lok = warp_wait(b_s, g & 1, &ctl->abort);
        tc_fence_after();
        float pg[64];
        // ALiBi, log2 units: -slope (i + qoff - j) = -slope (i - 128 I) + slope (j - 128 I - qoff)
        float bj = 0.f;
        if constexpr (SCORE == FA_S_ALIBI) bj = slope_l2 * (float)(j - (I * 128 + qoff));
        // learned bias: query column x of the tile (0..127) takes entry clamp(bq + x, 0, L - 1),
        // bq = 128 I + q_offset - j - d0 held within [-128, L] (which changes no entry)
        int bq = 0;
        if constexpr (SCORE == FA_S_RELBIAS)
          bq = (int)max((int64_t)-128, min((int64_t)I * 128 + qoff - j - p.bias_d0, (int64_t)p.bias_len));
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * half + c2;  // 32-column chunk of the 128 query columns
          const uint32_t w = (c2 == 0) ? wm0 : wm1;
          float sv[32];
          tmem_ld32f(tS + 32 * c, sv);
          uint32_t pk[16];
          const float4* nl4 = reinterpret_cast<const float4*>(nlse_s + 32 * c);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float4 nlq = nl4[e / 4];
            const float2 nl = (e % 4 == 0) ? make_float2(nlq.x, nlq.y) : make_float2(nlq.z, nlq.w);
            float2 a, gd = make_float2(1.0f, 1.0f);
            if constexpr (SCORE == FA_S_SOFTCAP) {
              // tanh(t) = 1 - 2 r with r = 1 / (1 + e^{2t}): the score c tanh(x / c) log2(e)
              // = c log2(e) - 2 c log2(e) r (the stats carry the c log2(e)), and
              // 1 - tanh^2 = 4 r (1 - r); packed in pairs
              const float2 u = mul2(make_float2(sv[e], sv[e + 1]), make_float2(sc_cap2, sc_cap2));
              const float2 d = add2(make_float2(ex2_approx(u.x), ex2_approx(u.y)), make_float2(1.0f, 1.0f));
              const float2 rr = make_float2(rcp_approx(d.x), rcp_approx(d.y));
              a = fma2(rr, make_float2(-2.0f * cap_l2, -2.0f * cap_l2), nl);
              gd = mul2(fma2(make_float2(-rr.x, -rr.y), rr, rr), make_float2(4.0f, 4.0f));
            } else if constexpr (SCORE == FA_S_ALIBI) {
              // the stats carry -slope (i - 128 I) of each query row; the key's part is bj
              a = fma2(make_float2(sv[e], sv[e + 1]), make_float2(sc_l2, sc_l2), add2(nl, make_float2(bj, bj)));
            } else if constexpr (SCORE == FA_S_RELBIAS) {
              const int x = 32 * c + e;
              const float2 bv = make_float2(__ldg(bias_h + min(max(bq + x, 0), p.bias_len - 1)),
                                            __ldg(bias_h + min(max(bq + x + 1, 0), p.bias_len - 1)));
              a = fma2(make_float2(sv[e], sv[e + 1]), make_float2(sc_l2, sc_l2),
                       fma2(bv, make_float2(kLog2e, kLog2e), nl));
            } else {
              a = fma2(make_float2(sv[e], sv[e + 1]), make_float2(sc_l2, sc_l2), nl);
            }
            float2 pv;
            pv.x = ((w >> e) & 1u) ? ex2_approx(a.x) : 0.f;
            pv.y = ((w >> (e + 1)) & 1u) ? ex2_approx(a.y) : 0.f;
            pk[e / 2] = pack_bf16x2(pv.x, pv.y);
            if constexpr (SCORE == FA_S_SOFTCAP) pv = mul2(pv, gd);
            pg[32 * c2 + e] = pv.x;
            pg[32 * c2 + e + 1] = pv.y;
          }
          tmem_st16(tS + 64 * half + 16 * c2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_pa);
        // -- phase B: dS = P (dP - Delta) [* d softcap], K-major into the dS buffer
        //    (free: dP^T of this step was issued after dK of the step before)
        lok = warp_wait(b_dp, g & 1, &ctl->abort) && lok;
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * half + c2;
          float dp[32];
          tmem_ld32f(tP + 32 * c, dp);
          uint32_t dk[16];
          const float4* nd4 = reinterpret_cast<const float4*>(ndel_s + 32 * c);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float4 ndq = nd4[e / 4];
            const float2 nd = (e % 4 == 0) ? make_float2(ndq.x, ndq.y) : make_float2(ndq.z, ndq.w);
            const float2 dsv = mul2(make_float2(pg[32 * c2 + e], pg[32 * c2 + e + 1]),
                                    add2(make_float2(dp[e], dp[e + 1]), nd));
            dk[e / 2] = pack_bf16x2(dsv.x, dsv.y);
            if constexpr (PGRAD) {  // kept for the parameter gradient below
              pg[32 * c2 + e] = dsv.x;
              pg[32 * c2 + e + 1] = dsv.y;
            }
          }
          store_row32(sDS, r, c, dk);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(b_pb);
        if constexpr (PGRAD && SCORE == FA_S_RELBIAS) {
          // dL/dbias[h][t] += dS of every pair mapped to entry t (ds/dbias = 1), once
          // dS is handed over; for one column the 32 lanes' entries are consecutive
          float* gh = p.param_grad + (int64_t)cur.h * p.bias_len;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (pg[e] != 0.f) atomicAdd(gh + min(max(bq + 64 * half + e, 0), p.bias_len - 1), pg[e]);
        }
        if constexpr (PGRAD && SCORE == FA_S_ALIBI) {
          // dL/dslope += dS * ds/dslope, ds/dslope = -(i - j) = j - i, once dS is
          // handed over (the dQ MMA does not wait for it)
          const float jb = (float)(j - (I * 128 + 64 * half + qoff));  // j - i of this half's first column (exact)
#pragma unroll
          for (int e = 0; e < 64; e += 2)
            pacc = fma2(make_float2(pg[e], pg[e + 1]), make_float2(jb - (float)e, jb - (float)(e + 1)), pacc);
        }
        // every thread of this half is done with this step's stats (and the
        // item's mask arguments): publish the next step's
        named_bar_sync(2 + half, 128);
        if (s + 1 < n || kn < items) reinterpret_cast<float*>(&ctl->stats)[st_idx] = st_next;
        if (s + 1 == n && kn < items && r < p.mask.n) arg_s[r] = node_arg(p.mask, r, nxt_bm);
      }
      if constexpr (PGRAD && SCORE == FA_S_ALIBI) {
        // the item's part of dL/dslope[h]: one atomic per warp (ok is uniform per half)
        if (ok) {
          float sum = pacc.x + pacc.y;
#pragma unroll
          for (int d = 16; d >= 1; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
          if (lane == 0 && sum != 0.f) atomicAdd(p.param_grad + cur.h, sum);
        }
      }
      __syncwarp();
      if (lane == 0) sched_release(u);
      k = kn;
      cur = nxt;
      ++u;
    }
    if (ok && !lok) ok = false;
    if (!ok) fail(p, ctl);
    teardown();
  }
}

// Per query row: -LSE * log2(e) and -Delta (Delta_i = dO_i . out_i, fp32)
// into the per-tile stats array [B*H][nq][2][128] -- with ALiBi the first also
// carries the query row's part of the bias within its tile, -slope_h (i - 128 I)
// log2(e), so that the main kernel adds only the key's part, and with the
// soft-cap the constant term c log2(e) of c tanh(x / c) log2(e) -- zero for the rows past
// q_len in the last tile; the fp32 dq accumulator rows, the score parameter's
// gradient (if requested) and the main kernel's item counter set to zero.
// D / 16 threads per row, each with two 16-byte loads of out and of dO in
// flight (256 / (D / 16) rows per 256-thread block: enough bytes in flight
// per SM for the HBM roof); the blocks after the rows' take one key tile
// (b, h, J) each and write zero dK and dV for a key tile
// that no query tile sees (the main kernel hands out only the others).
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ AttnArgs p,
                                                      const __nv_bfloat16* __restrict__ out,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const float* __restrict__ lse, float* __restrict__ stats,
                                                      float* __restrict__ dq_acc, int64_t rows, int64_t row_blocks,
                                                      float* __restrict__ param_grad, int64_t n_param_grad,
                                                      uint32_t* __restrict__ sched, __nv_bfloat16* __restrict__ dk,
                                                      __nv_bfloat16* __restrict__ dv) {
  const int q_len = p.q_len, nq = p.nq;
  // the main kernel adds into them
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_param_grad; k += (int64_t)gridDim.x * blockDim.x)
    param_grad[k] = 0.f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;
  if ((int64_t)blockIdx.x >= row_blocks) {
    const int64_t t = (int64_t)blockIdx.x - row_blocks;  // (b * H + h) * nkv + J
    const int J = (int)(t % p.nkv);
    const int bh = (int)(t / p.nkv), b = bh / p.H, h = bh % p.H;
    const int64_t col = ((int64_t)(p.Bm == 1 ? 0 : b) * p.Hm + (p.Hm == 1 ? 0 : h)) * p.nkv + J;
    if (__ldg(p.q_num + col) + __ldg(p.full_q_num + col) != 0) return;
    const int64_t r0 = (int64_t)J * 128, r1 = min((int64_t)p.kv_len, r0 + 128);
    const int64_t n8 = (r1 - r0) * D / 8;  // 16-byte pieces of each tensor's rows
    uint4* zk = reinterpret_cast<uint4*>(dk + ((int64_t)bh * p.kv_len + r0) * D);
    uint4* zv = reinterpret_cast<uint4*>(dv + ((int64_t)bh * p.kv_len + r0) * D);
    for (int64_t k = threadIdx.x; k < n8; k += blockDim.x) {
      zk[k] = make_uint4(0u, 0u, 0u, 0u);
      zv[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  constexpr int E = 16;        // elements per thread: two 16-byte pieces of each tensor
  constexpr int TPR = D / E;   // threads per row
  constexpr int RPB = 256 / TPR;
  const int64_t row = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR;
  const int t = threadIdx.x % TPR;
  float acc = 0.f;
  if (row < rows) {
    const uint4* o = reinterpret_cast<const uint4*>(out + row * D + t * E);
    const uint4* g = reinterpret_cast<const uint4*>(dout + row * D + t * E);
    const uint4 o0 = __ldg(o), o1 = __ldg(o + 1), g0 = __ldg(g), g1 = __ldg(g + 1);
    const uint32_t ow[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
    const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
      const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
      acc = fmaf(a.x, c.x, fmaf(a.y, c.y, acc));
    }
    if (!p.acc_zeroed) {  // (else a forward that prepared the workspace cleared it)
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D + t * E);
#pragma unroll
      for (int e = 0; e < E / 4; ++e) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int d = TPR / 2; d >= 1; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
  if (row < rows && t == 0) {
    const int64_t bh = row / q_len;
    const int i = (int)(row % q_len);
    float* st = stats + (bh * nq + i / 128) * 256;
    float nl = -__ldg(lse + row) * kLog2e;
    if (p.score_op == FA_S_ALIBI) nl -= (__ldg(p.score_param + (int)(bh % p.H)) * kLog2e) * (float)(i % 128);
    if (p.score_op == FA_S_SOFTCAP) nl += __ldg(p.score_param) * kLog2e;  // the soft-cap's constant term
    st[i % 128] = nl;
    st[128 + i % 128] = -acc;
    if (i == q_len - 1)  // rows past q_len in the last tile
      for (int k = i % 128 + 1; k < 128; ++k) st[k] = st[128 + k] = 0.f;
  }
}

// dq = bf16(scale * accumulator), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                             __nv_bfloat16* __restrict__ dq, int64_t n8,
                                                             float scale) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * k];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * k + 1];
  uint4 o;
  o.x = pack_bf16x2(a.x * scale, a.y * scale);
  o.y = pack_bf16x2(a.z * scale, a.w * scale);
  o.z = pack_bf16x2(b.x * scale, b.y * scale);
  o.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[k] = o;
}

template <int D, int SCORE, bool PGRAD>
cudaError_t launch_bwd_t(const AttnArgs& a, const BwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  const uint64_t bh = (uint64_t)a.B * a.H;
  const int64_t rows = (int64_t)bh * a.q_len;
  const int64_t row_blocks = (rows + 256 / (D / 16) - 1) / (256 / (D / 16));  // rows per block of bwd_pre
  bwd_pre_kernel<D><<<(unsigned)(row_blocks + (int64_t)bh * a.nkv), 256, 0, stream>>>(
      a, static_cast<const __nv_bfloat16*>(t.out), static_cast<const __nv_bfloat16*>(t.dout), t.lse, t.stats,
      t.dq_acc, rows, row_blocks, a.param_grad,
      PGRAD ? (SCORE == FA_S_RELBIAS ? (int64_t)a.H * a.bias_len : (int64_t)a.H) : (int64_t)0, t.sched,
      static_cast<__nv_bfloat16*>(t.dk),
      static_cast<__nv_bfloat16*>(t.dv));

  CUtensorMap mq, mk, mv, mdo, mdk, mdv;
  auto enc = [&](CUtensorMap* m, const void* ptr, int64_t len, uint32_t rows) {
    return encode_tmap_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, D, len, bh, 64, rows,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  };
  CUtensorMap mdq;
  const bool ok = enc(&mq, t.q, a.q_len, 128) && enc(&mk, t.k, a.kv_len, 128) && enc(&mv, t.v, a.kv_len, 128) &&
                  enc(&mdo, t.dout, a.q_len, 128) && enc(&mdk, t.dk, a.kv_len, 32) && enc(&mdv, t.dv, a.kv_len, 32) &&
                  encode_tmap_3d(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, t.dq_acc, D, a.q_len, bh, 32, 32,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    *enc_failed = true;
    return cudaErrorUnknown;
  }
  constexpr size_t smem = bwd_smem_bytes<D>();
  static PerDeviceOnce attr_once;
  cudaError_t e = attr_once.run([] {
    return cudaFuncSetAttribute(bwd_kernel<D, SCORE, PGRAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (or per item, when there are fewer)
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.B * a.H * a.nkv;
  if (items >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)std::min<int64_t>(items, sms);
  if (grid > 0)
    bwd_kernel<D, SCORE, PGRAD><<<grid, BwdCfg<D>::THREADS, smem, stream>>>(
        mq, mk, mv, mdo, mdk, mdv, mdq, a, t.stats, t.sched);
  const int64_t n8 = rows * D / 8;
  bwd_dq_convert_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(
      t.dq_acc, static_cast<__nv_bfloat16*>(t.dq), n8, a.scale);
  return cudaGetLastError();
}

// Scratch of fa_backward_noalloc: the fp32 dq accumulator and Delta, in
// library-owned device memory instead of a caller workspace.  Every call
// shares it; bwd_pre_kernel rewrites all of it that a call uses (zeroed dq
// accumulator, fresh Delta) before the main kernel reads it.
__device__ __align__(256) uint8_t g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

}  // namespace

cudaError_t noalloc_scratch(void** ptr) {
  // Device address of the scratch array on the current device, looked up once
  // per device with that device current.  (In host code the array's name is
  // only a stand-in for the symbol, never a device address.)
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

#ifdef FA_TEST_HOOKS
cudaError_t test_hook_backward(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(g_hook_skip_first_k, &v, sizeof(v));
}
#endif

cudaError_t launch_backward(const AttnArgs& a, const BwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  *enc_failed = false;
  const bool pgrad = a.param_grad != nullptr;  // learned ALiBi slopes or bias table (checked on the host)
  if (a.D == 64) {
    if (a.score_op == FA_S_SOFTCAP) return launch_bwd_t<64, FA_S_SOFTCAP, false>(a, t, stream, enc_failed);
    if (a.score_op == FA_S_ALIBI)
      return pgrad ? launch_bwd_t<64, FA_S_ALIBI, true>(a, t, stream, enc_failed)
                   : launch_bwd_t<64, FA_S_ALIBI, false>(a, t, stream, enc_failed);
    if (a.score_op == FA_S_RELBIAS)
      return pgrad ? launch_bwd_t<64, FA_S_RELBIAS, true>(a, t, stream, enc_failed)
                   : launch_bwd_t<64, FA_S_RELBIAS, false>(a, t, stream, enc_failed);
    return launch_bwd_t<64, FA_S_NONE, false>(a, t, stream, enc_failed);
  }
  if (a.score_op == FA_S_SOFTCAP) return launch_bwd_t<128, FA_S_SOFTCAP, false>(a, t, stream, enc_failed);
  if (a.score_op == FA_S_ALIBI)
    return pgrad ? launch_bwd_t<128, FA_S_ALIBI, true>(a, t, stream, enc_failed)
                 : launch_bwd_t<128, FA_S_ALIBI, false>(a, t, stream, enc_failed);
  if (a.score_op == FA_S_RELBIAS)
    return pgrad ? launch_bwd_t<128, FA_S_RELBIAS, true>(a, t, stream, enc_failed)
                 : launch_bwd_t<128, FA_S_RELBIAS, false>(a, t, stream, enc_failed);
  return launch_bwd_t<128, FA_S_NONE, false>(a, t, stream, enc_failed);
}

}  // namespace fa
