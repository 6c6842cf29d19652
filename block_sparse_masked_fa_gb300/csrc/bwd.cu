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
//                  tile for one bulk copy each, and a zeroed fp32 dq accumulator.
//  2. bwd_kernel -- one CTA per (b, h, key tile J), key tiles longest first:
//       warps 0-3  thread r owns key row r (TMEM lane r): P^T, dS^T
//       warps 8-11 dq reducers: dQ tile from TMEM, TMA bulk reduce-add into the accumulator
//       warp 8     TMA producer: K_J, V_J once; Q_I, dO_I (+ LSE_I, Delta_I) per step
//       warp 9     MMA issuer, five tcgen05 GEMMs per (I, J):
//                    S^T  = K Q^T           (TMEM [0,128))
//                    dP^T = V dO^T          (TMEM [128,256))
//                    dV  += P^T dO          (P^T bf16 read from TMEM [0,64))
//                    dK  += dS^T Q          (dS in shared memory, K-major)
//                    dQ   = dS K            (same shared buffer read MN-major; TMEM [128,128+D))
//     dK and dV stay in TMEM for the whole key tile and are written once
//     (no atomics); dQ partial tiles are added into the fp32 accumulator.
//  3. bwd_dq_convert -- dq = bf16(scale * accumulator).
#include <cfloat>
#include <cmath>

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
  static constexpr int NQ = 2;                     // Q ring slots (with LSE / Delta)
  static constexpr int NDO = (D == 64) ? 2 : 1;    // dO ring slots
  static constexpr uint32_t DS_BYTES = 128u * 128u * 2u;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr int THREADS = 448;  // 8 key-row warps, 4 dq warps, producer, MMA
};

struct TileStats {  // one bulk copy per query tile, from the workspace
  float nlse[128];    // -LSE * log2(e) of the tile's query rows
  float ndelta[128];  // -Delta of the tile's query rows
};

struct BwdCtl {
  alignas(16) TileStats stats[2];  // per Q slot
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full[2], do_empty[2];
  uint64_t s_full, p_full, dq_full, dq_free, acc_full, fin;
  uint32_t tmem;
  int abort;
  int32_t arg[FA_MAX_MASK_NODES];
};

template <int D>
constexpr size_t bwd_smem_bytes() {
  using C = BwdCfg<D>;
  return 1024 + (size_t)C::TILE * (2 + C::NQ + C::NDO) + C::DS_BYTES + sizeof(BwdCtl);
}

__device__ __forceinline__ void fail(const AttnArgs& p, BwdCtl* ctl) {
  atomicOr(p.status, kStatusTimeout);
  ctl->abort = 1;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  const bool r = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, r);
}

__device__ __forceinline__ float tanh_fast(float t) {
  const float e = ex2_approx(t * (2.0f * kLog2e));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return fmaf(-2.0f, r, 1.0f);
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
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

template <int D, int SCORE>
__global__ void __launch_bounds__(448, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
               const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ AttnArgs p,
               const float* __restrict__ stats_g) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::TILE;
  uint8_t* sQ0 = sV + C::TILE;             // Q ring
  uint8_t* sDO0 = sQ0 + C::NQ * C::TILE;   // dO ring
  uint8_t* sDS = sDO0 + C::NDO * C::TILE;
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(sDS + C::DS_BYTES);
  auto sQ = [&](int st) { return sQ0 + st * C::TILE; };
  auto sDO = [&](int st) { return sDO0 + st * C::TILE; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // ---- work item: (b, h, key tile J), columns taken longest first
  const int rep = (p.B / p.Bm) * (p.H / p.Hm);
  const int col = p.col_order[blockIdx.x / rep];  // index into [Bm][Hm][nkv]
  const int t = blockIdx.x % rep;
  const int J = col % p.nkv;
  const int hm = (col / p.nkv) % p.Hm;
  const int bm = col / (p.nkv * p.Hm);
  const int b = (p.Bm == 1) ? t / (p.H / p.Hm) : bm;
  const int h = (p.Hm == 1) ? t % (p.H / p.Hm) : hm;
  const int bh = b * p.H + h;
  const int n_full = p.full_q_num[col];
  int n = n_full + p.q_num[col];
  const int64_t list = (int64_t)col * p.nq;

  const uint32_t b_kv = smem_u32(&ctl->kv_full), b_s = smem_u32(&ctl->s_full), b_p = smem_u32(&ctl->p_full),
                 b_dq = smem_u32(&ctl->dq_full), b_dqf = smem_u32(&ctl->dq_free),
                 b_acc = smem_u32(&ctl->acc_full), b_fin = smem_u32(&ctl->fin);
  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(smem_u32(&ctl->q_full[s2]), 1);
      mbar_init(smem_u32(&ctl->q_empty[s2]), 1);
      mbar_init(smem_u32(&ctl->do_full[s2]), 1);
      mbar_init(smem_u32(&ctl->do_empty[s2]), 1);
    }
    mbar_init(b_s, 1);
    mbar_init(b_p, 256);
    mbar_init(b_dq, 1);
    mbar_init(b_dqf, 128);
    mbar_init(b_acc, 1);
    mbar_init(b_fin, 1);
    ctl->abort = (*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) ? 1 : 0;
    fence_mbar_init();
  }
  if (threadIdx.x < p.mask.n) ctl->arg[threadIdx.x] = node_arg(p.mask, threadIdx.x, bm);
  if (warp == 12) {
    tmem_alloc(smem_u32(&ctl->tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const bool skip = ctl->abort != 0;
  if (skip) n = 0;

  auto tile_of = [&](int it) -> int { return it < n_full ? p.full_q_idx[list + it] : p.q_idx[list + it - n_full]; };

  if (warp == 12) {
    // ------------------------------------------------------------ producer
    if (n > 0) {
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        mbar_arrive_expect_tx(b_kv, 2 * C::TILE);
        for (int c = 0; c < C::NC; ++c) {
          tma_load_3d(smem_u32(sK + c * 16384), &tm_k, b_kv, c * 64, J * 128, bh);
          tma_load_3d(smem_u32(sV + c * 16384), &tm_v, b_kv, c * 64, J * 128, bh);
        }
      }
      int q_issued = 0, do_issued = 0;
      bool ok = true;
      for (int it = 0; it < n; ++it) {
        const int I = tile_of(it);
        // Q slot, with the tile's -LSE (log2 units) and -Delta
        const int qs = it % C::NQ, quse = it / C::NQ;
        if (quse > 0 && !warp_wait(smem_u32(&ctl->q_empty[qs]), (quse - 1) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t qbar = smem_u32(&ctl->q_full[qs]);
          mbar_arrive_expect_tx(qbar, C::TILE + (uint32_t)sizeof(TileStats));
          for (int c = 0; c < C::NC; ++c)
            tma_load_3d(smem_u32(sQ(qs) + c * 16384), &tm_q, qbar, c * 64, I * 128, bh);
          bulk_load(smem_u32(&ctl->stats[qs]), stats_g + ((int64_t)bh * p.nq + I) * 256,
                    (uint32_t)sizeof(TileStats), qbar);
        }
        q_issued = it + 1;
        // dO slot
        const int ds = it % C::NDO, duse = it / C::NDO;
        if (duse > 0 && !warp_wait(smem_u32(&ctl->do_empty[ds]), (duse - 1) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t dbar = smem_u32(&ctl->do_full[ds]);
          mbar_arrive_expect_tx(dbar, C::TILE);
          for (int c = 0; c < C::NC; ++c)
            tma_load_3d(smem_u32(sDO(ds) + c * 16384), &tm_do, dbar, c * 64, I * 128, bh);
        }
        do_issued = it + 1;
      }
      if (!ok && lane == 0) fail(p, ctl);
      // drain: every copy this CTA started lands before it exits
      if (lane == 0) {
        mbar_wait(b_kv, 0, nullptr);
        for (int it = max(0, q_issued - C::NQ); it < q_issued; ++it)
          mbar_wait(smem_u32(&ctl->q_full[it % C::NQ]), (it / C::NQ) & 1, nullptr);
        for (int it = max(0, do_issued - C::NDO); it < do_issued; ++it)
          mbar_wait(smem_u32(&ctl->do_full[it % C::NDO]), (it / C::NDO) & 1, nullptr);
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t kIdKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKM = idesc_bf16(128, D, false, true);     // dV (A in TMEM), dK
      constexpr uint32_t kIdMM = idesc_bf16(128, D, true, true);      // dQ
      const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV), ds_base = smem_u32(sDS);
      bool ok = mbar_wait(b_kv, 0, &ctl->abort);
      for (int it = 0; ok && it < n; ++it) {
        const int qs = it % C::NQ, ds = it % C::NDO;
        if (!mbar_wait(smem_u32(&ctl->q_full[qs]), (it / C::NQ) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t q_base = smem_u32(sQ(qs)), do_base = smem_u32(sDO(ds));
        // S^T = K Q^T: its columns held P^T of the last step, read by the dV MMA issued before
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
          mma_ss(tmem + C::T_S, sdesc_sw128(k_base + off, 16, 1024), sdesc_sw128(q_base + off, 16, 1024), kIdKK,
                 kk > 0);
        }
        if (!mbar_wait(smem_u32(&ctl->do_full[ds]), (it / C::NDO) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        if (it > 0 && !mbar_wait(b_dqf, (it - 1) & 1, &ctl->abort)) {  // dQ of the last step read out
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
          mma_ss(tmem + C::T_DP, sdesc_sw128(v_base + off, 16, 1024), sdesc_sw128(do_base + off, 16, 1024), kIdKK,
                 kk > 0);
        }
        mma_commit(b_s);
        if (!mbar_wait(b_p, it & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dV += P^T dO; P^T of query columns [64 h, 64 h + 64) sits at TMEM columns [64 h, 64 h + 32)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + (kk / 4) * 64 + (kk % 4) * 8,
                 sdesc_sw128(do_base + kk * 2048, 16384, 1024), kIdKM, (it > 0 || kk > 0));
        mma_commit(smem_u32(&ctl->do_empty[ds]));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q
          mma_ss(tmem + C::T_DK, sdesc_sw128(ds_base + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                 sdesc_sw128(q_base + kk * 2048, 16384, 1024), kIdKM, (it > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ = dS K
          mma_ss(tmem + C::T_DP, sdesc_sw128(ds_base + kk * 2048, 16384, 1024),
                 sdesc_sw128(k_base + kk * 2048, 16384, 1024), kIdMM, kk > 0);
        mma_commit(b_dq);  // the dq reducers release the Q slot (they stage dQ in it)
      }
      if (ok)
        mma_commit(b_acc);
      else
        fail(p, ctl);
      mma_commit(b_fin);
      mbar_wait(b_fin, 0, nullptr);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dq reducers
    // dQ tile: TMEM -> registers -> 128-byte-swizzled fp32 boxes (32 columns x
    // 128 rows) staged in this step's Q slot (free: dK, the last reader of Q,
    // is done) -> TMA bulk reduce-add into the fp32 accumulator.  Half of the
    // tile fits the slot at a time.
    const int r = (warp % 4) * 32 + lane;  // TMEM lane = query row within the tile
    const uint32_t tq = tmem + ((uint32_t)((warp % 4) * 32) << 16) + C::T_DP;
    constexpr int kHalfCols = D / 2;  // dQ columns per staging round
    bool ok = true;
    for (int it = 0; ok && it < n; ++it) {
      const int I = tile_of(it);
      const int qs = it % C::NQ;
      ok = named_bar_and(2, 128, warp_wait(b_dq, it & 1, &ctl->abort));
      if (!ok) break;
      tc_fence_after();
      uint8_t* stage = sQ(qs);
#pragma unroll 1
      for (int h2 = 0; h2 < 2; ++h2) {
        float v[kHalfCols];
        if constexpr (kHalfCols == 64) {
          tmem_ld64f(tq + kHalfCols * h2, v);
        } else {
          tmem_ld32f(tq + kHalfCols * h2, v);
        }
        if (h2 == 1) {
          tc_fence_before();
          mbar_arrive(b_dqf);  // TMEM columns free for the next dP^T
          if (r == 0) bulk_wait_read0();  // the first half's reduce has read the staging
          named_bar_sync(2, 128);
        }
#pragma unroll
        for (int bx = 0; bx < kHalfCols / 32; ++bx) {
          uint8_t* rowp = stage + bx * 16384 + r * 128;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            *reinterpret_cast<float4*>(rowp + ((q4 ^ (r & 7)) << 4)) =
                make_float4(v[32 * bx + 4 * q4], v[32 * bx + 4 * q4 + 1], v[32 * bx + 4 * q4 + 2],
                            v[32 * bx + 4 * q4 + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (r == 0) {
          for (int bx = 0; bx < kHalfCols / 32; ++bx)
            tma_reduce_add_3d(&tm_dq, smem_u32(stage + bx * 16384), kHalfCols * h2 + 32 * bx, I * 128, bh);
          bulk_commit();
        }
      }
      if (r == 0) {
        bulk_wait_read0();
        mbar_arrive(smem_u32(&ctl->q_empty[qs]));  // the Q slot may be reloaded
      }
    }
    if (!ok) fail(p, ctl);
    if (r == 0) bulk_wait0();  // every reduce of this CTA has completed
  } else {
    // ------------------------------------------------------------ P^T / dS^T, then the epilogue
    // warps 0-7: key row r = 32 (warp % 4) + lane; query columns [64 half, 64 half + 64)
    const int r = (warp % 4) * 32 + lane;
    const int half = warp / 4;
    const int j = J * 128 + r;  // key row
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S, tP = tmem + lane_off + C::T_DP;
    const int32_t* doc_row = p.mask.has_doc ? p.mask.doc + (int64_t)bm * p.mask.doc_len : nullptr;
    const int32_t doc_j = doc_row ? __ldg(doc_row + min(j, p.kv_len - 1)) : 0;
    int run_lo = 0, run_hi = 0;  // with sorted ids: doc[i] == doc[j] exactly for i in [run_lo, run_hi)
    const bool use_run = doc_row != nullptr && doc_run(p.mask, bm, min(j, p.kv_len - 1), run_lo, run_hi);
    const float sc_l2 = p.scale * kLog2e;
    float cap_l2 = 0.f, sc_over_cap = 0.f, slope_l2 = 0.f;
    if constexpr (SCORE == FA_S_SOFTCAP) {
      const float cap = __ldg(p.score_param);
      cap_l2 = cap * kLog2e;
      sc_over_cap = p.scale / cap;
    }
    if constexpr (SCORE == FA_S_ALIBI) slope_l2 = __ldg(p.score_param + h) * kLog2e;
    const bool row_ok = j < p.kv_len;
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int I = tile_of(it);
      const bool partial = it >= n_full;
      const int qs = it % C::NQ;
      if (!warp_wait(b_s, it & 1, &ctl->abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* nlse_s = ctl->stats[qs].nlse;
      const float* ndel_s = ctl->stats[qs].ndelta;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c = 2 * half + c2;  // 32-column chunk of the 128 query columns
        const int i0 = I * 128 + 32 * c;
        uint32_t w = row_ok ? 0xffffffffu : 0u;
        if (partial && row_ok) {
          auto eq = [&]() {
            if (use_run) return range_bits(run_lo, run_hi, i0);
            uint32_t bits = 0;
            if (i0 + 32 <= p.q_len && p.mask.doc_vec_ok) {
              const int4* dv = reinterpret_cast<const int4*>(doc_row + i0);
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const int4 d = __ldg(dv + q4);
                bits |= (uint32_t)(d.x == doc_j) << (4 * q4) | (uint32_t)(d.y == doc_j) << (4 * q4 + 1) |
                        (uint32_t)(d.z == doc_j) << (4 * q4 + 2) | (uint32_t)(d.w == doc_j) << (4 * q4 + 3);
              }
            } else {
              const int in = min(i0 + 32, p.q_len);
              for (int i = i0; i < in; ++i) bits |= (uint32_t)(__ldg(doc_row + i) == doc_j) << (uint32_t)(i - i0);
            }
            return bits;
          };
          w = mask_word_t_rolled(p.mask, ctl->arg, bm, j, i0, eq);
        }
        float sv[32], dp[32];
        tmem_ld32x2f(tS + 32 * c, sv, tP + 32 * c, dp);
        uint32_t pk[16], dk[16];
        const float2* nl2 = reinterpret_cast<const float2*>(nlse_s + 32 * c);
        const float2* nd2 = reinterpret_cast<const float2*>(ndel_s + 32 * c);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 nl = nl2[e / 2], nd = nd2[e / 2];
          float2 a, g = make_float2(1.0f, 1.0f);
          if constexpr (SCORE == FA_S_SOFTCAP) {
            const float t0 = tanh_fast(sv[e] * sc_over_cap), t1 = tanh_fast(sv[e + 1] * sc_over_cap);
            a = fma2(make_float2(cap_l2, cap_l2), make_float2(t0, t1), nl);
            g = fma2(make_float2(-t0, -t1), make_float2(t0, t1), make_float2(1.0f, 1.0f));
          } else if constexpr (SCORE == FA_S_ALIBI) {
            a = fma2(make_float2(sv[e], sv[e + 1]), make_float2(sc_l2, sc_l2),
                     make_float2(fmaf(-slope_l2, (float)(i0 + e - j), nl.x),
                                 fmaf(-slope_l2, (float)(i0 + e + 1 - j), nl.y)));
          } else {
            a = fma2(make_float2(sv[e], sv[e + 1]), make_float2(sc_l2, sc_l2), nl);
          }
          float2 pv;
          pv.x = ((w >> e) & 1u) ? ex2_approx(a.x) : 0.f;
          pv.y = ((w >> (e + 1)) & 1u) ? ex2_approx(a.y) : 0.f;
          float2 dsv = mul2(pv, add2(make_float2(dp[e], dp[e + 1]), nd));
          if constexpr (SCORE == FA_S_SOFTCAP) dsv = mul2(dsv, g);
          pk[e / 2] = pack_bf16x2(pv.x, pv.y);
          dk[e / 2] = pack_bf16x2(dsv.x, dsv.y);
        }
        // P^T over this half's own S^T columns, already read: [64 half + 16 c2, +16)
        tmem_st16(tS + 64 * half + 16 * c2, pk);
        store_row32(sDS, r, c, dk);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(b_p);
    }
    if (!ok) fail(p, ctl);
    // ---- epilogue: dV and scale * dK from TMEM, once per key tile; each half writes D/2 columns
    if (ok && n > 0) {
      if (!warp_wait(b_acc, 0, &ctl->abort)) {
        ok = false;
        fail(p, ctl);
      }
      tc_fence_after();
    }
    // staging for dV / dK: the dS buffer and the first dO slot, whose last readers
    // (the dK / dQ and dV MMAs) are done once acc_full completes; the Q slots may
    // still hold the dq reducers' last staged tile
    uint8_t* stage_v = sDS;
    uint8_t* stage_k = sDO(0);
    if (ok && !skip) {
#pragma unroll 1
      for (int c2 = 0; c2 < D / 64; ++c2) {
        const int c = half * (D / 64) + c2;  // 32-column chunk of D
        float a[32], g[32];
        if (n > 0) {
          tmem_ld32f(tmem + lane_off + C::T_DV + 32 * c, a);
          tmem_ld32f(tmem + lane_off + C::T_DK + 32 * c, g);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = g[e] = 0.f;
        }
        uint32_t wv[16], wk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          wv[e] = pack_bf16x2(a[2 * e], a[2 * e + 1]);
          wk[e] = pack_bf16x2(g[2 * e] * p.scale, g[2 * e + 1] * p.scale);
        }
        store_row32(stage_v, r, c, wv);
        store_row32(stage_k, r, c, wk);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (threadIdx.x == 0 && !skip && !*reinterpret_cast<volatile int*>(&ctl->abort)) {
      for (int c = 0; c < C::NC; ++c) {
        tma_store_3d(&tm_dv, smem_u32(stage_v + c * 16384), c * 64, J * 128, bh);
        tma_store_3d(&tm_dk, smem_u32(stage_k + c * 16384), c * 64, J * 128, bh);
      }
      bulk_commit();
      bulk_wait_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Per query row: -LSE * log2(e) and -Delta (Delta_i = dO_i . out_i, fp32)
// into the per-tile stats array [B*H][nq][2][128], zero for the rows past
// q_len in the last tile; and the fp32 dq accumulator rows set to zero.
// 16 threads per row, 16 rows per 256-thread block.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ out,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const float* __restrict__ lse, float* __restrict__ stats,
                                                      float* __restrict__ dq_acc, int64_t rows, int q_len, int nq) {
  constexpr int E = D / 16;  // elements per thread
  const int64_t row = (int64_t)blockIdx.x * 16 + threadIdx.x / 16;
  const int t = threadIdx.x % 16;
  float acc = 0.f;
  if (row < rows) {
    const __nv_bfloat16* o = out + row * D + t * E;
    const __nv_bfloat16* g = dout + row * D + t * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + e));
      const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(g + e));
      acc = fmaf(a.x, c.x, fmaf(a.y, c.y, acc));
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * D + t * E);
#pragma unroll
    for (int e = 0; e < E / 4; ++e) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
  if (row < rows && t == 0) {
    const int64_t bh = row / q_len;
    const int i = (int)(row % q_len);
    float* st = stats + (bh * nq + i / 128) * 256;
    st[i % 128] = -__ldg(lse + row) * kLog2e;
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

template <int D, int SCORE>
cudaError_t launch_bwd_t(const AttnArgs& a, const BwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  const uint64_t bh = (uint64_t)a.B * a.H;
  const int64_t rows = (int64_t)bh * a.q_len;
  bwd_pre_kernel<D><<<(unsigned)((rows + 15) / 16), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(t.out), static_cast<const __nv_bfloat16*>(t.dout), t.lse, t.stats, t.dq_acc,
      rows, a.q_len, a.nq);

  CUtensorMap mq, mk, mv, mdo, mdk, mdv;
  auto enc = [&](CUtensorMap* m, const void* ptr, int64_t len) {
    return encode_tmap_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, D, len, bh, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  };
  CUtensorMap mdq;
  const bool ok = enc(&mq, t.q, a.q_len) && enc(&mk, t.k, a.kv_len) && enc(&mv, t.v, a.kv_len) &&
                  enc(&mdo, t.dout, a.q_len) && enc(&mdk, t.dk, a.kv_len) && enc(&mdv, t.dv, a.kv_len) &&
                  encode_tmap_3d(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, t.dq_acc, D, a.q_len, bh, 32, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    *enc_failed = true;
    return cudaErrorUnknown;
  }
  constexpr size_t smem = bwd_smem_bytes<D>();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t items = (int64_t)a.B * a.H * a.nkv;
  bwd_kernel<D, SCORE><<<(unsigned)items, BwdCfg<D>::THREADS, smem, stream>>>(mq, mk, mv, mdo, mdk, mdv, mdq, a, t.stats);
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

cudaError_t launch_backward(const AttnArgs& a, const BwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  *enc_failed = false;
  if (a.D == 64) {
    if (a.score_op == FA_S_SOFTCAP) return launch_bwd_t<64, FA_S_SOFTCAP>(a, t, stream, enc_failed);
    if (a.score_op == FA_S_ALIBI) return launch_bwd_t<64, FA_S_ALIBI>(a, t, stream, enc_failed);
    return launch_bwd_t<64, FA_S_NONE>(a, t, stream, enc_failed);
  }
  if (a.score_op == FA_S_SOFTCAP) return launch_bwd_t<128, FA_S_SOFTCAP>(a, t, stream, enc_failed);
  if (a.score_op == FA_S_ALIBI) return launch_bwd_t<128, FA_S_ALIBI>(a, t, stream, enc_failed);
  return launch_bwd_t<128, FA_S_NONE>(a, t, stream, enc_failed);
}

}  // namespace fa
