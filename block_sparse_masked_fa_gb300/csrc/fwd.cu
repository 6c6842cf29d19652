// fwd.cu -- tile-list-driven flash-attention forward for sm_103a.
//
// What it computes (speedrun notes "FlexAttention", Context paragraph and
// tile-summary paragraph; tutorial "FlexAttention in PyTorch", "The two hooks"
// and Pattern 3): for every query row i,
//     out_i = sum_{j visible} exp(s_ij - LSE_i) v_j,   LSE_i = ln sum_{j visible} exp(s_ij),
//     s_ij  = score_mod(scale * q_i . k_j),
// visiting only the key tiles listed for the row's query tile: FULL tiles with
// no mask work, PARTIAL tiles with the mask program evaluated per element.
//
// Persistent: two CTAs per SM, each taking every gridDim.x-th (b, h, query
// tile I) of the longest-first order, so that one CTA's softmax overlaps the
// other's matrix multiplies.  Warp roles:
//   warps 0-3  softmax + epilogue: thread r owns query row r (TMEM lane r)
//   warp 4     TMA producer (item descriptors, Q per item, K_j / V_j through a
//              ring of slots) and TMEM allocator
//   warp 5     MMA issuer (one thread): S = Q K_j^T into TMEM, then
//              O += P V_j with P read from TMEM, in two halves: keys [0, 64)
//              as soon as the softmax warps have written their P
// Across items the pipeline keeps going: the next item's Q loads once the last
// S has read the buffer, its first S runs while the epilogue reads O out of
// TMEM, and the output is staged in shared memory (the last V slot with two
// slots) and stored by TMA (thread 0) without waiting.
// TMEM (256 columns): S at [0, BK) and O at [128, 128 + D).  P (bf16 pairs, BK / 2
// columns) overwrites S's first columns after the softmax has read S when D = 128
// with 128-key tiles; in the other shapes it has columns of its own, and the next
// step's S is computed while the softmax warps work on this one where the K / V
// ring has loaded the next K in time (D = 64).
// Key tiles are BK = 128 positions, or 64 when the block mask's tiles are
// smaller (tutorial, sharp edge 4): then S is 128 x 64, the P V of a step is
// one group of four MMAs, and the output has a staging buffer of its own.
// The running maximum is only moved (and O rescaled) when a new row maximum
// exceeds it by more than 2^8, so most tiles need no O round trip.  With ALiBi
// a row's key tiles are visited nearest first (PARTIAL tiles, then FULL tiles,
// each list from its last entry), so that the largest bias of the row is met in
// the first step and the maximum then rarely moves; otherwise FULL tiles come
// first, so that an item's first step has no mask words to compute.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// BK: key positions per listed key tile -- 128, or 64 for block masks with
// smaller tiles (the builder's 128 x 64 lists).
template <int D, int BK>
struct FwdCfg {
  static constexpr int NC = D / 64;                      // 64-column (128-byte) chunks per tile row
  static constexpr uint32_t TILE = 128u * D * 2u;        // bytes of one 128 x D bf16 tile (Q, output)
  static constexpr uint32_t KV_TILE = (uint32_t)BK * D * 2u;  // one K or V tile
  static constexpr uint32_t KV_CHUNK = (uint32_t)BK * 128u;   // one 64-column chunk of it
  // K/V ring slots: two CTAs per SM must fit
  static constexpr int NS = (BK == 128) ? ((D == 64) ? 4 : 2) : ((D == 64) ? 6 : 2);
  static constexpr bool STAGE_IN_RING = (NS == 2 && BK == 128);  // output staged in the last V slot
  static constexpr int NW = BK / 32;                     // 32-column mask words per row and step
  static constexpr uint32_t TMEM_COLS = 256;
  // P in TMEM columns of its own when S (BK columns), O ([128, 128 + D)) and P
  // (BK / 2 columns) fit in the 256: then the next step's S is computed while
  // the softmax warps work on this one's; else P overwrites S's first columns
  static constexpr bool SP = (BK == 64) || (D == 64);
  static constexpr uint32_t T_P = !SP ? 0u : (BK == 64 ? 64u : 128u + D);
  // the next S ahead of this step's P V only where the ring has loaded the next K
  // by then (with two slots it is loaded once this step's S is done, and waiting
  // for it would hold up the P V)
  static constexpr bool EARLY_S = SP && NS >= 4;
};

// One work item: the query tile I of head (b, h), with the key tiles of its
// row lists: FULL then PARTIAL, or with ALiBi PARTIAL then FULL, each read
// backwards (highest key tile first).
struct FwdItem {
  int I, bh, bm, h, n_full, n;
  int J0;        // the first key tile (when n > 0)
  int64_t list;  // offset of the row's lists
};

constexpr int kMaxKvSlots = 8;  // K/V ring slots the control block has barriers for

struct FwdCtl {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kMaxKvSlots];
  uint64_t kv_empty[kMaxKvSlots];
  uint64_t s_full;
  uint64_t p_half, p_full;  // P of the first 64 keys, of all 128 keys
  uint64_t o_full, o_free;
  uint64_t stg_free;
  uint64_t s_free, p_free;  // separate P: S read by the softmax warps; P consumed by its P V
  uint64_t fin;
  uint32_t tmem;
  int abort;
  int32_t arg[FA_MAX_MASK_NODES];
  // items handed from the producer to the softmax warps, two at a time: the
  // descriptor and the tile's 128 rows of visible key intervals (block mask
  // row_segs, rows past the table left as they are)
  uint64_t desc_full[2], desc_empty[2];
  FwdItem desc[2];
  alignas(16) int4 seg[2][128];
};

// a block of zeros the producer copies over a buffer to be cleared (a backward
// workspace's dq accumulator), 4 KB a copy
constexpr uint32_t kZeroBytes = 4096;

template <int D, int BK>
constexpr size_t fwd_smem_bytes() {
  using C = FwdCfg<D, BK>;
  return 1024 + (size_t)C::TILE * (1 + (C::STAGE_IN_RING ? 0 : 1)) + (size_t)C::KV_TILE * C::NS + sizeof(FwdCtl) +
         128 + kZeroBytes;
}
// two CTAs per SM (228 KB of shared memory, 1 KB of it reserved per CTA)
static_assert(2 * (fwd_smem_bytes<128, 128>() + 1024) <= 228 * 1024, "forward shared memory, D = 128");
static_assert(2 * (fwd_smem_bytes<64, 128>() + 1024) <= 228 * 1024, "forward shared memory, D = 64");
static_assert(2 * (fwd_smem_bytes<128, 64>() + 1024) <= 228 * 1024, "forward shared memory, D = 128, BK = 64");
static_assert(2 * (fwd_smem_bytes<64, 64>() + 1024) <= 228 * 1024, "forward shared memory, D = 64, BK = 64");
static_assert(FwdCfg<128, 128>::NS <= kMaxKvSlots && FwdCfg<64, 128>::NS <= kMaxKvSlots &&
                  FwdCfg<128, 64>::NS <= kMaxKvSlots && FwdCfg<64, 64>::NS <= kMaxKvSlots,
              "every K/V ring slot needs its pair of barriers in FwdCtl");

// K-major descriptor of MMA step kk for a tile whose 64-column chunks are
// `chunk` bytes apart (rows x 128 B): byte 32 (kk % 4) of chunk kk / 4.
template <uint32_t CHUNK>
__device__ __forceinline__ uint64_t kmajor_step_c(uint64_t desc, int kk) {
  return desc + (uint64_t)((kk >> 2) * (CHUNK >> 4) + (kk & 3) * (32 >> 4));
}

#ifdef FA_TEST_HOOKS
__device__ int g_hook_skip_first_k;  // see test_hook_forward
#endif

__device__ __forceinline__ void fail(const AttnArgs& p, FwdCtl* ctl) {
  atomicOr(p.status, kStatusTimeout);
  ctl->abort = 1;
}

// A wait whose outcome is the same for the 32 lanes of the calling warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  const bool r = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, r);
}

// tanh(t) = 1 - 2 / (1 + e^{2t}); exact at both saturations, absolute error a few ulp of 1.
__device__ __forceinline__ float tanh_fast(float t) {
  const float e = ex2_approx(t * (2.0f * kLog2e));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return fmaf(-2.0f, r, 1.0f);
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ FwdItem fwd_item(const AttnArgs& p, int k) {
  const int rep = (p.B / p.Bm) * (p.H / p.Hm);
  const int row = __ldg(p.row_order + k / rep);  // index into [Bm][Hm][nq], longest first
  const int t = k % rep;
  FwdItem it;
  it.I = row % p.nq;
  const int hm = (row / p.nq) % p.Hm;
  it.bm = row / (p.nq * p.Hm);
  const int b = (p.Bm == 1) ? t / (p.H / p.Hm) : it.bm;
  it.h = (p.Hm == 1) ? t % (p.H / p.Hm) : hm;
  it.bh = b * p.H + it.h;
  it.n_full = __ldg(p.full_num + row);
  it.n = it.n_full + __ldg(p.kv_num + row);
  it.list = (int64_t)row * p.nkv;
  it.J0 = 0;
  return it;
}

// Whether step jj of an item is a PARTIAL tile, and its key tile.
template <bool NEAR_FIRST>
__device__ __forceinline__ bool step_partial(const FwdItem& it, int jj) {
  return NEAR_FIRST ? jj < it.n - it.n_full : jj >= it.n_full;
}
template <bool NEAR_FIRST>
__device__ __forceinline__ int tile_of(const AttnArgs& p, const FwdItem& it, int jj) {
  if constexpr (NEAR_FIRST) {
    const int n_part = it.n - it.n_full;
    return jj < n_part ? __ldg(p.kv_idx + it.list + (n_part - 1 - jj)) : __ldg(p.full_idx + it.list + (it.n - 1 - jj));
  } else {
    return jj < it.n_full ? __ldg(p.full_idx + it.list + jj) : __ldg(p.kv_idx + it.list + jj - it.n_full);
  }
}

// This CTA's first item at or after k (its items are k, k + gridDim.x, ...)
// with at least one visible key tile; a value >= items when none is left.
__device__ __forceinline__ int next_live(const AttnArgs& p, int k, int items, FwdItem& it) {
  for (; k < items; k += (int)gridDim.x) {
    it = fwd_item(p, k);
    if (it.n > 0) break;
  }
  return k;
}

template <int D, int SCORE, int BK>
__global__ void __launch_bounds__(192, 2)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const __grid_constant__ AttnArgs p, float* __restrict__ lse_out,
               __nv_bfloat16* __restrict__ out_g) {
  using C = FwdCfg<D, BK>;
  constexpr bool NF = (SCORE == FA_S_ALIBI);  // nearest key tiles first
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::TILE;
  // output staging: the V slot of an item's last step (with two slots every V
  // goes to slot 1), else a buffer of its own
  uint8_t* sOut = C::STAGE_IN_RING ? sKV + C::KV_TILE : sKV + C::NS * C::KV_TILE;
  // control block after the ring and the output buffer (when there is one)
  FwdCtl* ctl = reinterpret_cast<FwdCtl*>(sKV + C::NS * C::KV_TILE + (C::STAGE_IN_RING ? 0 : C::TILE));
  // the zero block after the control block, 128-byte aligned
  uint8_t* sZero = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ctl + 1) + 127) & ~uintptr_t(127));
  static_assert(C::NS * C::KV_TILE + (C::STAGE_IN_RING ? 0 : C::TILE) + C::TILE + sizeof(FwdCtl) + 128 + kZeroBytes +
                        1024 <=
                    fwd_smem_bytes<D, BK>(),
                "forward shared-memory layout");
  static_assert(!C::SP || (C::T_P >= (uint32_t)BK && C::T_P + BK / 2 <= 128u) ||
                    (C::T_P >= 128u + D && C::T_P + BK / 2 <= C::TMEM_COLS),
                "separate P: its columns clear of S and O");

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int items = p.B * p.H * p.nq;  // below 2^31: checked at launch

  const uint32_t b_q = smem_u32(&ctl->q_full), b_qe = smem_u32(&ctl->q_empty), b_s = smem_u32(&ctl->s_full),
                 b_p = smem_u32(&ctl->p_full), b_ph = smem_u32(&ctl->p_half), b_o = smem_u32(&ctl->o_full),
                 b_of = smem_u32(&ctl->o_free),
                 b_stg = smem_u32(&ctl->stg_free), b_fin = smem_u32(&ctl->fin),
                 b_sfree = smem_u32(&ctl->s_free), b_pfree = smem_u32(&ctl->p_free);
  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    mbar_init(b_qe, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(smem_u32(&ctl->kv_full[s]), 1);
      mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
    }
    mbar_init(b_s, 1);
    mbar_init(b_p, 128);
    mbar_init(b_ph, 128);
    mbar_init(b_o, 1);
    mbar_init(b_of, 128);
    mbar_init(b_stg, 1);
    mbar_init(b_sfree, 128);
    mbar_init(b_pfree, 1);
    mbar_init(b_fin, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->desc_full[s]), 1);
      mbar_init(smem_u32(&ctl->desc_empty[s]), 128);
    }
    // once any CTA has given up, later CTAs do no work (one decision per CTA)
    ctl->abort = (*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) ? 1 : 0;
    fence_mbar_init();
  }
  // mask program arguments: set here when there is one mask batch, else per item
  if (p.Bm == 1 && threadIdx.x < p.mask.n) ctl->arg[threadIdx.x] = node_arg(p.mask, threadIdx.x, 0);
  if (warp == 4) {
    tmem_alloc(smem_u32(&ctl->tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const int first = (ctl->abort != 0) ? items : (int)blockIdx.x;

  // The CTA stays resident and takes the items blockIdx.x, blockIdx.x +
  // gridDim.x, ...; every role walks the same sequence.  Steps (I, J) are
  // numbered across items (t) for the K / V ring and the per-step barriers;
  // items with visible key tiles are numbered (u) for Q and the O accumulator.
  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    // Every item's descriptor and row intervals to the softmax warps; Q of an
    // item once the last S of the item before has read the buffer; K_j / V_j
    // through the ring.  With two slots the first V of an item also waits
    // until the output staged in its slot has been stored.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_o);
    }
    int t = 0, u = 0, v = 0, issued = 0, q_issued = 0, published = 0;
    // A buffer to clear while the forward runs (a backward workspace's dq
    // accumulator): this CTA's share, in copies of the zero block issued after
    // the K / V loads (so that no load waits behind them) and the rest at the
    // end; an evict-first L2 policy keeps the stream from pushing out K / V.
    int64_t z_next = 0, z_end = 0;
    uint64_t z_pol = 0;
    const uint32_t s_zero = smem_u32(sZero);
    if (p.zero_dst != nullptr) {
      const int64_t per = ((p.zero_n16 + gridDim.x - 1) / gridDim.x + 255) / 256 * 256;  // whole 4 KB copies
      z_next = min((int64_t)blockIdx.x * per, p.zero_n16);
      z_end = min(z_next + per, p.zero_n16);
      for (int q = lane; q < (int)(kZeroBytes / 16); q += 32) reinterpret_cast<uint4*>(sZero)[q] = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      __syncwarp();
      z_pol = l2_evict_first_policy();
    }
    auto zero_some = [&](int copies) {
      if (z_next >= z_end) return;
      if (lane == 0) {
        for (int c = 0; c < copies && z_next < z_end; ++c) {
          const int64_t n = min((int64_t)(kZeroBytes / 16), z_end - z_next);
          bulk_store(p.zero_dst + z_next, s_zero, (uint32_t)(n * 16), z_pol);
          z_next += n;
        }
        bulk_commit();
      }
      z_next = __shfl_sync(0xffffffffu, z_next, 0);
    };
    bool ok = true;
    for (int k = first; ok && k < items; k += (int)gridDim.x, ++v) {
      FwdItem cur = fwd_item(p, k);
      if (cur.n > 0) cur.J0 = tile_of<NF>(p, cur, 0);
      // hand the item to the softmax warps (every item, with or without visible tiles)
      const int dsl = v & 1;
      const uint32_t dfull = smem_u32(&ctl->desc_full[dsl]);
      if (v >= 2 && !warp_wait(smem_u32(&ctl->desc_empty[dsl]), ((v >> 1) - 1) & 1, &ctl->abort)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        ctl->desc[dsl] = cur;
        if (cur.n > 0) {
          const int64_t row0 = (int64_t)cur.I * 128;
          const uint32_t bytes = (uint32_t)min((int64_t)128, p.seg_len - row0) * 16u;
          mbar_arrive_expect_tx(dfull, bytes);
          bulk_load(smem_u32(&ctl->seg[dsl][0]), p.row_segs + (int64_t)cur.bm * 2 * p.seg_len + row0, bytes, dfull);
        } else {
          mbar_arrive(dfull);
        }
      }
      published = v + 1;
      if (cur.n == 0) continue;
      if (u > 0 && !warp_wait(b_qe, (u - 1) & 1, &ctl->abort)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(b_q, C::TILE);
        for (int c = 0; c < C::NC; ++c) tma_load_3d(smem_u32(sQ + c * 16384), &tm_q, b_q, c * 64, cur.I * 128, cur.bh);
      }
      q_issued = u + 1;
      for (int jj = 0; ok && jj < cur.n; ++jj, ++t) {
        const int J = jj == 0 ? cur.J0 : tile_of<NF>(p, cur, jj);
        // rows of key tile J: in the caller's [B*H][kv_len] tensors, or (paged,
        // BK = 128 only) in the page the table names, of this head's
        // [n_pages * 128] pool rows
        int kv_row = J * BK, kv_z = cur.bh;
        if (p.page_table != nullptr && lane == 0) {
          int page = __ldg(p.page_table + (int64_t)(cur.bh / p.H) * p.nkv + J);
          if (page < 0 || page >= p.n_pages) {  // reported; page 0 is read instead
            atomicOr(p.status, kStatusCheck);
            page = 0;
          }
          kv_row = page * 128;
          kv_z = cur.h;
        }
        for (int kv = 0; kv < 2; ++kv) {
          const int pos = 2 * t + kv, slot = pos % C::NS, use = pos / C::NS;
          if (use > 0 && !warp_wait(smem_u32(&ctl->kv_empty[slot]), (use - 1) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          if (C::STAGE_IN_RING && kv == 1 && jj == 0 && u > 0 && !warp_wait(b_stg, (u - 1) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
#ifdef FA_TEST_HOOKS
          const bool hook_skip = g_hook_skip_first_k != 0 && blockIdx.x == 0 && t == 0 && kv == 0;
#else
          constexpr bool hook_skip = false;
#endif
          if (lane == 0 && !hook_skip) {
            const uint32_t bar = smem_u32(&ctl->kv_full[slot]);
            mbar_arrive_expect_tx(bar, C::KV_TILE);
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            for (int c = 0; c < C::NC; ++c)
              tma_load_3d(smem_u32(sKV + slot * C::KV_TILE + c * C::KV_CHUNK), m, bar, c * 64, kv_row, kv_z);
          }
          issued = pos + 1;
          zero_some(2);
        }
      }
      ++u;
    }
    if (ok)
      while (z_next < z_end) zero_some(64);
    if (!ok && lane == 0) fail(p, ctl);
    // drain: every copy this CTA started lands before it exits (each buffer's
    // earlier loads were waited for before the last one was issued)
    if (lane == 0) {
      if (q_issued > 0) mbar_wait(b_q, (q_issued - 1) & 1, nullptr);
      for (int w = max(0, published - 2); w < published; ++w)
        mbar_wait(smem_u32(&ctl->desc_full[w & 1]), (w >> 1) & 1, nullptr);
      for (int pos = max(0, issued - C::NS); pos < issued; ++pos)
        mbar_wait(smem_u32(&ctl->kv_full[pos % C::NS]), (pos / C::NS) & 1, nullptr);
      if (p.zero_dst != nullptr) bulk_wait0();  // the zero copies have landed
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, BK, false, false);   // Q (K-major) x K (K-major)
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);     // P (TMEM) x V (MN-major)
      const uint32_t q_base = smem_u32(sQ);
      int t = 0, u = 0;
      bool ok = true;
      FwdItem cur;
      for (int k = next_live(p, first, items, cur); ok && k < items; ++u) {
        const int n = cur.n;
        FwdItem nxt;
        int kn = items;
        if (!mbar_wait(b_q, u & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        // S of step tt = Q K^T into TMEM [0, BK); `last`: the item's last S
        auto issue_s = [&](int tt, bool last) -> bool {
          const int pk = 2 * tt, sk = pk % C::NS;
          if (!mbar_wait(smem_u32(&ctl->kv_full[sk]), (pk / C::NS) & 1, &ctl->abort)) return false;
          tc_fence_after();
          const uint32_t k_base = smem_u32(sKV + sk * C::KV_TILE);
          const uint64_t a0 = opaque(sdesc_sw128(q_base, 16, 1024)), b0 = opaque(sdesc_sw128(k_base, 16, 1024));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem, kmajor_step(a0, kk), kmajor_step_c<C::KV_CHUNK>(b0, kk), kIdS, kk > 0);
          mma_commit(smem_u32(&ctl->kv_empty[sk]));
          if (last) mma_commit(b_qe);  // Q read for the last time in this item
          mma_commit(b_s);
          return true;
        };
        for (int jj = 0; jj < n; ++jj, ++t) {
          const int pk = 2 * t;
          // S of this step (with P in columns of its own, issued at the step before
          // except for an item's first)
          if ((!C::EARLY_S || jj == 0) && !issue_s(t, jj == n - 1)) {
            ok = false;
            break;
          }
          // the next item, looked up while the softmax runs
          if (jj == 0) kn = next_live(p, k + (int)gridDim.x, items, nxt);
          if constexpr (C::EARLY_S) {
            // the softmax warps have read S: the next step's S into the same
            // columns now, ahead of this step's P V
            if (!mbar_wait(b_sfree, t & 1, &ctl->abort) || (jj + 1 < n && !issue_s(t + 1, jj + 1 == n - 1))) {
              ok = false;
              break;
            }
          }
          // P V in two halves: keys [0, 64) as soon as their P is in TMEM, while
          // the softmax warps compute the rest
          if (!mbar_wait(b_ph, t & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          const int pv = pk + 1, sv = pv % C::NS;
          if (!mbar_wait(smem_u32(&ctl->kv_full[sv]), (pv / C::NS) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          // O of the item before has been read out of TMEM
          if (jj == 0 && u > 0 && !mbar_wait(b_of, (u - 1) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_base = smem_u32(sKV + sv * C::KV_TILE);
          const uint64_t v0 = opaque(sdesc_sw128(v_base, C::KV_CHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + 128, tmem + C::T_P + kk * 8, mnmajor_step(v0, kk), kIdO, (jj > 0 || kk > 0));
          if constexpr (BK == 128) {  // keys [64, 128) once the rest of P is in
            if (!mbar_wait(b_p, t & 1, &ctl->abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 4; kk < 8; ++kk) mma_ts(tmem + 128, tmem + C::T_P + kk * 8, mnmajor_step(v0, kk), kIdO, true);
          }
          mma_commit(smem_u32(&ctl->kv_empty[sv]));
          if constexpr (C::SP) mma_commit(b_pfree);  // P of this step consumed, O updated
        }
        if (!ok) break;
        mma_commit(b_o);
        cur = nxt;
        k = kn;
      }
      if (!ok) fail(p, ctl);
      // drain: no tcgen05 operation of this CTA is in flight past this point
      mma_commit(b_fin);
      mbar_wait(b_fin, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x;  // 0..127, TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off;
    const uint32_t tO = tmem + lane_off + 128;
    const uint64_t mask_ops = pack_ops(p.mask);
    const float sc_l2 = p.scale * kLog2e;  // logit -> log2 units
    float cap_l2 = 0.f, sc_over_cap = 0.f, sc_cap2 = 0.f;
    if constexpr (SCORE == FA_S_SOFTCAP) {
      const float cap = __ldg(p.score_param);
      cap_l2 = cap * kLog2e;
      sc_over_cap = p.scale / cap;
      sc_cap2 = sc_over_cap * (2.0f * kLog2e);  // S -> the exponent of e^{2 x / c}, base 2
    }
    int t = 0, u = 0, v = 0;
    bool ok = true;
    bool stg_pending = false;  // thread 0: an output store whose read of the staging is not yet confirmed
    for (int k = first; k < items; k += (int)gridDim.x, ++v) {
      // the item's descriptor, from the producer; one decision for the whole
      // group, so that every thread takes the same named barriers
      const int dsl = v & 1;
      ok = named_bar_and(1, 128, ok && warp_wait(smem_u32(&ctl->desc_full[dsl]), (v >> 1) & 1, &ctl->abort));
      if (!ok) break;
      const FwdItem cur = ctl->desc[dsl];
      const int n = cur.n, I = cur.I, bh = cur.bh, bm = cur.bm;
      const int i = I * 128 + r;
      // the row's position in the sequence the program describes (rows past
      // q_len, which store nothing, take the last row's)
      const int64_t ipos = (int64_t)i + p.mask.q_off;
      const int64_t ipos_c = (int64_t)min(i, p.q_len - 1) + p.mask.q_off;
      if (p.Bm > 1) {  // this item's mask arguments, once every thread is done with the last item's
        named_bar_sync(1, 128);
        if (r < p.mask.n) ctl->arg[r] = node_arg(p.mask, r, bm);
        named_bar_sync(1, 128);
      }
      if (n == 0) {  // no visible key tile: out = 0, LSE = -inf (direct stores; such tiles are rare)
        if (i < p.q_len) {
          uint4* orow = reinterpret_cast<uint4*>(out_g + ((int64_t)bh * p.q_len + i) * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
          lse_out[(int64_t)bh * p.q_len + i] = -INFINITY;
        }
        mbar_arrive(smem_u32(&ctl->desc_empty[dsl]));
        continue;
      }
      // the list entry of the first step and this row's visible key columns as
      // two intervals (kept in shared memory: read on partial tiles only); the
      // document id and run of the row only for rows the intervals do not
      // describe, which evaluate the program per word
      int J_next = cur.J0;
      const int4* seg_s = &ctl->seg[dsl][r];
      const int4 seg0 = *seg_s;
      const int32_t* doc_row = p.mask.has_doc ? p.mask.doc + (int64_t)bm * p.mask.doc_len : nullptr;
      int32_t doc_i = 0;
      int run_lo = 0, run_hi = 0;  // with sorted ids: doc[j] == doc[i] exactly for j in [run_lo, run_hi)
      bool use_run = false;
      if (seg0.x < 0 && doc_row != nullptr) {
        doc_i = __ldg(doc_row + ipos_c);
        use_run = doc_run(p.mask, bm, ipos_c, run_lo, run_hi);
      }
      float slope_l2 = 0.f, slope_sc = 0.f;
      if constexpr (SCORE == FA_S_ALIBI) {
        const float slope = __ldg(p.score_param + cur.h);
        slope_l2 = slope * kLog2e;
        slope_sc = slope / p.scale;
      }
      const float* bias_h = nullptr;  // RELBIAS: this head's table
      if constexpr (SCORE == FA_S_RELBIAS) bias_h = p.score_param + (int64_t)cur.h * p.bias_len;

      float m = -INFINITY;  // reference maximum, log2 units
      float l = 0.f;
      // the list entry of the next step is fetched one step ahead, off the path
      // from the S wait to the mask words
      for (int jj = 0; jj < n; ++jj, ++t) {
        const bool partial = step_partial<NF>(cur, jj);
        const int J = J_next;
        if (jj + 1 < n) J_next = tile_of<NF>(p, cur, jj + 1);
        const int64_t j0 = (int64_t)J * BK;
        const bool ragged = j0 + BK > p.kv_len;
        const bool msk = partial || ragged;
        // visibility words of the NW x 32 key columns, computed before S is loaded
        uint32_t wd[C::NW];
  #pragma unroll
        for (int c = 0; c < C::NW; ++c) wd[c] = 0xffffffffu;
        if (msk) {
  #pragma unroll 1
          for (int c = 0; c < C::NW; ++c) {
            const int jc = (int)j0 + 32 * c;
            uint32_t w = low_bits((int64_t)p.kv_len - jc);
            const int4 sg = *seg_s;
            if (partial && sg.x >= 0) {
              w &= seg_word(sg, jc);
            } else if (partial) {
              // doc ids of the 32 key columns: the same addresses for every thread (broadcast loads)
              auto eq = [&]() {
                if (use_run) return range_bits(run_lo, run_hi, jc);
                uint32_t bits = 0;
                if (!ragged && p.mask.doc_vec_ok) {
                  const int4* dv = reinterpret_cast<const int4*>(doc_row + jc);
  #pragma unroll
                  for (int q4 = 0; q4 < 8; ++q4) {
                    const int4 d = __ldg(dv + q4);
                    bits |= (uint32_t)(d.x == doc_i) << (4 * q4) | (uint32_t)(d.y == doc_i) << (4 * q4 + 1) |
                            (uint32_t)(d.z == doc_i) << (4 * q4 + 2) | (uint32_t)(d.w == doc_i) << (4 * q4 + 3);
                  }
                } else {
                  const int jn = min(jc + 32, p.kv_len);
                  for (int j = jc; j < jn; ++j) bits |= (uint32_t)(__ldg(doc_row + j) == doc_i) << (uint32_t)(j - jc);
                }
                return bits;
              };
              w &= mask_word_rolled(p.mask.n, mask_ops, ctl->arg, ipos, jc, eq);
            }
            // select by c without dynamic indexing
  #pragma unroll
            for (int c2 = 0; c2 < C::NW; ++c2) wd[c2] = (c == c2) ? w : wd[c2];
          }
        }
        // the staging of the last item's output has been read by its store
        if (r == 0 && stg_pending) {
          bulk_wait_read0();
          if (C::STAGE_IN_RING) mbar_arrive(b_stg);
          stg_pending = false;
        }
        if (!warp_wait(b_s, t & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[BK];
        if constexpr (BK == 128)
          tmem_ld128f(tS, s);
        else
          tmem_ld64f(tS, s);
        if constexpr (C::EARLY_S) {  // S is in registers: the next step's S may overwrite it
          tc_fence_before();
          mbar_arrive(b_sfree);
        }
        if (msk) {
  #pragma unroll
          for (int e = 0; e < BK; ++e) s[e] = ((wd[e >> 5] >> (e & 31)) & 1u) ? s[e] : -INFINITY;
        }

        // ALiBi: -slope (i - j) = slope e - slope (i - j0) for column e of the tile.
        // The e term joins S in place, in units of the scaled logit
        // (s_e + e slope / scale), so that the maximum and the exponent
        // arguments below are those of the plain score; the j0 term is `base`.
        const float base = slope_l2 * (float)(ipos - j0);
        if constexpr (SCORE == FA_S_ALIBI) {
  #pragma unroll
          for (int e = 0; e < BK; ++e) s[e] = fmaf(slope_sc, (float)e, s[e]);
        }
        // Learned bias: column e's entry is clamp(b - e, 0, L - 1) with b the
        // distance q_pos - j0 - d0 (held within [-BK, L + BK], which changes no
        // entry, so that the per-column arithmetic stays in 32 bits); it joins S
        // in place in units of the scaled logit, like ALiBi's column term.
        if constexpr (SCORE == FA_S_RELBIAS) {
          const int64_t bb = ipos - j0 - p.bias_d0;
          const int b = (int)max((int64_t)-BK, min(bb, (int64_t)p.bias_len + BK));
          const float inv_scale = 1.0f / p.scale;
  #pragma unroll
          for (int e = 0; e < BK; ++e) s[e] = fmaf(__ldg(bias_h + min(max(b - e, 0), p.bias_len - 1)), inv_scale, s[e]);
        }
        // -- row maximum in log2 units (4 independent chains)
        float mx;
        {
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
  #pragma unroll
          for (int e = 0; e < BK; e += 8) {
            a0 = max3f(a0, s[e], s[e + 1]);
            a1 = max3f(a1, s[e + 2], s[e + 3]);
            a2 = max3f(a2, s[e + 4], s[e + 5]);
            a3 = max3f(a3, s[e + 6], s[e + 7]);
          }
          mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
          if constexpr (SCORE == FA_S_SOFTCAP) {
            mx = (mx == -INFINITY) ? -INFINITY : cap_l2 * tanh_fast(mx * sc_over_cap);  // soft-cap is increasing
          } else {
            mx *= sc_l2;  // scale > 0 keeps the order
            if constexpr (SCORE == FA_S_ALIBI) mx -= base;
          }
        }

        const float m_new = fmaxf(m, mx);
        bool need = false;
        if (jj == 0)
          m = m_new;
        else
          need = m_new > m + kRescaleThreshold;
        float alpha = 1.0f;
        if (need) {
          alpha = ex2_approx(m - m_new);
          l *= alpha;
          m = m_new;
        }
        const bool rescale = __any_sync(0xffffffffu, need);  // O is rescaled below, once S is no longer live
        const float m_use = (m == -INFINITY) ? 0.f : m;
        // P and O may be written once the last P V is done (with P in columns of its
        // own that is a wait -- met at once unless the next S runs ahead; else S of
        // this step came after it)
        if constexpr (C::SP) {
          if (jj > 0 && !warp_wait(b_pfree, (t - 1) & 1, &ctl->abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // -- P = 2^(x - m) as bf16 into TMEM (over the consumed S columns, or its
        //    own), row sum (4 chains)
        {
          float2 c01 = make_float2(0.f, 0.f), c23 = make_float2(0.f, 0.f);
          const float off = -(base + m_use);
          // exponent arguments of elements e, e + 1 (two lanes of packed arithmetic)
          auto parg = [&](int e) -> float2 {
            if constexpr (SCORE == FA_S_NONE) {
              return fma2(make_float2(s[e], s[e + 1]), make_float2(sc_l2, sc_l2), make_float2(-m_use, -m_use));
            } else if constexpr (SCORE == FA_S_SOFTCAP) {
              // c tanh(x / c) log2(e) - m with tanh(t) = 1 - 2 / (1 + e^{2t}):
              // (c log2(e) - m) - 2 c log2(e) / (1 + 2^{S sc_cap2}), packed in pairs
              const float2 u = mul2(make_float2(s[e], s[e + 1]), make_float2(sc_cap2, sc_cap2));
              const float2 d = add2(make_float2(ex2_approx(u.x), ex2_approx(u.y)), make_float2(1.0f, 1.0f));
              float2 x = fma2(make_float2(rcp_approx(d.x), rcp_approx(d.y)), make_float2(-2.0f * cap_l2, -2.0f * cap_l2),
                              make_float2(cap_l2 - m_use, cap_l2 - m_use));
              if (msk) {
                x.x = (s[e] == -INFINITY) ? -INFINITY : x.x;
                x.y = (s[e + 1] == -INFINITY) ? -INFINITY : x.y;
              }
              return x;
            } else {
              return fma2(make_float2(s[e], s[e + 1]), make_float2(sc_l2, sc_l2), make_float2(off, off));
            }
          };
  #pragma unroll
          for (int c = 0; c < C::NW; ++c) {
            uint32_t pk[16];
  #pragma unroll
            for (int e2 = 0; e2 < 16; e2 += 2) {
              const int e = 32 * c + 2 * e2;
              const float2 x01 = parg(e), x23 = parg(e + 2);
              const float2 p01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
              const float2 p23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
              c01 = add2(c01, p01);
              c23 = add2(c23, p23);
              pk[e2] = pack_bf16x2(p01.x, p01.y);
              pk[e2 + 1] = pack_bf16x2(p23.x, p23.y);
            }
            tmem_st16(tS + C::T_P + 16 * c, pk);
            if (c == 1) {
              // P of the first 64 keys is in: P V over them may start, once O has
              // been rescaled (the last P V is done: see above)
              if (rescale) {
  #pragma unroll 1
                for (int c3 = 0; c3 < D / 32; ++c3) {
                  float o[32];
                  tmem_ld32f(tO + 32 * c3, o);
  #pragma unroll
                  for (int e = 0; e < 32; ++e) o[e] *= alpha;
                  tmem_st32f(tO + 32 * c3, o);
                }
              }
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(b_ph);
            }
          }
          const float2 cs = add2(c01, c23);
          l += cs.x + cs.y;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_p);
      }
      // ---- epilogue: out = O / l (0 for a row that saw nothing), LSE = ln(2) (m + log2 l);
      //      one decision for the whole group, so that every thread takes the
      //      same named barriers (the first also orders thread 0's confirmation
      //      that the last store has read the staging before it is rewritten)
      if (ok && !warp_wait(b_o, u & 1, &ctl->abort)) ok = false;
      ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.0f / l : 0.f;
      {
        float o[D];
        if constexpr (D == 128)
          tmem_ld128f(tO, o);
        else
          tmem_ld64f(tO, o);
        tc_fence_before();
        mbar_arrive(b_of);  // O may be overwritten by the next item's first P V
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint8_t* chunk = sOut + (c / 2) * 16384 + r * 128;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float* oc = o + 32 * c + 8 * q4;
            uint4 w;
            w.x = pack_bf16x2(oc[0] * inv, oc[1] * inv);
            w.y = pack_bf16x2(oc[2] * inv, oc[3] * inv);
            w.z = pack_bf16x2(oc[4] * inv, oc[5] * inv);
            w.w = pack_bf16x2(oc[6] * inv, oc[7] * inv);
            const int piece = (c % 2) * 4 + q4;  // 16-byte piece within the 128-byte row
            *reinterpret_cast<uint4*>(chunk + ((piece ^ (r & 7)) << 4)) = w;
          }
        }
      }
      if (i < p.q_len) lse_out[(int64_t)bh * p.q_len + i] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (r == 0) {
        for (int c = 0; c < C::NC; ++c) tma_store_3d(&tm_o, smem_u32(sOut + c * 16384), c * 64, I * 128, bh);
        bulk_commit();
        stg_pending = true;
      }
      mbar_arrive(smem_u32(&ctl->desc_empty[dsl]));
      ++u;
    }
    if (!ok) fail(p, ctl);
    if (r == 0 && stg_pending) bulk_wait0();  // the last output store has completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int SCORE, int BK>
cudaError_t launch_fwd_t(const AttnArgs& a, const FwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  const uint64_t bh = (uint64_t)a.B * a.H;
  // keys / values: [B*H][kv_len][D], or the paged pools [H][n_pages * 128][D]
  const bool paged = a.page_table != nullptr;
  const uint64_t kv_rows = paged ? (uint64_t)a.n_pages * 128 : (uint64_t)a.kv_len;
  const uint64_t kv_z = paged ? (uint64_t)a.H : bh;
  CUtensorMap mq, mk, mv, mo;
  const bool ok = encode_tmap_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.q, D, a.q_len, bh, 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_tmap_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.k, D, kv_rows, kv_z, 64, BK,
                                 CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_tmap_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.v, D, kv_rows, kv_z, 64, BK,
                                 CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_tmap_3d(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.out, D, a.q_len, bh, 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    *enc_failed = true;
    return cudaErrorUnknown;
  }
  constexpr size_t smem = fwd_smem_bytes<D, BK>();
  static PerDeviceOnce attr_once;
  cudaError_t e = attr_once.run([] {
    return cudaFuncSetAttribute(fwd_kernel<D, SCORE, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  // persistent: two CTAs per SM (or one per item, when there are fewer)
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.B * a.H * a.nq;
  if (items >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)std::min<int64_t>(items, 2 * (int64_t)sms);
  if (grid > 0)
    fwd_kernel<D, SCORE, BK><<<grid, 192, smem, stream>>>(mq, mk, mv, mo, a, t.lse,
                                                          static_cast<__nv_bfloat16*>(t.out));
  return cudaGetLastError();
}

}  // namespace

#ifdef FA_TEST_HOOKS
cudaError_t test_hook_forward(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(g_hook_skip_first_k, &v, sizeof(v));
}
#endif

template <int BK>
cudaError_t launch_forward_bk(const AttnArgs& a, const FwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  if (a.D == 64) {
    if (a.score_op == FA_S_SOFTCAP) return launch_fwd_t<64, FA_S_SOFTCAP, BK>(a, t, stream, enc_failed);
    if (a.score_op == FA_S_ALIBI) return launch_fwd_t<64, FA_S_ALIBI, BK>(a, t, stream, enc_failed);
    if (a.score_op == FA_S_RELBIAS) return launch_fwd_t<64, FA_S_RELBIAS, BK>(a, t, stream, enc_failed);
    return launch_fwd_t<64, FA_S_NONE, BK>(a, t, stream, enc_failed);
  }
  if (a.score_op == FA_S_SOFTCAP) return launch_fwd_t<128, FA_S_SOFTCAP, BK>(a, t, stream, enc_failed);
  if (a.score_op == FA_S_ALIBI) return launch_fwd_t<128, FA_S_ALIBI, BK>(a, t, stream, enc_failed);
  if (a.score_op == FA_S_RELBIAS) return launch_fwd_t<128, FA_S_RELBIAS, BK>(a, t, stream, enc_failed);
  return launch_fwd_t<128, FA_S_NONE, BK>(a, t, stream, enc_failed);
}

cudaError_t launch_forward(const AttnArgs& a, const FwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  *enc_failed = false;
  if (a.kv_block == 64) {
    if (a.page_table != nullptr) return cudaErrorInvalidValue;  // paged caches use 128-row pages
    return launch_forward_bk<64>(a, t, stream, enc_failed);
  }
  return launch_forward_bk<128>(a, t, stream, enc_failed);
}

}  // namespace fa
