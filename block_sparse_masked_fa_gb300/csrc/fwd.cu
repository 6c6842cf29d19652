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
// One CTA owns one 128-row query tile of one (b, h); two CTAs share an SM so
// that one's softmax overlaps the other's matrix multiplies.  Warp roles:
//   warps 0-3  softmax + epilogue: thread r owns query row r (TMEM lane r)
//   warp 4     TMA producer (Q once, then K_j / V_j through a ring of slots)
//              and TMEM allocator
//   warp 5     MMA issuer (one thread): S = Q K_j^T into TMEM, then
//              O += P V_j with P read from TMEM
// TMEM (256 columns): S at [0, 128) -- P (bf16 pairs) overwrites its first 64
// columns after the softmax has read S -- and O at [128, 128 + D).
// The running maximum is only moved (and O rescaled) when a new row maximum
// exceeds it by more than 2^8, so most tiles need no O round trip.
#include <cfloat>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
  static constexpr int NC = D / 64;                      // 64-column (128-byte) chunks per tile row
  static constexpr uint32_t TILE = 128u * D * 2u;        // bytes of one 128 x D bf16 tile
  static constexpr int NS = (D == 64) ? 4 : 2;           // K/V ring slots
  static constexpr uint32_t TMEM_COLS = 256;
};

struct FwdCtl {
  uint64_t q_full;
  uint64_t kv_full[4];
  uint64_t kv_empty[4];
  uint64_t s_full;
  uint64_t p_full;
  uint64_t o_full;
  uint64_t fin;
  uint32_t tmem;
  int abort;
  int32_t arg[FA_MAX_MASK_NODES];
  int4 seg[128];  // per query row: its two visible key intervals (block mask row_segs)
};

template <int D>
constexpr size_t fwd_smem_bytes() {
  return 1024 + (size_t)FwdCfg<D>::TILE * (1 + FwdCfg<D>::NS) + sizeof(FwdCtl);
}

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

template <int D, int SCORE>
__global__ void __launch_bounds__(192, 2)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const __grid_constant__ AttnArgs p, float* __restrict__ lse_out) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::TILE;
  FwdCtl* ctl = reinterpret_cast<FwdCtl*>(sKV + C::NS * C::TILE);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // ---- work item: (b, h, query tile I), rows taken longest first
  const int rep = (p.B / p.Bm) * (p.H / p.Hm);
  const int row = p.row_order[blockIdx.x / rep];  // index into [Bm][Hm][nq]
  const int t = blockIdx.x % rep;
  const int I = row % p.nq;
  const int hm = (row / p.nq) % p.Hm;
  const int bm = row / (p.nq * p.Hm);
  const int b = (p.Bm == 1) ? t / (p.H / p.Hm) : bm;
  const int h = (p.Hm == 1) ? t % (p.H / p.Hm) : hm;
  const int bh = b * p.H + h;
  const int n_full = p.full_num[row];
  int n = n_full + p.kv_num[row];
  const int64_t list = (int64_t)row * p.nkv;

  const uint32_t b_q = smem_u32(&ctl->q_full), b_s = smem_u32(&ctl->s_full), b_p = smem_u32(&ctl->p_full),
                 b_o = smem_u32(&ctl->o_full), b_fin = smem_u32(&ctl->fin);
  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(smem_u32(&ctl->kv_full[s]), 1);
      mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
    }
    mbar_init(b_s, 1);
    mbar_init(b_p, 128);
    mbar_init(b_o, 1);
    mbar_init(b_fin, 1);
    // once any CTA has given up, later CTAs do no work (one decision per CTA)
    ctl->abort = (*reinterpret_cast<volatile uint32_t*>(p.status) & kStatusTimeout) ? 1 : 0;
    fence_mbar_init();
  }
  if (threadIdx.x < p.mask.n) ctl->arg[threadIdx.x] = node_arg(p.mask, threadIdx.x, bm);
  if (warp == 4) {
    tmem_alloc(smem_u32(&ctl->tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const bool skip = ctl->abort != 0;
  if (skip) n = 0;

  auto tile_of = [&](int jj) -> int { return jj < n_full ? p.full_idx[list + jj] : p.kv_idx[list + jj - n_full]; };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(b_q, C::TILE);
      for (int c = 0; c < C::NC; ++c) tma_load_3d(smem_u32(sQ + c * 16384), &tm_q, b_q, c * 64, I * 128, bh);
      int issued = 0;
      bool ok = true;
      for (int t2 = 0; t2 < 2 * n; ++t2) {
        const int slot = t2 % C::NS, use = t2 / C::NS;
        if (use > 0 && !mbar_wait(smem_u32(&ctl->kv_empty[slot]), (use - 1) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        const int J = tile_of(t2 >> 1);
        const uint32_t bar = smem_u32(&ctl->kv_full[slot]);
        mbar_arrive_expect_tx(bar, C::TILE);
        const CUtensorMap* m = (t2 & 1) ? &tm_v : &tm_k;
        for (int c = 0; c < C::NC; ++c)
          tma_load_3d(smem_u32(sKV + slot * C::TILE + c * 16384), m, bar, c * 64, J * 128, bh);
        issued = t2 + 1;
      }
      if (!ok) fail(p, ctl);
      // drain: every copy this CTA started lands before it exits
      mbar_wait(b_q, 0, nullptr);
      for (int t2 = max(0, issued - C::NS); t2 < issued; ++t2)
        mbar_wait(smem_u32(&ctl->kv_full[t2 % C::NS]), (t2 / C::NS) & 1, nullptr);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);  // Q (K-major) x K (K-major)
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);     // P (TMEM) x V (MN-major)
      bool ok = mbar_wait(b_q, 0, &ctl->abort);
      const uint32_t q_base = smem_u32(sQ);
      for (int jj = 0; ok && jj < n; ++jj) {
        const int tk = 2 * jj, sk = tk % C::NS;
        if (!mbar_wait(smem_u32(&ctl->kv_full[sk]), (tk / C::NS) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_u32(sKV + sk * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
          mma_ss(tmem, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024), kIdS, kk > 0);
        }
        mma_commit(smem_u32(&ctl->kv_empty[sk]));
        mma_commit(b_s);
        if (!mbar_wait(b_p, jj & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        const int tv = tk + 1, sv = tv % C::NS;
        if (!mbar_wait(smem_u32(&ctl->kv_full[sv]), (tv / C::NS) & 1, &ctl->abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_base = smem_u32(sKV + sv * C::TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 128, tmem + kk * 8, sdesc_sw128(v_base + kk * 2048, 16384, 1024), kIdO, (jj > 0 || kk > 0));
        mma_commit(smem_u32(&ctl->kv_empty[sv]));
      }
      if (ok)
        mma_commit(b_o);
      else
        fail(p, ctl);
      // drain: no tcgen05 operation of this CTA is in flight past this point
      mma_commit(b_fin);
      mbar_wait(b_fin, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x;  // 0..127, TMEM lane
    const int i = I * 128 + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off;
    const uint32_t tO = tmem + lane_off + 128;
    // the list entry of the first step and this row's visible key columns as
    // two intervals (kept in shared memory: read on partial tiles only); the
    // document id and run of the row only for rows the intervals do not
    // describe, which evaluate the program per word
    int J_next = n > 0 ? tile_of(0) : 0;
    const int4 seg0 = __ldg(p.row_segs + (int64_t)bm * 2 * p.seg_len + min(i, p.q_len - 1));
    ctl->seg[r] = seg0;
    const int32_t* doc_row = p.mask.has_doc ? p.mask.doc + (int64_t)bm * p.mask.doc_len : nullptr;
    int32_t doc_i = 0;
    int run_lo = 0, run_hi = 0;  // with sorted ids: doc[j] == doc[i] exactly for j in [run_lo, run_hi)
    bool use_run = false;
    if (seg0.x < 0 && doc_row != nullptr) {
      doc_i = __ldg(doc_row + min(i, p.q_len - 1));
      use_run = doc_run(p.mask, bm, min(i, p.q_len - 1), run_lo, run_hi);
    }

    const uint64_t mask_ops = pack_ops(p.mask);
    const float sc_l2 = p.scale * kLog2e;  // logit -> log2 units
    float cap_l2 = 0.f, sc_over_cap = 0.f, slope_l2 = 0.f;
    if constexpr (SCORE == FA_S_SOFTCAP) {
      const float cap = __ldg(p.score_param);
      cap_l2 = cap * kLog2e;
      sc_over_cap = p.scale / cap;
    }
    if constexpr (SCORE == FA_S_ALIBI) slope_l2 = __ldg(p.score_param + h) * kLog2e;

    float m = -INFINITY;  // reference maximum, log2 units
    float l = 0.f;
    bool ok = true;
    // the list entry of the next step is fetched one step ahead, off the path
    // from the S wait to the mask words
    for (int jj = 0; jj < n; ++jj) {
      const bool partial = jj >= n_full;
      const int J = J_next;
      if (jj + 1 < n) J_next = tile_of(jj + 1);
      const int64_t j0 = (int64_t)J * 128;
      const bool ragged = j0 + 128 > p.kv_len;
      const bool msk = partial || ragged;
      // visibility words of the 4 x 32 key columns, computed before S is loaded
      uint32_t wd[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (msk) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const int jc = (int)j0 + 32 * c;
          uint32_t w = low_bits((int64_t)p.kv_len - jc);
          const int4 sg = ctl->seg[r];
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
            w &= mask_word_rolled(p.mask.n, mask_ops, ctl->arg, i, jc, eq);
          }
          // select by c without dynamic indexing
          wd[0] = (c == 0) ? w : wd[0];
          wd[1] = (c == 1) ? w : wd[1];
          wd[2] = (c == 2) ? w : wd[2];
          wd[3] = (c == 3) ? w : wd[3];
        }
      }
      if (!warp_wait(b_s, jj & 1, &ctl->abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
      tmem_ld128f(tS, s);
      if (msk) {
#pragma unroll
        for (int e = 0; e < 128; ++e) s[e] = ((wd[e >> 5] >> (e & 31)) & 1u) ? s[e] : -INFINITY;
      }

      const float base = slope_l2 * (float)(i - (int)j0);  // ALiBi: -slope (i - j) = -base + slope * e
      // -- row maximum in log2 units (4 independent chains)
      float mx;
      {
        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
        for (int e = 0; e < 128; e += 8) {
          if constexpr (SCORE == FA_S_ALIBI) {
            float t[8];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
              const float2 v = fma2(make_float2(s[e + u], s[e + u + 1]), make_float2(sc_l2, sc_l2),
                                    make_float2(slope_l2 * (float)(e + u), slope_l2 * (float)(e + u + 1)));
              t[u] = v.x;
              t[u + 1] = v.y;
            }
            a0 = max3f(a0, t[0], t[1]);
            a1 = max3f(a1, t[2], t[3]);
            a2 = max3f(a2, t[4], t[5]);
            a3 = max3f(a3, t[6], t[7]);
          } else {
            a0 = max3f(a0, s[e], s[e + 1]);
            a1 = max3f(a1, s[e + 2], s[e + 3]);
            a2 = max3f(a2, s[e + 4], s[e + 5]);
            a3 = max3f(a3, s[e + 6], s[e + 7]);
          }
        }
        mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        if constexpr (SCORE == FA_S_NONE) {
          mx *= sc_l2;  // scale > 0 keeps the order
        } else if constexpr (SCORE == FA_S_SOFTCAP) {
          mx = (mx == -INFINITY) ? -INFINITY : cap_l2 * tanh_fast(mx * sc_over_cap);  // soft-cap is increasing
        } else {
          mx -= base;
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
      // -- P = 2^(x - m) as bf16 into TMEM (over the consumed S columns), row sum (4 chains)
      {
        float2 c01 = make_float2(0.f, 0.f), c23 = make_float2(0.f, 0.f);
        const float off = -(base + m_use);
        // exponent arguments of elements e, e + 1 (two lanes of packed arithmetic)
        auto parg = [&](int e) -> float2 {
          if constexpr (SCORE == FA_S_NONE) {
            return fma2(make_float2(s[e], s[e + 1]), make_float2(sc_l2, sc_l2), make_float2(-m_use, -m_use));
          } else if constexpr (SCORE == FA_S_SOFTCAP) {
            float2 x = fma2(make_float2(cap_l2, cap_l2),
                            make_float2(tanh_fast(s[e] * sc_over_cap), tanh_fast(s[e + 1] * sc_over_cap)),
                            make_float2(-m_use, -m_use));
            if (msk) {
              x.x = (s[e] == -INFINITY) ? -INFINITY : x.x;
              x.y = (s[e + 1] == -INFINITY) ? -INFINITY : x.y;
            }
            return x;
          } else {
            return fma2(make_float2(s[e], s[e + 1]), make_float2(sc_l2, sc_l2),
                        make_float2(fmaf(slope_l2, (float)e, off), fmaf(slope_l2, (float)(e + 1), off)));
          }
        };
#pragma unroll
        for (int c = 0; c < 4; ++c) {
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
          tmem_st16(tS + 16 * c, pk);
        }
        const float2 cs = add2(c01, c23);
        l += cs.x + cs.y;
      }
      if (rescale) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32f(tO + 32 * c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32f(tO + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_p);
    }
    if (!ok) fail(p, ctl);
    // ---- epilogue: out = O / l (0 for a row that saw nothing), LSE = ln(2) (m + log2 l)
    if (ok && n > 0) {
      if (!warp_wait(b_o, 0, &ctl->abort)) {
        ok = false;
        fail(p, ctl);
      }
      tc_fence_after();
    }
    if (ok && !skip) {
      const float inv = (l > 0.f) ? 1.0f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        if (n > 0) {
          tmem_ld32f(tO + 32 * c, o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        uint8_t* chunk = sQ + (c / 2) * 16384 + r * 128;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16x2(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
          v.y = pack_bf16x2(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
          v.z = pack_bf16x2(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
          v.w = pack_bf16x2(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
          const int piece = (c % 2) * 4 + q4;  // 16-byte piece within the 128-byte row
          *reinterpret_cast<uint4*>(chunk + ((piece ^ (r & 7)) << 4)) = v;
        }
      }
      if (i < p.q_len) lse_out[(int64_t)bh * p.q_len + i] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
    }
    // every softmax thread reaches this barrier, whatever happened above
    named_bar_sync(1, 128);
    if (r == 0 && !skip && !*reinterpret_cast<volatile int*>(&ctl->abort)) {
      for (int c = 0; c < C::NC; ++c) tma_store_3d(&tm_o, smem_u32(sQ + c * 16384), c * 64, I * 128, bh);
      bulk_commit();
      bulk_wait_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int SCORE>
cudaError_t launch_fwd_t(const AttnArgs& a, const FwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  const uint64_t bh = (uint64_t)a.B * a.H;
  CUtensorMap mq, mk, mv, mo;
  const bool ok = encode_tmap_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.q, D, a.q_len, bh, 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_tmap_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.k, D, a.kv_len, bh, 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_tmap_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.v, D, a.kv_len, bh, 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B) &&
                  encode_tmap_3d(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.out, D, a.q_len, bh, 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    *enc_failed = true;
    return cudaErrorUnknown;
  }
  constexpr size_t smem = fwd_smem_bytes<D>();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t items = (int64_t)a.B * a.H * a.nq;
  fwd_kernel<D, SCORE><<<(unsigned)items, 192, smem, stream>>>(mq, mk, mv, mo, a, t.lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(const AttnArgs& a, const FwdTensors& t, cudaStream_t stream, bool* enc_failed) {
  *enc_failed = false;
  if (a.D == 64) {
    if (a.score_op == FA_S_SOFTCAP) return launch_fwd_t<64, FA_S_SOFTCAP>(a, t, stream, enc_failed);
    if (a.score_op == FA_S_ALIBI) return launch_fwd_t<64, FA_S_ALIBI>(a, t, stream, enc_failed);
    return launch_fwd_t<64, FA_S_NONE>(a, t, stream, enc_failed);
  }
  if (a.score_op == FA_S_SOFTCAP) return launch_fwd_t<128, FA_S_SOFTCAP>(a, t, stream, enc_failed);
  if (a.score_op == FA_S_ALIBI) return launch_fwd_t<128, FA_S_ALIBI>(a, t, stream, enc_failed);
  return launch_fwd_t<128, FA_S_NONE>(a, t, stream, enc_failed);
}

}  // namespace fa
