// decode.cu -- the short-query forward (tutorial "FlexAttention in PyTorch",
// "Decoding and paged KV caches": a dedicated decoding path for short queries,
// on a plain or a paged key / value cache).
//
// With q_len <= 16 the work is one pass over the listed key / value tiles of
// each (b, h): reading K and V dominates, so it runs on CUDA cores, and the
// tiles of every (b, h) are split over several CTAs (split-KV) so that a small
// batch still keeps every SM loading:
//
//  decode_partial_kernel  grid (splits, B*H), 8 compute warps and a loader
//      warp.  Its share of the (b, h)'s listed key tiles (FULL ones first,
//      then PARTIAL, as the forward), three K / V stages loaded by TMA with
//      the forward's swizzled maps (so a paged pool works the same way) and
//      released by the compute warps through mbarriers.  Each compute warp
//      owns 16 keys of every tile and runs on its own: scores with a lane
//      pair per key (half of the head dim each), the mask on PARTIAL tiles
//      (row intervals, else the program) and the score mod, an online softmax
//      over its keys, and P V into its own accumulators (4 or 2 output columns
//      per lane); the warps merge by their running maxima after the last tile.
//      Keys past kv_len are never read, so the rows of a last page past kv_len
//      do not matter.  Writes the share's out (normalised) and LSE to the
//      workspace.
//  decode_combine_kernel  one block per (b, h, query row), launched as a
//      programmatic dependent of the partial kernel (its launch overlaps the
//      partial kernel's tail; it waits for its results before reading):
//      lse = log sum_s e^{lse_s},  out = sum_s e^{lse_s - lse} out_s.
#include <cfloat>
#include <cmath>

#include <algorithm>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDecWarps = 8;                       // compute warps; warp kDecWarps loads
constexpr int kDecThreads = 32 * (kDecWarps + 1);
constexpr int kDecStages = 3;
constexpr int kDecMaxSplits = 64;
constexpr int kKeysPerWarp = 128 / kDecWarps;     // 16 keys of every tile per compute warp

template <int D>
struct DecCfg {
  static constexpr int TILE = 128 * D * 2;  // bytes of one K or V tile: D / 64 swizzled boxes of 128 x 64
  static constexpr int NH = D / 16;         // 16-byte chunks in half a key row
  static constexpr int CPL = D / 32;        // output columns per lane
};

template <int D>
constexpr size_t dec_smem_bytes() {
  return 1024 + (size_t)kDecStages * 2 * DecCfg<D>::TILE  // K / V stages (1024-aligned for the swizzle)
         + (size_t)FA_DECODE_MAX_Q * D * 4                // q, fp32
         + (size_t)kDecWarps * FA_DECODE_MAX_Q * kKeysPerWarp * 4  // each warp's probabilities
         + (size_t)2 * kDecWarps * FA_DECODE_MAX_Q * 4    // each warp's running max and sum per row
         + 2 * kDecStages * 8 + 16;                       // mbarriers, abort flag
}

// 1 / x by the special-function unit (the soft-cap's tanh(t) = 1 - 2 / (1 + e^{2t}),
// exact at both saturations, absolute error a few ulp of 1)
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Warp roles: warps 0..7 compute, each on keys [16 w, 16 w + 16) of every tile
// with its own online softmax and output accumulators (no block barrier per
// tile); warp 8 loads K / V into the stages.  Within a compute warp, lane
// pair (2k, 2k + 1) owns key 16 w + k for the scores (one half of the head dim
// each; the second half starts four chunks on, so that with the 128-byte
// swizzle the eight lanes of a shared-memory phase hit eight distinct bank
// groups), and lane l owns output columns [CPL l, CPL l + CPL) for P V.
template <int D, int SCORE, int QB>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ AttnArgs p, const __nv_bfloat16* __restrict__ q,
                          float* __restrict__ ws_out, float* __restrict__ ws_lse, int splits) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sKV = base;
  float* sQ = reinterpret_cast<float*>(base + kDecStages * 2 * C::TILE);
  float* sPw = sQ + FA_DECODE_MAX_Q * D;                              // [warp][row][key]
  float* sMw = sPw + kDecWarps * FA_DECODE_MAX_Q * kKeysPerWarp;      // [warp][row]
  float* sLw = sMw + kDecWarps * FA_DECODE_MAX_Q;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sLw + kDecWarps * FA_DECODE_MAX_Q);
  uint64_t* empty_bar = full_bar + kDecStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty_bar + kDecStages);
  __shared__ int32_t s_arg[FA_MAX_MASK_NODES];

  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int bm = (p.Bm == 1) ? 0 : b, hm = (p.Hm == 1) ? 0 : h;
  const int ql = p.q_len;
  const int64_t row = ((int64_t)bm * p.Hm + hm) * p.nq;  // the (only) query-tile row
  __shared__ int s_count[2];
  if (t == 0) {
    // A block mask built for a longer, bucketed cache lists key tiles past the
    // current kv_len too; the lists are ascending, so those are their tails.
    int nf = __ldg(p.full_num + row), np = __ldg(p.kv_num + row);
    while (nf > 0 && (int64_t)__ldg(p.full_idx + row * p.nkv + nf - 1) * 128 >= p.kv_len) --nf;
    while (np > 0 && (int64_t)__ldg(p.kv_idx + row * p.nkv + np - 1) * 128 >= p.kv_len) --np;
    s_count[0] = nf;
    s_count[1] = nf + np;
  }

  for (int e = t; e < ql * D; e += kDecThreads) sQ[e] = __bfloat162float(q[(int64_t)bh * ql * D + e]);
  if (t < p.mask.n) s_arg[t] = node_arg(p.mask, t, bm);
  if (t == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kDecWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int n_full = s_count[0], n = s_count[1];
  const int p0 = (int)((int64_t)n * split / splits), p1 = (int)((int64_t)n * (split + 1) / splits);
  auto tile_at = [&](int pos) {
    return pos < n_full ? __ldg(p.full_idx + row * p.nkv + pos) : __ldg(p.kv_idx + row * p.nkv + pos - n_full);
  };

  bool ok = true;
  float m_run[QB], l_run[QB];
  float o[QB][C::CPL];
  if (warp == kDecWarps) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int issued_end = p0;
      for (int pos = p0; pos < p1; ++pos) {
        const int st = (pos - p0) % kDecStages, use = (pos - p0) / kDecStages;
        if (use > 0 && !mbar_wait(smem_u32(&empty_bar[st]), (use - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int J = tile_at(pos);
        int kv_row = J * 128, kv_z = bh;
        if (p.page_table != nullptr) {
          int page = __ldg(p.page_table + (int64_t)b * p.nkv + J);
          if (page < 0 || page >= p.n_pages) {  // reported; page 0 is read instead
            atomicOr(p.status, kStatusCheck);
            page = 0;
          }
          kv_row = page * 128;
          kv_z = h;
        }
        const uint32_t bar = smem_u32(&full_bar[st]);
        mbar_arrive_expect_tx(bar, 2 * C::TILE);
        uint8_t* dk = sKV + (size_t)st * 2 * C::TILE;
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(smem_u32(dk + c * 16384), &tm_k, bar, c * 64, kv_row, kv_z);
          tma_load_3d(smem_u32(dk + C::TILE + c * 16384), &tm_v, bar, c * 64, kv_row, kv_z);
        }
        issued_end = pos + 1;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.status, kStatusTimeout);
      }
      // every copy issued lands before the CTA moves on (bounded waits)
      for (int pos = max(p0, issued_end - kDecStages); pos < issued_end; ++pos)
        mbar_wait(smem_u32(&full_bar[(pos - p0) % kDecStages]), ((pos - p0) / kDecStages) & 1, nullptr);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const uint64_t mask_ops = pack_ops(p.mask);
    const int32_t* doc_row = p.mask.has_doc ? p.mask.doc + (int64_t)bm * p.mask.doc_len : nullptr;
    const int qoff = (int)p.mask.q_off;
    float slope_l2 = 0.f, cap = 1.f;
    if constexpr (SCORE == FA_S_ALIBI) slope_l2 = __ldg(p.score_param + h) * kLog2e;
    const float* bias_h = nullptr;  // RELBIAS: this head's table
    if constexpr (SCORE == FA_S_RELBIAS) bias_h = p.score_param + (int64_t)h * p.bias_len;
    float cap_l2 = 0.f, sc_cap2 = 0.f;  // soft-cap: c log2(e), and S -> the exponent of e^{2 x / c} in base 2
    if constexpr (SCORE == FA_S_SOFTCAP) {
      cap = __ldg(p.score_param);
      cap_l2 = cap * kLog2e;
      sc_cap2 = (p.scale / cap) * (2.0f * kLog2e);
    }
#pragma unroll
    for (int i = 0; i < QB; ++i) {
      m_run[i] = -INFINITY;
      l_run[i] = 0.f;
#pragma unroll
      for (int c = 0; c < C::CPL; ++c) o[i][c] = 0.f;
    }
    const int kk = lane / 2, half = lane % 2;
    const int r = kKeysPerWarp * warp + kk;  // this lane pair's key row in the tile
    float* pw = sPw + warp * FA_DECODE_MAX_Q * kKeysPerWarp;
    // P V: columns [CPL lane, CPL lane + CPL): box, 16-byte chunk and byte within it
    const int col0 = C::CPL * lane;
    const int vbox = col0 / 64, vchunk = (col0 % 64) / 8, vbyte = (col0 % 8) * 2;
    for (int pos = p0; pos < p1; ++pos) {
      const int st = (pos - p0) % kDecStages, use = (pos - p0) / kDecStages;
      const bool got = mbar_wait(smem_u32(&full_bar[st]), use & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const int J = tile_at(pos);
      const bool full = pos < n_full;
      const int rows_valid = min(128, p.kv_len - J * 128);
      const uint8_t* sK = sKV + (size_t)st * 2 * C::TILE;
      const uint8_t* sV = sK + C::TILE;
      const bool key_ok = r < rows_valid;
      const int j = J * 128 + r;

      // -- scores of key r: this lane's half of q . k, the pair's sum by a shuffle
      float a[QB];
#pragma unroll
      for (int i = 0; i < QB; ++i) a[i] = 0.f;
      if (key_ok) {
#pragma unroll
        for (int cc = 0; cc < C::NH; ++cc) {
          const int c = half * C::NH + ((cc + 4 * half) % C::NH);
          const uint4 kw =
              *reinterpret_cast<const uint4*>(sK + (c / 8) * 16384 + r * 128 + (((c % 8) ^ (r & 7)) << 4));
          float kf[8];
          const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(k2[e]);
            kf[2 * e] = f.x;
            kf[2 * e + 1] = f.y;
          }
#pragma unroll
          for (int i = 0; i < QB; ++i) {
            if (i < ql) {
              const float4 qa = *reinterpret_cast<const float4*>(sQ + i * D + c * 8);
              const float4 qb = *reinterpret_cast<const float4*>(sQ + i * D + c * 8 + 4);
              float x = a[i];
              x = fmaf(qa.x, kf[0], x);
              x = fmaf(qa.y, kf[1], x);
              x = fmaf(qa.z, kf[2], x);
              x = fmaf(qa.w, kf[3], x);
              x = fmaf(qb.x, kf[4], x);
              x = fmaf(qb.y, kf[5], x);
              x = fmaf(qb.z, kf[6], x);
              x = fmaf(qb.w, kf[7], x);
              a[i] = x;
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < QB; ++i) a[i] += __shfl_xor_sync(0xffffffffu, a[i], 1);
      // mask (FULL tiles: every in-range pair) and score mod, log2 units
      uint32_t w = 0;  // bit i: (i, j) visible
      if (key_ok) {
        if (full) {
          w = 0xffffffffu;
        } else {
          const int4 seg = __ldg(p.row_segs + ((int64_t)bm * 2 + 1) * p.seg_len + j);
          if (seg.x >= 0) {
            w = seg_word(seg, 0);
          } else {
            int run_lo = 0, run_hi = 0;
            const bool use_run = doc_row != nullptr && doc_run(p.mask, bm, j, run_lo, run_hi);
            const int32_t doc_j = doc_row != nullptr ? __ldg(doc_row + j) : 0;
            // query row i is position i + q_off of the sequence
            auto eq = [&]() {
              if (use_run) return range_bits(run_lo, run_hi, qoff);
              uint32_t bits = 0;
              for (int i = 0; i < ql; ++i) bits |= (uint32_t)(__ldg(doc_row + i + qoff) == doc_j) << i;
              return bits;
            };
            w = mask_word_t_rolled(p.mask.n, mask_ops, s_arg, j, qoff, eq);
          }
        }
      }
      // -- online softmax over this warp's 16 keys (lane pairs hold equal values,
      //    so the reductions run over the lanes of one parity)
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        if (i < ql) {
          float sc = -INFINITY;
          if ((w >> i) & 1u) {
            const float x = a[i] * p.scale;
            if constexpr (SCORE == FA_S_SOFTCAP) {
              // c tanh(x / c) log2(e) with tanh(t) = 1 - 2 / (1 + e^{2t})
              sc = fmaf(-2.0f * cap_l2, rcp_approx(1.0f + ex2_approx(a[i] * sc_cap2)), cap_l2);
            } else if constexpr (SCORE == FA_S_ALIBI) {
              sc = fmaf(x, kLog2e, -slope_l2 * (float)(i + qoff - j));
            } else if constexpr (SCORE == FA_S_RELBIAS) {  // entry clamp(q_pos - j - d0, 0, L - 1)
              const int64_t d = (int64_t)(i + qoff) - j - p.bias_d0;
              const int te = (int)max((int64_t)0, min(d, (int64_t)p.bias_len - 1));
              sc = (x + __ldg(bias_h + te)) * kLog2e;
            } else {
              sc = x * kLog2e;
            }
          }
          float mx = sc;
#pragma unroll
          for (int o2 = 2; o2 <= 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
          const float m_new = fmaxf(m_run[i], mx);
          const float mu = (m_new == -INFINITY) ? 0.f : m_new;
          const float pv = ex2_approx(sc - mu);
          float sum = pv;
#pragma unroll
          for (int o2 = 2; o2 <= 16; o2 <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
          const float alpha = ex2_approx(m_run[i] - mu);
          l_run[i] = fmaf(l_run[i], alpha, sum);
          m_run[i] = m_new;
#pragma unroll
          for (int c = 0; c < C::CPL; ++c) o[i][c] *= alpha;
          if (half == 0) pw[i * kKeysPerWarp + kk] = pv;
        }
      }
      __syncwarp();
      // -- P V over this warp's valid keys
      const int kn = min(kKeysPerWarp, rows_valid - kKeysPerWarp * warp);
#pragma unroll 4
      for (int k2 = 0; k2 < kn; ++k2) {
        const int jr = kKeysPerWarp * warp + k2;
        const uint8_t* vp = sV + vbox * 16384 + jr * 128 + ((vchunk ^ (jr & 7)) << 4) + vbyte;
        float vv[C::CPL];
        if constexpr (C::CPL == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(vp);
          const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
          const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
          vv[0] = v01.x;
          vv[1] = v01.y;
          vv[2] = v23.x;
          vv[3] = v23.y;
        } else {
          const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vp));
          vv[0] = v01.x;
          vv[1] = v01.y;
        }
#pragma unroll
        for (int i = 0; i < QB; ++i) {
          if (i < ql) {
            const float pij = pw[i * kKeysPerWarp + k2];
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) o[i][c] = fmaf(pij, vv[c], o[i][c]);
          }
        }
      }
      __syncwarp();  // this warp is done with the stage and its probabilities
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.status, kStatusTimeout);
    }
  }
  __syncthreads();  // every warp is done with the stages
  if (*abort_flag) return;

  // the warps' rows merge: running max and sum per warp, outputs through the idle stages
  float* red = reinterpret_cast<float*>(sKV);  // [warp][row][D]
  if (warp < kDecWarps) {
#pragma unroll
    for (int i = 0; i < QB; ++i) {
      if (i < ql) {
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) red[((size_t)warp * FA_DECODE_MAX_Q + i) * D + C::CPL * lane + c] = o[i][c];
        if (lane == 0) {
          sMw[warp * FA_DECODE_MAX_Q + i] = m_run[i];
          sLw[warp * FA_DECODE_MAX_Q + i] = l_run[i];
        }
      }
    }
  }
  __syncthreads();
  const int64_t r0 = ((int64_t)split * p.B * p.H + bh) * ql;  // this share's first row in the workspace
  for (int e = t; e < ql * D; e += kDecThreads) {
    const int i = e / D, dd = e % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kDecWarps; ++w2) mx = fmaxf(mx, sMw[w2 * FA_DECODE_MAX_Q + i]);
    float acc = 0.f, l = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < kDecWarps; ++w2) {
        const float mw = sMw[w2 * FA_DECODE_MAX_Q + i];
        if (mw == -INFINITY) continue;
        const float sc = ex2_approx(mw - mx);
        l = fmaf(sLw[w2 * FA_DECODE_MAX_Q + i], sc, l);
        acc = fmaf(red[((size_t)w2 * FA_DECODE_MAX_Q + i) * D + dd], sc, acc);
      }
    }
    ws_out[(r0 + i) * D + dd] = (l > 0.f) ? acc / l : 0.f;
    if (dd == 0) ws_lse[r0 + i] = (l > 0.f) ? (mx + log2f(l)) * kLn2 : -INFINITY;
  }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ ws_out,
                                                           const float* __restrict__ ws_lse, int splits,
                                                           int64_t rows, __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
  pdl_wait_then_release();       // launched while the partial kernel drains
  const int64_t r = blockIdx.x;  // (b, h, query row)
  const int d = threadIdx.x;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, __ldg(ws_lse + s * rows + r));
  float wsum = 0.f, acc = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ls = __ldg(ws_lse + s * rows + r);
      if (ls == -INFINITY) continue;
      const float wgt = expf(ls - m);
      wsum += wgt;
      acc = fmaf(wgt, __ldg(ws_out + (s * rows + r) * D + d), acc);
    }
  }
  out[r * D + d] = __float2bfloat16_rn(m == -INFINITY ? 0.f : acc / wsum);
  if (d == 0) lse[r] = (m == -INFINITY) ? -INFINITY : m + logf(wsum);
}

template <int D, int SCORE, int QB>
cudaError_t launch_decode_t(const AttnArgs& a, const FwdTensors& t, float* ws, int splits, cudaStream_t stream,
                            bool* enc_failed) {
  const uint64_t bh = (uint64_t)a.B * a.H;
  const bool paged = a.page_table != nullptr;
  // rows of each (b, h) in the key / value tensors: the block mask's (bucketed) length
  const uint64_t kv_rows = paged ? (uint64_t)a.n_pages * 128 : (uint64_t)a.kv_cap;
  const uint64_t kv_z = paged ? (uint64_t)a.H : bh;
  CUtensorMap mk, mv;
  if (!encode_tmap_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.k, D, kv_rows, kv_z, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.v, D, kv_rows, kv_z, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B)) {
    *enc_failed = true;
    return cudaErrorUnknown;
  }
  constexpr size_t smem = dec_smem_bytes<D>();
  static PerDeviceOnce attr_once;
  cudaError_t e0 = attr_once.run([] {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D, SCORE, QB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    // all of the unified L1 as shared memory, so that two CTAs fit an SM at D = 64
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_partial_kernel<D, SCORE, QB>,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
  });
  if (e0 != cudaSuccess) return e0;
  const int64_t rows = (int64_t)bh * a.q_len;
  float* ws_out = ws;
  float* ws_lse = ws + (size_t)splits * rows * D;
  decode_partial_kernel<D, SCORE, QB><<<dim3((unsigned)splits, (unsigned)bh), kDecThreads, smem, stream>>>(
      mk, mv, a, static_cast<const __nv_bfloat16*>(t.q), ws_out, ws_lse, splits);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_k(decode_combine_kernel<D>, dim3((unsigned)rows), dim3(D), 0, stream, (const float*)ws_out,
                  (const float*)ws_lse, splits, rows, static_cast<__nv_bfloat16*>(t.out), t.lse);
}

template <int D, int SCORE>
cudaError_t launch_decode_q(const AttnArgs& a, const FwdTensors& t, float* ws, int splits, cudaStream_t stream,
                            bool* enc_failed) {
  if (a.q_len == 1) return launch_decode_t<D, SCORE, 1>(a, t, ws, splits, stream, enc_failed);
  if (a.q_len <= 4) return launch_decode_t<D, SCORE, 4>(a, t, ws, splits, stream, enc_failed);
  return launch_decode_t<D, SCORE, 16>(a, t, ws, splits, stream, enc_failed);
}

}  // namespace

cudaError_t decode_plan(int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, int* splits,
                        size_t* ws_bytes) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // CTAs that fit at once: one per SM at D = 128, two at D = 64 with one query
  // row (registers); the split minimises waves x (tiles per share + a CTA's
  // start-up, about 1.5 tiles), taking the key tiles as all listed
  const int64_t slots = (int64_t)sms * ((D == 64 && q_len == 1) ? 2 : 1);
  const int64_t items = (int64_t)B * H;
  const int64_t nkv = (kv_len + 127) / 128;
  const int64_t s_max = std::max<int64_t>(1, std::min<int64_t>(nkv, kDecMaxSplits));
  int64_t s = 1;
  double best = 0.0;
  for (int64_t c = 1; c <= s_max; ++c) {
    const double waves = (double)((items * c + slots - 1) / slots);
    const double cost = waves * ((double)((nkv + c - 1) / c) + 1.5);
    if (c == 1 || cost < best) {
      best = cost;
      s = c;
    }
  }
  *splits = (int)s;
  *ws_bytes = (size_t)s * items * q_len * (D + 1) * sizeof(float);
  return cudaSuccess;
}

cudaError_t launch_decode(const AttnArgs& a, const FwdTensors& t, void* workspace, int splits, cudaStream_t stream,
                          bool* enc_failed) {
  *enc_failed = false;
  float* ws = static_cast<float*>(workspace);
  if (a.D == 64) {
    if (a.score_op == FA_S_SOFTCAP) return launch_decode_q<64, FA_S_SOFTCAP>(a, t, ws, splits, stream, enc_failed);
    if (a.score_op == FA_S_ALIBI) return launch_decode_q<64, FA_S_ALIBI>(a, t, ws, splits, stream, enc_failed);
    if (a.score_op == FA_S_RELBIAS) return launch_decode_q<64, FA_S_RELBIAS>(a, t, ws, splits, stream, enc_failed);
    return launch_decode_q<64, FA_S_NONE>(a, t, ws, splits, stream, enc_failed);
  }
  if (a.score_op == FA_S_SOFTCAP) return launch_decode_q<128, FA_S_SOFTCAP>(a, t, ws, splits, stream, enc_failed);
  if (a.score_op == FA_S_ALIBI) return launch_decode_q<128, FA_S_ALIBI>(a, t, ws, splits, stream, enc_failed);
  if (a.score_op == FA_S_RELBIAS) return launch_decode_q<128, FA_S_RELBIAS>(a, t, ws, splits, stream, enc_failed);
  return launch_decode_q<128, FA_S_NONE>(a, t, ws, splits, stream, enc_failed);
}

}  // namespace fa
