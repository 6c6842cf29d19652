// decode.cu -- the short-query forward (tutorial "FlexAttention in PyTorch",
// "Decoding and paged KV caches": a dedicated decoding path for short queries,
// on a plain or a paged key / value cache).
//
// With q_len <= 16 the work is one pass over the listed key / value tiles of
// each (b, h): reading K and V dominates, so it runs on CUDA cores, and the
// tiles of every (b, h) are split over several CTAs (split-KV) so that a small
// batch still keeps every SM loading:
//
//  decode_partial_kernel  grid (splits, B*H), 256 threads.  Its share of the
//      (b, h)'s listed key tiles (FULL ones first, then PARTIAL, as the
//      forward), three K / V stages loaded by thread 0 with the forward's
//      swizzled TMA maps (so a paged pool works the same way).  Per tile:
//      scores with two threads per key row, each over half of the head dim
//      (the 128-byte swizzle makes the row reads conflict-free; q is read as
//      a broadcast), the mask on PARTIAL tiles (row intervals, else the
//      program) and the score mod; an online softmax per query row (a warp
//      per row); P V with a column pair per thread over a group of keys, the
//      groups added after the last tile.  Keys past kv_len are never read, so
//      the rows of a last page past kv_len do not matter.  Writes the share's
//      out (normalised) and LSE to the workspace.
//  decode_combine_kernel  one block per (b, h, query row):
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
constexpr int kDecThreads = 256;
constexpr int kDecStages = 3;
constexpr int kDecMaxSplits = 64;

template <int D>
struct DecCfg {
  static constexpr int TILE = 128 * D * 2;       // bytes of one K or V tile: D / 64 swizzled boxes of 128 x 64
  static constexpr int NCH = D / 8;              // 16-byte chunks of a key row
  static constexpr int PAIRS = D / 2;            // column pairs of the P V phase
  static constexpr int NG = kDecThreads / PAIRS; // key groups of the P V phase
  static constexpr int KPG = 128 / NG;           // keys per group
};

template <int D>
constexpr size_t dec_smem_bytes() {
  return 1024 + (size_t)kDecStages * 2 * DecCfg<D>::TILE  // K / V stages (1024-aligned for the swizzle)
         + (size_t)FA_DECODE_MAX_Q * D * 4                // q, fp32
         + (size_t)FA_DECODE_MAX_Q * 128 * 4              // scores, then probabilities
         + 3 * FA_DECODE_MAX_Q * 4                        // alpha, m, l per row
         + kDecStages * 8;                                // mbarriers
}

// tanh(t) = 1 - 2 / (1 + e^{2t}); exact at both saturations, absolute error a few ulp of 1.
__device__ __forceinline__ float tanh_fast(float t) {
  const float e = ex2_approx(t * (2.0f * kLog2e));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return fmaf(-2.0f, r, 1.0f);
}

// Thread roles per tile (256 threads):
//   scores   thread (half, key r): t = 128 * half + r sums q . k over chunks
//            [half * NCH / 2, (half + 1) * NCH / 2) of key row r; the halves
//            meet in shared memory, half 0 applies mask and score mod;
//   softmax  warp w owns query rows w, w + 8;
//   P V      thread (group g, pair c): t = PAIRS * g + c accumulates columns
//            2c, 2c + 1 over keys [KPG g, KPG (g + 1)); the groups' sums are
//            added once, after the last tile.
template <int D, int SCORE, int QB>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ AttnArgs p, const __nv_bfloat16* __restrict__ q,
                          float* __restrict__ ws_out, float* __restrict__ ws_lse, int splits) {
  using C = DecCfg<D>;
  constexpr int RW = (QB + 7) / 8;  // query rows per warp in the softmax
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sKV = base;
  float* sQ = reinterpret_cast<float*>(base + kDecStages * 2 * C::TILE);
  float* sP = sQ + FA_DECODE_MAX_Q * D;
  float* sAlpha = sP + FA_DECODE_MAX_Q * 128;
  float* sM = sAlpha + FA_DECODE_MAX_Q;
  float* sL = sM + FA_DECODE_MAX_Q;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sL + FA_DECODE_MAX_Q);
  __shared__ int32_t s_arg[FA_MAX_MASK_NODES];

  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int bm = (p.Bm == 1) ? 0 : b, hm = (p.Hm == 1) ? 0 : h;
  const int ql = p.q_len;
  const int64_t row = ((int64_t)bm * p.Hm + hm) * p.nq;  // the (only) query-tile row
  const int n_full = __ldg(p.full_num + row);
  const int n = n_full + __ldg(p.kv_num + row);
  const int p0 = (int)((int64_t)n * split / splits), p1 = (int)((int64_t)n * (split + 1) / splits);
  auto tile_at = [&](int pos) {
    return pos < n_full ? __ldg(p.full_idx + row * p.nkv + pos) : __ldg(p.kv_idx + row * p.nkv + pos - n_full);
  };

  for (int e = t; e < ql * D; e += kDecThreads) sQ[e] = __bfloat162float(q[(int64_t)bh * ql * D + e]);
  if (t < p.mask.n) s_arg[t] = node_arg(p.mask, t, bm);
  if (t == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // K and V of list position pos into its stage (thread 0, which counts them)
  int issued_end = p0;
  auto issue = [&](int pos) {
    issued_end = pos + 1;
    const int st = (pos - p0) % kDecStages;
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
    const uint32_t bar = smem_u32(&bars[st]);
    mbar_arrive_expect_tx(bar, 2 * C::TILE);
    uint8_t* dk = sKV + (size_t)st * 2 * C::TILE;
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(smem_u32(dk + c * 16384), &tm_k, bar, c * 64, kv_row, kv_z);
      tma_load_3d(smem_u32(dk + C::TILE + c * 16384), &tm_v, bar, c * 64, kv_row, kv_z);
    }
  };
  if (t == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    for (int pos = p0; pos < min(p1, p0 + kDecStages); ++pos) issue(pos);
  }

  const uint64_t mask_ops = pack_ops(p.mask);
  const int32_t* doc_row = p.mask.has_doc ? p.mask.doc + (int64_t)bm * p.mask.doc_len : nullptr;
  float slope_l2 = 0.f, cap = 1.f;
  if constexpr (SCORE == FA_S_ALIBI) slope_l2 = __ldg(p.score_param + h) * kLog2e;
  if constexpr (SCORE == FA_S_SOFTCAP) cap = __ldg(p.score_param);
  float m_run[RW], l_run[RW];
#pragma unroll
  for (int k = 0; k < RW; ++k) m_run[k] = -INFINITY, l_run[k] = 0.f;
  float2 o[QB];  // P V: columns 2c, 2c + 1 of every query row, this thread's key group
#pragma unroll
  for (int i = 0; i < QB; ++i) o[i] = make_float2(0.f, 0.f);
  const int half = t / 128, r = t % 128;          // scores
  const int pc = t % C::PAIRS, grp = t / C::PAIRS;  // P V
  const int pbox = (2 * pc) / 64, pdc = (2 * pc) % 64;
  const int pchunk = pdc / 8, pbyte = (pdc % 8) * 2;

  bool ok = true;
  for (int pos = p0; pos < p1; ++pos) {
    const int st = (pos - p0) % kDecStages, use = (pos - p0) / kDecStages;
    const bool got = mbar_wait(smem_u32(&bars[st]), use & 1, nullptr);
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    const int J = tile_at(pos);
    const bool full = pos < n_full;
    const int rows_valid = min(128, p.kv_len - J * 128);
    const uint8_t* sK = sKV + (size_t)st * 2 * C::TILE;
    const uint8_t* sV = sK + C::TILE;

    // -- scores: this thread's half of q . k for key row r
    float s[QB];
#pragma unroll
    for (int i = 0; i < QB; ++i) s[i] = 0.f;
    if (r < rows_valid) {
#pragma unroll
      for (int cc = 0; cc < C::NCH / 2; ++cc) {
        const int c = half * (C::NCH / 2) + cc;  // 16-byte chunk of the key row, at its swizzled place
        const uint4 kw = *reinterpret_cast<const uint4*>(sK + (c / 8) * 16384 + r * 128 + (((c % 8) ^ (r & 7)) << 4));
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
            float a = s[i];
            a = fmaf(qa.x, kf[0], a);
            a = fmaf(qa.y, kf[1], a);
            a = fmaf(qa.z, kf[2], a);
            a = fmaf(qa.w, kf[3], a);
            a = fmaf(qb.x, kf[4], a);
            a = fmaf(qb.y, kf[5], a);
            a = fmaf(qb.z, kf[6], a);
            a = fmaf(qb.w, kf[7], a);
            s[i] = a;
          }
        }
      }
    }
    if (half == 1) {
#pragma unroll
      for (int i = 0; i < QB; ++i)
        if (i < ql) sP[i * 128 + r] = s[i];
    }
    __syncthreads();
    if (half == 0) {
      // key j: mask (FULL tiles: every in-range pair) and score mod, log2 units
      const int j = J * 128 + r;
      uint32_t w = 0;  // bit i: (i, j) visible
      if (r < rows_valid) {
        if (full) {
          w = 0xffffffffu;
        } else {
          // this key's visible query rows: two intervals, else the program per row
          const int4 seg = __ldg(p.row_segs + ((int64_t)bm * 2 + 1) * p.seg_len + j);
          if (seg.x >= 0) {
            w = seg_word(seg, 0);
          } else {
            int run_lo = 0, run_hi = 0;
            const bool use_run = doc_row != nullptr && doc_run(p.mask, bm, j, run_lo, run_hi);
            const int32_t doc_j = doc_row != nullptr ? __ldg(doc_row + j) : 0;
            auto eq = [&]() {
              if (use_run) return range_bits(run_lo, run_hi, 0);
              uint32_t bits = 0;
              for (int i = 0; i < ql; ++i) bits |= (uint32_t)(__ldg(doc_row + i) == doc_j) << i;
              return bits;
            };
            w = mask_word_t_rolled(p.mask.n, mask_ops, s_arg, j, 0, eq);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        if (i < ql) {
          float a = -INFINITY;
          if ((w >> i) & 1u) {
            const float x = (s[i] + sP[i * 128 + r]) * p.scale;
            if constexpr (SCORE == FA_S_SOFTCAP) {
              a = cap * tanh_fast(x / cap) * kLog2e;
            } else if constexpr (SCORE == FA_S_ALIBI) {
              a = fmaf(x, kLog2e, -slope_l2 * (float)(i - j));
            } else {
              a = x * kLog2e;
            }
          }
          sP[i * 128 + r] = a;
        }
      }
    }
    __syncthreads();

    // -- online softmax: warp w owns query rows w, w + 8
#pragma unroll
    for (int k = 0; k < RW; ++k) {
      const int i = warp + 8 * k;
      if (i < ql) {
        float4 a = *reinterpret_cast<const float4*>(sP + i * 128 + 4 * lane);
        float mx = fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w));
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float m_new = fmaxf(m_run[k], mx);
        const float mu = (m_new == -INFINITY) ? 0.f : m_new;
        a.x = ex2_approx(a.x - mu);
        a.y = ex2_approx(a.y - mu);
        a.z = ex2_approx(a.z - mu);
        a.w = ex2_approx(a.w - mu);
        float sum = (a.x + a.y) + (a.z + a.w);
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        const float alpha = ex2_approx(m_run[k] - mu);
        l_run[k] = fmaf(l_run[k], alpha, sum);
        m_run[k] = m_new;
        *reinterpret_cast<float4*>(sP + i * 128 + 4 * lane) = a;
        if (lane == 0) sAlpha[i] = alpha;
      }
    }
    __syncthreads();

    // -- P V: column pair pc of every query row over this group's valid keys
    {
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        if (i < ql) {
          const float al = sAlpha[i];
          o[i].x *= al;
          o[i].y *= al;
        }
      }
      const uint8_t* vcol = sV + pbox * 16384 + pbyte;
      const int j0 = grp * C::KPG, j1 = min(j0 + C::KPG, rows_valid);
#pragma unroll 4
      for (int jj = j0; jj < j1; ++jj) {
        const float2 vv = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(vcol + jj * 128 + ((pchunk ^ (jj & 7)) << 4)));
#pragma unroll
        for (int i = 0; i < QB; ++i) {
          if (i < ql) {
            const float pij = sP[i * 128 + jj];
            o[i].x = fmaf(pij, vv.x, o[i].x);
            o[i].y = fmaf(pij, vv.y, o[i].y);
          }
        }
      }
    }
    __syncthreads();  // the stage and the scores are free
    if (t == 0 && pos + kDecStages < p1) {
      fence_proxy_async_smem();
      issue(pos + kDecStages);
    }
  }

  if (!ok) {
    if (t == 0) {
      atomicOr(p.status, kStatusTimeout);
      // the last copy issued into each stage lands before the CTA exits (bounded waits)
      for (int pos = max(p0, issued_end - kDecStages); pos < issued_end; ++pos)
        mbar_wait(smem_u32(&bars[(pos - p0) % kDecStages]), ((pos - p0) / kDecStages) & 1, nullptr);
    }
    return;
  }
  // the key groups' sums meet in the (now idle) stage memory: [group][row][D]
  float* red = reinterpret_cast<float*>(sKV);
#pragma unroll
  for (int i = 0; i < QB; ++i)
    if (i < ql) *reinterpret_cast<float2*>(red + ((size_t)grp * FA_DECODE_MAX_Q + i) * D + 2 * pc) = o[i];
#pragma unroll
  for (int k = 0; k < RW; ++k) {
    const int i = warp + 8 * k;
    if (i < ql && lane == 0) {
      sM[i] = m_run[k];
      sL[i] = l_run[k];
    }
  }
  __syncthreads();
  const int64_t r0 = ((int64_t)split * p.B * p.H + bh) * ql;  // this share's first row in the workspace
  for (int e = t; e < ql * D; e += kDecThreads) {
    const int i = e / D, dd = e % D;
    float acc = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < C::NG; ++g2) acc += red[((size_t)g2 * FA_DECODE_MAX_Q + i) * D + dd];
    const float l = sL[i];
    ws_out[(r0 + i) * D + dd] = (l > 0.f) ? acc / l : 0.f;
  }
  if (t < ql) {
    const float l = sL[t];
    ws_lse[r0 + t] = (l > 0.f) ? (sM[t] + log2f(l)) * kLn2 : -INFINITY;
  }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ ws_out,
                                                           const float* __restrict__ ws_lse, int splits,
                                                           int64_t rows, __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
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
  const uint64_t kv_rows = paged ? (uint64_t)a.n_pages * 128 : (uint64_t)a.kv_len;
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
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D, SCORE, QB>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t rows = (int64_t)bh * a.q_len;
  float* ws_out = ws;
  float* ws_lse = ws + (size_t)splits * rows * D;
  decode_partial_kernel<D, SCORE, QB><<<dim3((unsigned)splits, (unsigned)bh), kDecThreads, smem, stream>>>(
      mk, mv, a, static_cast<const __nv_bfloat16*>(t.q), ws_out, ws_lse, splits);
  decode_combine_kernel<D><<<(unsigned)rows, D, 0, stream>>>(ws_out, ws_lse, splits, rows,
                                                             static_cast<__nv_bfloat16*>(t.out), t.lse);
  return cudaGetLastError();
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
  // about one wave of CTAs (one per SM at D = 128, two at D = 64), at most one per key tile
  const int64_t per_sm = (D == 128) ? 1 : 2;
  const int64_t items = (int64_t)B * H;
  const int64_t nkv = (kv_len + 127) / 128;
  int64_t s = (sms * per_sm + items - 1) / items;
  s = std::max<int64_t>(1, std::min<int64_t>(s, std::min<int64_t>(nkv, kDecMaxSplits)));
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
    return launch_decode_q<64, FA_S_NONE>(a, t, ws, splits, stream, enc_failed);
  }
  if (a.score_op == FA_S_SOFTCAP) return launch_decode_q<128, FA_S_SOFTCAP>(a, t, ws, splits, stream, enc_failed);
  if (a.score_op == FA_S_ALIBI) return launch_decode_q<128, FA_S_ALIBI>(a, t, ws, splits, stream, enc_failed);
  return launch_decode_q<128, FA_S_NONE>(a, t, ws, splits, stream, enc_failed);
}

}  // namespace fa
