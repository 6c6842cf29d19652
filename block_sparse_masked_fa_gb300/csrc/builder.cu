// builder.cu -- the block-mask builder (create_block_mask of the speedrun
// notes "FlexAttention", tile-summary paragraph: evaluate mask_mod over the
// index grid and store, per query-tile row, the count and the column indices
// of the tiles that are not fully masked; tutorial "The two hooks": tiles are
// empty, partial or full).
//
// Kernels, all stream-ordered, no host synchronisation:
//  1. tile_summary -- doc-id min / max of every query and key tile, and
//     doc_runs        the range of equal ids around every position (only when
//                     the program has SAME_DOC).
//  2. classify     -- one warp per (query-tile row, chunk of 32 key tiles).
//                     Each lane classifies one tile with a three-valued
//                     interval test per atom (nothing / everything / undecided
//                     visible, combined with Kleene AND / OR); undecided tiles
//                     are settled exactly by the whole warp, counting each
//                     row's visible pairs from its row_segs intervals (or, for
//                     rows they do not describe, evaluating all its pairs).
//                     Writes one class byte per tile.
//     or select    -- for caller-chosen tiles, one warp per query-tile row
//                     writes the class bytes from the caller's lists instead.
//  3. compact      -- one warp per query-tile row and one per key-tile
//                     column: ballot + popcount prefix sums turn the class
//                     bytes into ascending PARTIAL and FULL index lists with
//                     zeroed tails (the columns' lists feed the backward).
//  4. order        -- the order the attention kernels take rows and columns
//                     in: longest first (rows by exact, columns by quantized
//                     tile count), index order within a bucket.
//  and row_segs    -- every query row's visible key columns (and every key
//                     column's visible query rows) as at most two intervals,
//                     which the attention kernels' PARTIAL tiles read instead
//                     of running the program per word.
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// Interval classes of a predicate over a tile: nothing visible, everything
// visible, certainly partial (both kinds of pairs exist), or unknown.
enum : int { K_NONE = 0, K_ALL = 1, K_PART = 2, K_SOME = 3 };

__device__ __forceinline__ int kleene_and(int a, int b) {
  if (a == K_NONE || b == K_NONE) return K_NONE;
  if (a == K_ALL) return b;
  if (b == K_ALL) return a;
  return K_SOME;  // two partial or unknown operands: the conjunction may be empty
}
__device__ __forceinline__ int kleene_or(int a, int b) {
  if (a == K_ALL || b == K_ALL) return K_ALL;
  if (a == K_NONE) return b;
  if (b == K_NONE) return a;
  return K_SOME;
}

// Class of the whole program over rows [i0, i1] x cols [j0, j1] (inclusive).
// q_mn/q_mx (k_mn/k_mx) bound the doc ids of the row (column) range; *_run is
// set when the ids there step by 0 or +1 only, so every id in [mn, mx] occurs.
__device__ int program_interval(const DevMask& m, const int32_t* arg, int64_t i0, int64_t i1, int64_t j0, int64_t j1,
                                int q_mn, int q_mx, int q_run, int k_mn, int k_mx, int k_run) {
  int s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0, s5 = 0, s6 = 0, s7 = 0;
#pragma unroll
  for (int k = 0; k < FA_MAX_MASK_NODES; ++k) {
    if (k < m.n) {
      const int op = m.op[k];
      if (op == FA_M_AND || op == FA_M_OR) {
        s0 = (op == FA_M_AND) ? kleene_and(s1, s0) : kleene_or(s1, s0);
        s1 = s2; s2 = s3; s3 = s4; s4 = s5; s5 = s6; s6 = s7; s7 = K_NONE;
      } else {
        int c;
        const int64_t a = arg[k];
        // the three monotone atoms are exactly partial when neither extreme holds
        if (op == FA_M_CAUSAL) {            // i >= j
          c = (i0 >= j1) ? K_ALL : (i1 < j0 ? K_NONE : K_PART);
        } else if (op == FA_M_WINDOW) {     // i - j < W
          c = (i1 - j0 < a) ? K_ALL : (i0 - j1 >= a ? K_NONE : K_PART);
        } else if (op == FA_M_SINK || op == FA_M_PREFIX) {  // j < n
          c = (j1 < a) ? K_ALL : (j0 >= a ? K_NONE : K_PART);
        } else if (op == FA_M_SAME_DOC) {
          if (q_mx < k_mn || k_mx < q_mn)
            c = K_NONE;
          else if (q_mn == q_mx && k_mn == k_mx && q_mn == k_mn)
            c = K_ALL;
          else  // overlapping ranges in which every id occurs share an id and hold a distinct one
            c = (q_run && k_run) ? K_PART : K_SOME;
        } else {
          c = K_ALL;
        }
        s7 = s6; s6 = s5; s5 = s4; s4 = s3; s3 = s2; s2 = s1; s1 = s0; s0 = c;
      }
    }
  }
  return s0;
}

__global__ void tile_summary_kernel(const __grid_constant__ BuildArgs a) {
  pdl_wait_then_release();
  const int warps = blockDim.x / 32;
  const int64_t w = (int64_t)blockIdx.x * warps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int tmax = max(a.nq, a.nkv);
  if (w < a.Bm && lane == 0) {  // preset "sorted"; doc_runs clears it at the first decrease
    const int64_t L = max(a.q_len, a.kv_len);
    a.doc_runs[(int64_t)a.Bm * L * 2 + w] = 1;
  }
  if (w >= (int64_t)a.Bm * 2 * tmax) return;
  const int t = (int)(w % tmax);
  const int which = (int)((w / tmax) % 2);  // 0: query tiles, 1: key tiles
  const int bm = (int)(w / (2 * tmax));
  const int64_t len = which ? a.kv_len : a.q_len;
  const int ntiles = which ? a.nkv : a.nq;
  if (t >= ntiles) return;
  const int32_t* doc = a.mask.doc + (int64_t)bm * a.mask.doc_len;
  const int64_t off = which ? 0 : a.mask.q_off;  // query rows sit at positions row + q_off
  const int64_t i0 = (int64_t)t * a.block + off;
  const int64_t i1 = min((int64_t)t * a.block + a.block, len) + off;
  int mn = INT_MAX, mx = INT_MIN;
  bool run = true;
  for (int64_t i = i0 + lane; i < i1; i += 32) {
    const int d = __ldg(doc + i);
    mn = min(mn, d);
    mx = max(mx, d);
    if (i + 1 < i1) {
      const int step = __ldg(doc + i + 1) - d;
      run = run && (step == 0 || step == 1);
    }
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  run = __all_sync(0xffffffffu, run);
  if (lane == 0) {
    int32_t* s = a.summary + (((int64_t)bm * 2 + which) * tmax + t) * 4;
    s[0] = mn;
    s[1] = mx;
    s[2] = run ? 1 : 0;
    s[3] = 0;
  }
}

// Runs of equal document ids, for PARTIAL tiles: for every position x < L =
// max(q_len, kv_len) of batch row bm, [lo, hi) is the range of positions whose
// id equals doc[x], valid when the row's ids never decrease (sorted[bm] = 1,
// preset by tile_summary and cleared here at the first decrease): then
// doc[y] == doc[x] exactly for y in [lo, hi), and lo / hi are the lower /
// upper bound of doc[x] in the row, found by binary search.
__global__ void __launch_bounds__(256) doc_runs_kernel(const __grid_constant__ BuildArgs a) {
  pdl_wait_then_release();
  const int L = (int)max(a.q_len, a.kv_len);
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)a.Bm * L) return;
  const int bm = (int)(gid / L), x = (int)(gid % L);
  const int32_t* doc = a.mask.doc + (int64_t)bm * a.mask.doc_len;
  const int d = __ldg(doc + x);
  if (x > 0 && __ldg(doc + x - 1) > d) atomicAnd(a.doc_runs + (int64_t)a.Bm * L * 2 + bm, 0);
  int lo = 0, hi = x;  // first position with id >= d lies in [0, x]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(doc + mid) < d) lo = mid + 1; else hi = mid;
  }
  int lo2 = x + 1, hi2 = L;  // first position with id > d lies in [x + 1, L]
  while (lo2 < hi2) {
    const int mid = (lo2 + hi2) >> 1;
    if (__ldg(doc + mid) <= d) lo2 = mid + 1; else hi2 = mid;
  }
  reinterpret_cast<int2*>(a.doc_runs)[gid] = make_int2(lo, lo2);
}

// ---- The visible set of one row as intervals
//
// Fix one index x and let the other, y, vary: x = query row i and y = key
// column j, or (transposed) x = key column j and y = query row i.  Every atom
// is then visible on an interval of y -- SAME_DOC too when the ids never
// decrease, through the run [lo, hi) holding x -- so the program's value can
// only change at the atoms' interval ends.  row_segments evaluates the program
// once between consecutive ends and keeps the visible pieces, merged, when
// there are at most two; the attention kernels then build a 32-bit word from
// two range tests (seg_word) instead of running the program.  Rows that need
// more pieces, or ids that decrease somewhere, keep the per-word evaluation.
struct RowSegs {
  int n;  // visible intervals (0..2), or -1 when the row is not represented
  int lo0, hi0, lo1, hi1;
};

// The program's value at one pair (x, y).
__device__ __forceinline__ bool mask_bit(int nn, uint64_t ops, const int32_t* arg, bool transposed, int64_t x,
                                         int64_t y, int run_lo, int run_hi, int64_t off) {
  const int64_t i = (transposed ? y : x) + off, j = transposed ? x : y;  // i: the query's position
  uint32_t st = 0;  // bit stack, top at bit 0
#pragma unroll 1
  for (int k = 0; k < nn; ++k, ops >>= 4) {
    const int op = (int)(ops & 15u);
    if (op == FA_M_AND || op == FA_M_OR) {
      const uint32_t a = st & 1u, b = (st >> 1) & 1u;
      st = ((st >> 2) << 1) | (op == FA_M_AND ? (a & b) : (a | b));
    } else {
      bool v = true;
      if (op == FA_M_CAUSAL) v = i >= j;
      else if (op == FA_M_WINDOW) v = i - j < (int64_t)arg[k];
      else if (op == FA_M_SINK || op == FA_M_PREFIX) v = j < (int64_t)arg[k];
      else if (op == FA_M_SAME_DOC) v = y >= run_lo && y < run_hi;
      st = (st << 1) | (v ? 1u : 0u);
    }
  }
  return (st & 1u) != 0;
}

//  len            extent of y (kv_len, or q_len when transposed)
//  have_run       the ids never decrease and [run_lo, run_hi) is the run of x's
//                 position (x + off for a query row)
//  off            position of query row 0: a query row x is position x + off,
//                 and the intervals of a key column are over query rows
// Everything stays in registers (constant indices only): at most kRowBreaks
// interval ends besides 0, else the row is left to the per-word evaluation.
constexpr int kRowBreaks = 8;

__device__ __forceinline__ void cswap(int& a, int& b) {
  const int lo = min(a, b), hi = max(a, b);
  a = lo;
  b = hi;
}

__device__ RowSegs row_segments(int nn, uint64_t ops, const int32_t* arg, bool transposed,
                                                    int64_t x, bool have_run, int run_lo, int run_hi, int64_t len,
                                                    int64_t off) {
  RowSegs seg{-1, 0, 0, 0, 0};
  if (transposed) {  // the run, in query rows
    run_lo -= (int)off;
    run_hi -= (int)off;
  }
  int64_t bp[kRowBreaks];
#pragma unroll
  for (int t = 0; t < kRowBreaks; ++t) bp[t] = len;
  bp[0] = 0;
  int nb = 1;
  uint64_t o = ops;
#pragma unroll 1
  for (int k = 0; k < nn; ++k, o >>= 4) {
    const int op = (int)(o & 15u);
    int64_t v0 = 0, v1 = 0;
    int add = 0;
    if (op == FA_M_SAME_DOC) {
      if (!have_run) return seg;
      v0 = run_lo;
      v1 = run_hi;
      add = 2;
    } else if (op == FA_M_CAUSAL) {
      v0 = transposed ? x - off : x + off + 1;
      add = 1;
    } else if (op == FA_M_WINDOW) {
      v0 = transposed ? x + (int64_t)arg[k] - off : x + off - (int64_t)arg[k] + 1;
      add = 1;
    } else if (!transposed && (op == FA_M_SINK || op == FA_M_PREFIX)) {
      v0 = arg[k];
      add = 1;
    }
    if (nb + add > kRowBreaks) return seg;
#pragma unroll
    for (int t = 0; t < kRowBreaks; ++t) {
      if (add >= 1 && t == nb) bp[t] = v0;
      if (add == 2 && t == nb + 1) bp[t] = v1;
    }
    nb += add;
  }
  // clamped to [0, len] (len < 2^31), so the sort and the segments run in 32 bits
  int b32[kRowBreaks];
#pragma unroll
  for (int t = 0; t < kRowBreaks; ++t) b32[t] = (int)(bp[t] < 0 ? 0 : (bp[t] > len ? len : bp[t]));
  // sorting network for 8 values (19 compare-exchanges)
  cswap(b32[0], b32[2]); cswap(b32[1], b32[3]); cswap(b32[4], b32[6]); cswap(b32[5], b32[7]);
  cswap(b32[0], b32[4]); cswap(b32[1], b32[5]); cswap(b32[2], b32[6]); cswap(b32[3], b32[7]);
  cswap(b32[0], b32[1]); cswap(b32[2], b32[3]); cswap(b32[4], b32[5]); cswap(b32[6], b32[7]);
  cswap(b32[2], b32[4]); cswap(b32[3], b32[5]);
  cswap(b32[1], b32[4]); cswap(b32[3], b32[6]);
  cswap(b32[1], b32[2]); cswap(b32[3], b32[4]); cswap(b32[5], b32[6]);
  int n = 0;
  int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
#pragma unroll
  for (int t = 0; t + 1 < kRowBreaks; ++t) {
    const int y0 = b32[t], y1 = b32[t + 1];
    if (y0 < y1 && mask_bit(nn, ops, arg, transposed, x, y0, run_lo, run_hi, off)) {
      if (n == 1 && hi0 == (int)y0) {
        hi0 = (int)y1;
      } else if (n == 2 && hi1 == (int)y0) {
        hi1 = (int)y1;
      } else if (n == 0) {
        lo0 = (int)y0;
        hi0 = (int)y1;
        n = 1;
      } else if (n == 1) {
        lo1 = (int)y0;
        hi1 = (int)y1;
        n = 2;
      } else {
        return seg;  // a third interval
      }
    }
  }
  seg.n = n;
  seg.lo0 = lo0;
  seg.hi0 = hi0;
  seg.lo1 = lo1;
  seg.hi1 = hi1;
  return seg;
}

// Visible intervals of every query row over the key columns ([bm][0][x]) and
// of every key column over the query rows ([bm][1][x]), for x < L =
// max(q_len, kv_len); lo0 = -1 where two intervals do not describe the row.
__global__ void __launch_bounds__(256) row_segs_kernel(const __grid_constant__ BuildArgs a) {
  pdl_wait_then_release();
  const int64_t L = max(a.q_len, a.kv_len);
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)a.Bm * 2 * L) return;
  const int64_t x = gid % L;
  const int which = (int)((gid / L) % 2);
  const int bm = (int)(gid / (2 * L));
  const int64_t off = a.mask.q_off;
  if (which == 0 && x + off >= L) {  // past the last query row's position: no row
    reinterpret_cast<int4*>(a.row_segs)[gid] = make_int4(-1, -1, 0, 0);
    return;
  }
  int32_t arg[FA_MAX_MASK_NODES];
  for (int k = 0; k < a.mask.n; ++k) arg[k] = node_arg(a.mask, k, bm);
  int lo = 0, hi = 0;
  const bool have_run = a.mask.has_doc && doc_run(a.mask, bm, which == 0 ? x + off : x, lo, hi);
  const RowSegs s = row_segments(a.mask.n, pack_ops(a.mask), arg, which == 1, x, have_run, lo, hi,
                                 which ? a.q_len : a.kv_len, off);
  reinterpret_cast<int4*>(a.row_segs)[gid] = (s.n < 0) ? make_int4(-1, -1, 0, 0) : make_int4(s.lo0, s.hi0, s.lo1, s.hi1);
}

constexpr int kBuildWarps = 8;

// One warp per query-tile row.  The row's key tiles go in chunks of 32, one
// chunk per lane first: the interval test of the program over the chunk's whole
// key range (its document ids bounded by its tiles' summaries) proves most
// chunks of a windowed or document mask EMPTY, and those are written as zeros.
// The warp then classifies the other chunks one at a time, a tile per lane;
// undecided tiles are settled exactly by the whole warp.  Writes the class
// bytes only; compaction into lists is a separate pass.
__global__ void __launch_bounds__(kBuildWarps * 32) classify_kernel(const __grid_constant__ BuildArgs a) {
  pdl_wait_then_release();
  __shared__ int32_t s_arg[kBuildWarps][FA_MAX_MASK_NODES];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nchunk = (a.nkv + 31) / 32;
  const int64_t row = (int64_t)blockIdx.x * kBuildWarps + warp;  // (bm, hm, I)
  if (row >= (int64_t)a.Bm * a.Hm * a.nq) return;
  const int I = (int)(row % a.nq);
  const int bm = (int)(row / ((int64_t)a.Hm * a.nq));
  if (lane < a.mask.n) s_arg[warp][lane] = node_arg(a.mask, lane, bm);
  __syncwarp();
  const int32_t* arg = s_arg[warp];
  const uint64_t ops = pack_ops(a.mask);
  const int tmax = max(a.nq, a.nkv);
  const int32_t* doc = a.mask.has_doc ? a.mask.doc + (int64_t)bm * a.mask.doc_len : nullptr;
  const bool doc_vec = a.mask.doc_vec_ok != 0;

  const int64_t i0 = (int64_t)I * a.block;
  const int64_t i1 = min(i0 + a.block, a.q_len) - 1;
  int q_mn = 0, q_mx = 0, q_run = 0;
  if (doc) {
    const int32_t* sm = a.summary + (((int64_t)bm * 2 + 0) * tmax + I) * 4;
    q_mn = sm[0];
    q_mx = sm[1];
    q_run = sm[2];
  }
  uint8_t* out = a.tile_class + row * a.nkv;
  // chunk c: tiles [32 c, min(32 c + 32, nkv)); EMPTY as a whole when the test over its range says so
  for (int cb = 0; cb < nchunk; cb += 32) {
    const int c = cb + lane;
    bool live = false;
    if (c < nchunk) {
      const int t0 = 32 * c, t1 = min(t0 + 32, a.nkv);
      const int64_t j0 = (int64_t)t0 * a.block;
      const int64_t j1 = min((int64_t)t1 * a.block, (int64_t)a.kv_len) - 1;
      int k_mn = 0, k_mx = 0;
      if (doc) {
        k_mn = INT_MAX;
        k_mx = INT_MIN;
        const int32_t* ks = a.summary + (((int64_t)bm * 2 + 1) * tmax + t0) * 4;
#pragma unroll
        for (int t = 0; t < 32; ++t) {  // all 32 loads in flight at once
          if (t0 + t < t1) {
            const int2 sm = __ldg(reinterpret_cast<const int2*>(ks + 4 * t));
            k_mn = min(k_mn, sm.x);
            k_mx = max(k_mx, sm.y);
          }
        }
      }
      // (no "every id occurs" claim for the chunk: SAME_DOC then decides only disjoint ranges)
      live = program_interval(a.mask, arg, i0 + a.mask.q_off, i1 + a.mask.q_off, j0, j1, q_mn, q_mx, q_run, k_mn,
                              k_mx, 0) != K_NONE;
      if (!live) {
        if (t1 - t0 == 32 && (reinterpret_cast<uintptr_t>(out + t0) & 15) == 0) {
          reinterpret_cast<uint4*>(out + t0)[0] = make_uint4(0u, 0u, 0u, 0u);
          reinterpret_cast<uint4*>(out + t0)[1] = make_uint4(0u, 0u, 0u, 0u);
        } else {
          for (int t = t0; t < t1; ++t) out[t] = 0;
        }
      }
    }
    uint32_t live_mask = __ballot_sync(0xffffffffu, live);
    while (live_mask) {
      const int c0 = 32 * (cb + __ffs(live_mask) - 1);
      live_mask &= live_mask - 1;
      const int J = c0 + lane;
      const bool valid = J < a.nkv;
      int cls = 0, k3 = K_NONE;
      if (valid) {
        const int64_t j0 = (int64_t)J * a.block;
        const int64_t j1 = min(j0 + a.block, a.kv_len) - 1;
        int k_mn = 0, k_mx = 0, k_run = 0;
        if (doc) {
          const int32_t* sm = a.summary + (((int64_t)bm * 2 + 1) * tmax + J) * 4;
          k_mn = sm[0];
          k_mx = sm[1];
          k_run = sm[2];
        }
        k3 = program_interval(a.mask, arg, i0 + a.mask.q_off, i1 + a.mask.q_off, j0, j1, q_mn, q_mx, q_run, k_mn, k_mx,
                              k_run);
        cls = (k3 == K_ALL) ? 2 : (k3 == K_PART ? 1 : 0);
      }
      uint32_t undecided = __ballot_sync(0xffffffffu, valid && k3 == K_SOME);
      while (undecided) {
        const int t = __ffs(undecided) - 1;
        undecided &= undecided - 1;
        const int64_t j0 = (int64_t)(c0 + t) * a.block;
        const int64_t j1 = min(j0 + a.block, a.kv_len) - 1;
        const int64_t rows = i1 - i0 + 1, cols = j1 - j0 + 1;
        int cnt = 0;
        const int64_t L = max(a.q_len, a.kv_len);
        for (int64_t r = lane; r < rows; r += 32) {
          const int64_t i = i0 + r;
          // the row's visible columns as two intervals (row_segs_kernel ran first):
          // its count inside the tile is two overlaps
          const int4 sg = reinterpret_cast<const int4*>(a.row_segs)[((int64_t)bm * 2) * L + i];
          if (sg.x >= 0) {
            cnt += (int)(max((int64_t)0, min((int64_t)sg.y, j1 + 1) - max((int64_t)sg.x, j0)) +
                         max((int64_t)0, min((int64_t)sg.w, j1 + 1) - max((int64_t)sg.z, j0)));
            continue;
          }
          const int64_t ip = i + a.mask.q_off;  // the query's position
          const int32_t doc_i = doc ? __ldg(doc + ip) : 0;
          int run_lo = 0, run_hi = 0;
          const bool use_run = doc != nullptr && doc_run(a.mask, bm, ip, run_lo, run_hi);
          for (int64_t jc = j0; jc <= j1; jc += 32) {
            auto eq = [&]() {
              if (use_run) return range_bits(run_lo, run_hi, (int)jc);
              uint32_t w = 0;
              if (doc_vec && jc + 32 <= j1 + 1) {
                const int4* dv = reinterpret_cast<const int4*>(doc + jc);  // same addresses in every lane
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  const int4 d = __ldg(dv + q4);
                  w |= (uint32_t)(d.x == doc_i) << (4 * q4) | (uint32_t)(d.y == doc_i) << (4 * q4 + 1) |
                       (uint32_t)(d.z == doc_i) << (4 * q4 + 2) | (uint32_t)(d.w == doc_i) << (4 * q4 + 3);
                }
              } else {
                const int64_t jn = min(jc + 32, j1 + 1);
                for (int64_t j = jc; j < jn; ++j) w |= (uint32_t)(__ldg(doc + j) == doc_i) << (uint32_t)(j - jc);
              }
              return w;
            };
            cnt += __popc(mask_word_rolled(a.mask.n, ops, arg, ip, jc, eq) & low_bits(j1 + 1 - jc));
          }
        }
        const int total = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
        const int c = (total == 0) ? 0 : ((int64_t)total == rows * cols ? 2 : 1);
        if (lane == t) cls = c;
      }
      if (valid) out[J] = (uint8_t)cls;
    }
  }
}

// Caller-chosen tiles (tutorial "FlexAttention in PyTorch": block-selection
// sparse patterns; "Decoding and paged KV caches": BlockMask.from_kv_blocks).
// One warp per query-tile row clears the row's class bytes, marks the listed
// PARTIAL tiles 1 and then the listed FULL tiles 2 (a tile in both lists ends
// FULL), and checks the lists: a count outside [0, min(nkv, stride)] (clamped),
// an index outside [0, nkv) (dropped) or a tile listed twice sets the status
// word's check bit.  Compaction then rebuilds the lists ascending, with the
// per-column lists the backward needs.
__global__ void __launch_bounds__(kBuildWarps * 32) select_kernel(const __grid_constant__ BuildArgs a) {
  pdl_wait_then_release();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t row = (int64_t)blockIdx.x * kBuildWarps + warp;  // (bm, hm, I)
  if (row >= (int64_t)a.Bm * a.Hm * a.nq) return;
  uint8_t* cls = a.tile_class + row * a.nkv;
  for (int J = lane; J < a.nkv; J += 32) cls[J] = 0;
  __syncwarp();
  const int cap = min(a.nkv, a.sel_stride);
  bool bad = false;
  int listed = 0;
  for (int code = 1; code <= 2; ++code) {
    const int32_t* num = (code == 1) ? a.sel_num : a.sel_full_num;
    if (num == nullptr) continue;
    const int32_t* idx = ((code == 1) ? a.sel_idx : a.sel_full_idx) + row * (int64_t)a.sel_stride;
    int n = __ldg(num + row);
    if (n < 0 || n > cap) {
      bad = true;
      n = max(0, min(n, cap));
    }
    for (int t = lane; t < n; t += 32) {
      const int J = __ldg(idx + t);
      if (J < 0 || J >= a.nkv) {
        bad = true;
        continue;
      }
      cls[J] = (uint8_t)code;
      ++listed;
    }
    __syncwarp();  // the FULL marks land after every PARTIAL one
  }
  // a tile listed twice leaves fewer marked tiles than valid entries
  int marked = 0;
  for (int J = lane; J < a.nkv; J += 32) marked += cls[J] != 0;
  const unsigned tot_marked = __reduce_add_sync(0xffffffffu, (unsigned)marked);
  const unsigned tot_listed = __reduce_add_sync(0xffffffffu, (unsigned)listed);
  if (__any_sync(0xffffffffu, bad) || tot_marked != tot_listed) {
    if (lane == 0) atomicOr(a.status, kStatusCheck);
  }
}

// Compaction of one class grid [planes][n_r][n_c] into lists, ascending, with
// zero tails.  Warps [0, rows) build the per-row lists, the next [0, cols) warps
// the per-column lists (rows or columns without list pointers are skipped).  A
// row's class bytes are read 16 at a time by every lane when the grid's rows
// are 16-byte aligned (n_c a multiple of 16), and its entries placed by a
// prefix count over the lanes; otherwise, and for the columns, one byte a lane
// with ballots.  The tails are written in 16-byte stores where the list allows.
constexpr int kColGroup = 16;

__device__ __forceinline__ bool compact_vec(const ListJob& j) {
  return j.n_c % kColGroup == 0 && (reinterpret_cast<uintptr_t>(j.cls) & 15) == 0;
}

// byte k (0..15) of a 16-byte load
__device__ __forceinline__ int byte_of(const uint4& v, int k) {
  const uint32_t w = (k < 4) ? v.x : (k < 8) ? v.y : (k < 12) ? v.z : v.w;
  return (int)((w >> (8 * (k & 3))) & 0xffu);
}

// list[from, n) = 0 by the 32 lanes, in 16-byte stores where the list allows
__device__ __forceinline__ void zero_tail(int32_t* list, int from, int n, int lane) {
  const int v0 = (from + 3) / 4, v1 = n / 4;  // the int4 groups [v0, v1) lie inside [from, n)
  if ((reinterpret_cast<uintptr_t>(list) & 15) != 0 || v0 >= v1) {
    for (int x = from + lane; x < n; x += 32) list[x] = 0;
    return;
  }
  if (lane < 4 * v0 - from) list[from + lane] = 0;
  for (int q = v0 + lane; q < v1; q += 32) reinterpret_cast<int4*>(list)[q] = make_int4(0, 0, 0, 0);
  if (lane < n - 4 * v1) list[4 * v1 + lane] = 0;
}

__global__ void __launch_bounds__(kBuildWarps * 32) compact_kernel(const __grid_constant__ ListJob j) {
  pdl_wait_then_release();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t wid = (int64_t)blockIdx.x * kBuildWarps + warp;
  const int64_t rows = j.row_num ? (int64_t)j.planes * j.n_r : 0, cols = j.col_num ? (int64_t)j.planes * j.n_c : 0;
  if (wid >= rows + cols) return;
  const uint32_t lt = (1u << lane) - 1u;
  if (wid < rows && compact_vec(j)) {
    // ---- row id: 512 tiles a round, 16 per lane
    const int64_t id = wid;
    const int n = j.n_c;
    const uint8_t* rb = j.cls + id * n;
    int32_t* part_idx = j.row_idx + id * n;
    int32_t* full_idx = j.row_full_idx + id * n;
    int n_part = 0, n_full = 0;
    for (int s0 = 0; s0 < n; s0 += 32 * kColGroup) {
      const int x0 = s0 + kColGroup * lane;
      const uint4 v = (x0 < n) ? __ldg(reinterpret_cast<const uint4*>(rb + x0)) : make_uint4(0u, 0u, 0u, 0u);
      int np = 0, nf = 0;
#pragma unroll
      for (int k = 0; k < kColGroup; ++k) {
        const int b = byte_of(v, k);
        np += (b == 1);
        nf += (b == 2);
      }
      int ip = np, iF = nf;  // inclusive prefix counts over the lanes
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int yp = __shfl_up_sync(0xffffffffu, ip, d), yf = __shfl_up_sync(0xffffffffu, iF, d);
        if (lane >= d) {
          ip += yp;
          iF += yf;
        }
      }
      int op = n_part + ip - np, of = n_full + iF - nf;
#pragma unroll
      for (int k = 0; k < kColGroup; ++k) {
        const int b = byte_of(v, k);
        if (b == 1) part_idx[op++] = x0 + k;
        if (b == 2) full_idx[of++] = x0 + k;
      }
      n_part += __shfl_sync(0xffffffffu, ip, 31);
      n_full += __shfl_sync(0xffffffffu, iF, 31);
    }
    zero_tail(part_idx, n_part, n, lane);
    zero_tail(full_idx, n_full, n, lane);
    if (lane == 0) {
      j.row_num[id] = n_part;
      j.row_full_num[id] = n_full;
    }
    return;
  }
  // ---- one byte at a time: a row (grid rows not 16-byte aligned) or a column per warp
  const bool by_row = wid < rows;
  const int64_t id = by_row ? wid : wid - rows;
  const int n = by_row ? j.n_c : j.n_r;                   // list length
  const int64_t stride = by_row ? 1 : j.n_c;              // class-byte stride along the list
  const uint8_t* cls_base = by_row ? j.cls + id * j.n_c
                                   : j.cls + (id / j.n_c) * j.n_r * j.n_c + (id % j.n_c);
  int32_t* part_idx = (by_row ? j.row_idx : j.col_idx) + id * n;
  int32_t* full_idx = (by_row ? j.row_full_idx : j.col_full_idx) + id * n;
  int n_part = 0, n_full = 0;
  // class bytes of eight 32-tile chunks are loaded before any list entry is
  // stored: the stores (int32) could alias the bytes for the compiler, which
  // would otherwise keep each load behind the stores of the chunk before it
  constexpr int kBatch = 8;
  for (int c0 = 0; c0 < n; c0 += 32 * kBatch) {
    int cls[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int x = c0 + 32 * u + lane;
      cls[u] = (x < n) ? __ldg(cls_base + (int64_t)x * stride) : 0;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int x = c0 + 32 * u + lane;
      const uint32_t pb = __ballot_sync(0xffffffffu, cls[u] == 1);
      const uint32_t fb = __ballot_sync(0xffffffffu, cls[u] == 2);
      if (cls[u] == 1) part_idx[n_part + __popc(pb & lt)] = x;
      if (cls[u] == 2) full_idx[n_full + __popc(fb & lt)] = x;
      n_part += __popc(pb);
      n_full += __popc(fb);
    }
  }
  zero_tail(part_idx, n_part, n, lane);
  zero_tail(full_idx, n_full, n, lane);
  if (lane == 0) {
    (by_row ? j.row_num : j.col_num)[id] = n_part;
    (by_row ? j.row_full_num : j.col_full_num)[id] = n_full;
  }
}

// Coarse classes for the attention kernels' tiles when the block mask's tiles
// are smaller: coarse tile (I, J) of [planes][n_r][n_c] covers fine rows
// [fr I, fr I + fr) and columns [fc J, fc J + fc) (cut at the fine grid's
// edge); it is EMPTY when every fine tile there is, FULL when every one is, and
// PARTIAL otherwise -- exact, since a union of tiles has no visible pair iff
// none of them has one, and only visible pairs iff all of them have only those.
__global__ void __launch_bounds__(256) coarsen_kernel(const uint8_t* __restrict__ fine, int fine_nq, int fine_nkv,
                                                      uint8_t* __restrict__ coarse, int n_r, int n_c, int fr, int fc,
                                                      int64_t n) {
  pdl_wait_then_release();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= n) return;
  const int J = (int)(gid % n_c);
  const int I = (int)((gid / n_c) % n_r);
  const int64_t plane = gid / ((int64_t)n_r * n_c);
  const uint8_t* f = fine + plane * fine_nq * fine_nkv;
  const int i1 = min((I + 1) * fr, fine_nq), j1 = min((J + 1) * fc, fine_nkv);
  bool any = false, all = true;
  for (int i = I * fr; i < i1; ++i)
    for (int jj = J * fc; jj < j1; ++jj) {
      const int c = __ldg(f + (int64_t)i * fine_nkv + jj);
      any = any || c != 0;
      all = all && c == 2;
    }
  coarse[gid] = (uint8_t)(!any ? 0 : (all ? 2 : 1));
}

// Work order: block 0 orders the rows (forward), block 1 the columns
// (backward), longest first so that long lists do not end the grid.  Rows /
// columns go in chunks of 32 neighbours (one warp), the chunks ordered by
// their longest count and, inside a chunk, the entries longest first (index
// order among equals), so that neighbouring tiles, which share most of their
// key (query) tiles under a window, run in the same few waves of CTAs and
// share those tiles in L2; sorting every entry by its own count scatters them
// when counts are noisy (document masks).  Counts are exact for the forward
// and quantized to q = ceil(cmax / 16) for the backward (cmax: the largest
// count), with everything in one bucket when cmax <= 16.  A stable counting
// sort over the chunk keys keeps chunks in index order inside each bucket.
// The histogram has kOrderBuckets entries; coarser buckets are used if the
// counts would need more.
constexpr int kOrderBuckets = 4096;

__global__ void __launch_bounds__(1024) order_kernel(const __grid_constant__ ListJob j) {
  pdl_wait_then_release();
  extern __shared__ int32_t hist[];  // kOrderBuckets entries
  __shared__ int s_cmax;
  const bool rows = blockIdx.x == 0;
  if ((rows ? j.row_num : j.col_num) == nullptr) return;
  const int32_t* num = rows ? j.row_num : j.col_num;
  const int32_t* full_num = rows ? j.row_full_num : j.col_full_num;
  int32_t* order = rows ? j.row_order : j.col_order;
  const int n = rows ? j.planes * j.n_r : j.planes * j.n_c;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) s_cmax = 0;
  __syncthreads();
  int cm = 0;
  for (int r = threadIdx.x; r < n; r += blockDim.x) cm = max(cm, num[r] + full_num[r]);
  cm = __reduce_max_sync(0xffffffffu, cm);
  if (lane == 0) atomicMax(&s_cmax, cm);
  __syncthreads();
  const int cmax = s_cmax;
  int qz = rows ? 1 : ((cmax <= 16) ? cmax + 1 : (cmax + 15) / 16);  // bucket width
  qz = max(qz, (cmax + kOrderBuckets) / kOrderBuckets);              // at most kOrderBuckets buckets
  const int top = min(cmax / qz, kOrderBuckets - 1);                 // largest bucket
  const int nb = top + 1;
  for (int k = threadIdx.x; k < nb; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  // the bucket of entry r: its chunk's (this warp's 32 entries') longest count
  auto chunk_bucket = [&](int r) {
    const int key = __reduce_max_sync(0xffffffffu, r < n ? num[r] + full_num[r] : 0);
    return top - min(key / qz, top);
  };
  for (int round = 0; round < n; round += blockDim.x) {
    const int r = round + threadIdx.x;
    const int bucket = chunk_bucket(r);
    if (r < n) atomicAdd(&hist[bucket], 1);
  }
  __syncthreads();
  // exclusive scan, one warp
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < nb; base += 32) {
      const int k = base + lane;
      const int h = (k < nb) ? hist[k] : 0;
      int incl = h;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      if (k < nb) hist[k] = carry + incl - h;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  // scatter in index order: warps take their turn inside each round of blockDim items
  for (int round = 0; round < n; round += blockDim.x) {
    const int r = round + threadIdx.x;
    const bool valid = r < n;
    const int cb = chunk_bucket(r);
    const int bucket = valid ? cb : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, bucket);
    // rank inside the chunk: longer first, index order among equals
    const int mine = valid ? (num[r] + full_num[r]) / qz : -1;
    int rank = 0;
    for (int l = 0; l < 32; ++l) {
      const int other = __shfl_sync(0xffffffffu, mine, l);
      rank += (((peers >> l) & 1u) && (other > mine || (other == mine && l < lane))) ? 1 : 0;
    }
    const int leader = __ffs(peers) - 1;
    int off = 0;
    for (int w = 0; w < (int)(blockDim.x / 32); ++w) {
      if (warp == w && valid && lane == leader) {
        off = hist[bucket];
        hist[bucket] = off + __popc(peers);
      }
      __syncthreads();
    }
    off = __shfl_sync(0xffffffffu, off, leader);
    if (valid) order[off + rank] = r;
  }
}


// Compaction and work order of one class grid (rows / columns: how many lists).
cudaError_t launch_lists(const ListJob& j, int64_t rows, int64_t cols, cudaStream_t stream) {
  cudaError_t e = launch_k(compact_kernel, dim3((unsigned)((rows + cols + kBuildWarps - 1) / kBuildWarps)),
                           dim3(kBuildWarps * 32), 0, stream, j);
  if (e != cudaSuccess) return e;
  return launch_k(order_kernel, dim3(2), dim3(1024), kOrderBuckets * sizeof(int32_t), stream, j);
}

}  // namespace

cudaError_t launch_build(const BuildArgs& a, cudaStream_t stream) {
  const int tmax = a.nq > a.nkv ? a.nq : a.nkv;
  cudaError_t e = cudaSuccess;
  if (a.mask.has_doc) {
    const int64_t warps = (int64_t)a.Bm * 2 * tmax;
    e = launch_k(tile_summary_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
    const int64_t L = a.q_len > a.kv_len ? a.q_len : a.kv_len;
    e = launch_k(doc_runs_kernel, dim3((unsigned)((a.Bm * L + 255) / 256)), dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  {
    const int64_t L = a.q_len > a.kv_len ? a.q_len : a.kv_len;
    e = launch_k(row_segs_kernel, dim3((unsigned)((a.Bm * 2 * L + 255) / 256)), dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  const int64_t rows = (int64_t)a.Bm * a.Hm * a.nq;
  const int64_t cols = (int64_t)a.Bm * a.Hm * a.nkv;
  if (a.sel_num != nullptr)
    e = launch_k(select_kernel, dim3((unsigned)((rows + kBuildWarps - 1) / kBuildWarps)), dim3(kBuildWarps * 32), 0,
                 stream, a);
  else
    e = launch_k(classify_kernel, dim3((unsigned)((rows + kBuildWarps - 1) / kBuildWarps)),
                 dim3(kBuildWarps * 32), 0, stream, a);
  if (e != cudaSuccess) return e;
  ListJob fine;
  fine.cls = a.tile_class;
  fine.planes = a.Bm * a.Hm;
  fine.n_r = a.nq;
  fine.n_c = a.nkv;
  fine.row_num = a.kv_num;
  fine.row_idx = a.kv_idx;
  fine.row_full_num = a.full_num;
  fine.row_full_idx = a.full_idx;
  fine.col_num = a.q_num;
  fine.col_idx = a.q_idx;
  fine.col_full_num = a.full_q_num;
  fine.col_full_idx = a.full_q_idx;
  fine.row_order = a.row_order;
  fine.col_order = a.col_order;
  e = launch_lists(fine, rows, cols, stream);
  if (e != cudaSuccess || a.fwd.cls == nullptr) return e;
  // tiles smaller than the attention kernels': their classes, coarsened, and lists
  for (const ListJob* jb : {&a.fwd, &a.bwd}) {
    const int64_t n = (int64_t)jb->planes * jb->n_r * jb->n_c;
    e = launch_k(coarsen_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, (const uint8_t*)a.tile_class,
                 a.nq, a.nkv, jb->cls, jb->n_r, jb->n_c, (128 / a.block), (jb == &a.fwd ? a.fwd_kv_block : 128) / a.block,
                 n);
    if (e != cudaSuccess) return e;
    e = launch_lists(*jb, jb->row_num ? (int64_t)jb->planes * jb->n_r : 0,
                     jb->col_num ? (int64_t)jb->planes * jb->n_c : 0, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace fa
