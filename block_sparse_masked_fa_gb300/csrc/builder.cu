// builder.cu -- the block-mask builder (create_block_mask of the speedrun
// notes "FlexAttention", tile-summary paragraph: evaluate mask_mod over the
// index grid and store, per query-tile row, the count and the column indices
// of the tiles that are not fully masked; tutorial "The two hooks": tiles are
// empty, partial or full).
//
// Kernels, all stream-ordered, no host synchronisation:
//  1. tile_summary  -- doc-id min / max of every query and key tile (only when
//                      the program has SAME_DOC); reads the doc ids once.
//  2. classify_rows -- one warp per query-tile row.  Each lane classifies one
//                      tile of a 32-tile chunk with a three-valued interval
//                      test per atom (nothing / everything / undecided visible,
//                      combined with Kleene AND / OR); undecided tiles are
//                      settled exactly by evaluating all their pairs with the
//                      whole warp.  Ballot + popcount prefix sums compact the
//                      PARTIAL and FULL column indices; tails are zeroed.
//  3. classify_cols -- one warp per key-tile column, same compaction over the
//                      tile classes written by (2): the backward's lists.
//  4. order         -- rows (then columns) sorted by descending tile count
//                      with a counting sort, the order the attention kernels
//                      take their work in (longest first).
#include "internal.h"

namespace fa {
namespace {

enum : int { K_NONE = 0, K_ALL = 1, K_SOME = 2 };

__device__ __forceinline__ int kleene_and(int a, int b) {
  return (a == K_NONE || b == K_NONE) ? K_NONE : ((a == K_ALL && b == K_ALL) ? K_ALL : K_SOME);
}
__device__ __forceinline__ int kleene_or(int a, int b) {
  return (a == K_ALL || b == K_ALL) ? K_ALL : ((a == K_NONE && b == K_NONE) ? K_NONE : K_SOME);
}

// Three-valued class of the whole program over rows [i0, i1] x cols [j0, j1]
// (inclusive).  q_mn/q_mx and k_mn/k_mx bound the doc ids of the two ranges.
__device__ int program_interval(const DevMask& m, const int32_t* arg, int64_t i0, int64_t i1, int64_t j0, int64_t j1,
                                int q_mn, int q_mx, int k_mn, int k_mx) {
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
        if (op == FA_M_CAUSAL) {            // i >= j
          c = (i0 >= j1) ? K_ALL : (i1 < j0 ? K_NONE : K_SOME);
        } else if (op == FA_M_WINDOW) {     // i - j < W
          c = (i1 - j0 < a) ? K_ALL : (i0 - j1 >= a ? K_NONE : K_SOME);
        } else if (op == FA_M_SINK || op == FA_M_PREFIX) {  // j < n
          c = (j1 < a) ? K_ALL : (j0 >= a ? K_NONE : K_SOME);
        } else if (op == FA_M_SAME_DOC) {
          c = (q_mx < k_mn || k_mx < q_mn) ? K_NONE
                                           : ((q_mn == q_mx && k_mn == k_mx && q_mn == k_mn) ? K_ALL : K_SOME);
        } else {
          c = K_ALL;
        }
        s7 = s6; s6 = s5; s5 = s4; s4 = s3; s3 = s2; s2 = s1; s1 = s0; s0 = c;
      }
    }
  }
  return s0;
}

__global__ void tile_summary_kernel(BuildArgs a) {
  const int warps = blockDim.x / 32;
  const int64_t w = (int64_t)blockIdx.x * warps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int tmax = max(a.nq, a.nkv);
  if (w >= (int64_t)a.Bm * 2 * tmax) return;
  const int t = (int)(w % tmax);
  const int which = (int)((w / tmax) % 2);  // 0: query tiles, 1: key tiles
  const int bm = (int)(w / (2 * tmax));
  const int64_t len = which ? a.kv_len : a.q_len;
  const int ntiles = which ? a.nkv : a.nq;
  if (t >= ntiles) return;
  const int32_t* doc = a.mask.doc + (int64_t)bm * a.mask.doc_len;
  const int64_t i0 = (int64_t)t * a.block;
  const int64_t i1 = min(i0 + a.block, len);
  int mn = INT_MAX, mx = INT_MIN;
  for (int64_t i = i0 + lane; i < i1; i += 32) {
    const int d = __ldg(doc + i);
    mn = min(mn, d);
    mx = max(mx, d);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    int32_t* s = a.summary + (((int64_t)bm * 2 + which) * tmax + t) * 2;
    s[0] = mn;
    s[1] = mx;
  }
}

constexpr int kBuildWarps = 8;

__global__ void __launch_bounds__(kBuildWarps * 32) classify_rows_kernel(BuildArgs a) {
  __shared__ int32_t s_arg[kBuildWarps][FA_MAX_MASK_NODES];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t row = (int64_t)blockIdx.x * kBuildWarps + warp;  // (bm, hm, I)
  if (row >= (int64_t)a.Bm * a.Hm * a.nq) return;
  const int I = (int)(row % a.nq);
  const int bm = (int)(row / ((int64_t)a.Hm * a.nq));
  if (lane < a.mask.n) s_arg[warp][lane] = node_arg(a.mask, lane, bm);
  __syncwarp();
  const int32_t* arg = s_arg[warp];
  const int tmax = max(a.nq, a.nkv);
  const int32_t* doc = a.mask.has_doc ? a.mask.doc + (int64_t)bm * a.mask.doc_len : nullptr;

  const int64_t i0 = (int64_t)I * a.block;
  const int64_t i1 = min(i0 + a.block, a.q_len) - 1;
  int q_mn = 0, q_mx = 0;
  if (a.mask.has_doc) {
    const int32_t* s = a.summary + (((int64_t)bm * 2 + 0) * tmax + I) * 2;
    q_mn = s[0];
    q_mx = s[1];
  }
  const int64_t base = row * a.nkv;
  int n_part = 0, n_full = 0;
  for (int c0 = 0; c0 < a.nkv; c0 += 32) {
    const int J = c0 + lane;
    const bool valid = J < a.nkv;
    int cls = 0;
    int k3 = K_NONE;
    if (valid) {
      const int64_t j0 = (int64_t)J * a.block;
      const int64_t j1 = min(j0 + a.block, a.kv_len) - 1;
      int k_mn = 0, k_mx = 0;
      if (a.mask.has_doc) {
        const int32_t* s = a.summary + (((int64_t)bm * 2 + 1) * tmax + J) * 2;
        k_mn = s[0];
        k_mx = s[1];
      }
      k3 = program_interval(a.mask, arg, i0, i1, j0, j1, q_mn, q_mx, k_mn, k_mx);
      cls = (k3 == K_ALL) ? 2 : 0;
    }
    // Settle undecided tiles exactly, one at a time with the whole warp.
    uint32_t undecided = __ballot_sync(0xffffffffu, valid && k3 == K_SOME);
    while (undecided) {
      const int t = __ffs(undecided) - 1;
      undecided &= undecided - 1;
      const int Jt = c0 + t;
      const int64_t j0 = (int64_t)Jt * a.block;
      const int64_t j1 = min(j0 + a.block, a.kv_len) - 1;
      const int64_t rows = i1 - i0 + 1, cols = j1 - j0 + 1;
      long long cnt = 0;
      for (int64_t r = lane; r < rows; r += 32) {
        const int64_t i = i0 + r;
        const int32_t doc_i = doc ? __ldg(doc + i) : 0;
        for (int64_t jc = j0; jc <= j1; jc += 32) {
          auto eq = [&]() {
            uint32_t w = 0;
            const int64_t jn = min(jc + 32, j1 + 1);
            for (int64_t j = jc; j < jn; ++j) w |= (uint32_t)(__ldg(doc + j) == doc_i) << (uint32_t)(j - jc);
            return w;
          };
          const uint32_t w = mask_word(a.mask, arg, i, jc, eq) & low_bits(j1 + 1 - jc);
          cnt += __popc(w);
        }
      }
      // warp sum (counts fit in 32 bits: at most 128 * 128 per tile)
      const int total = __reduce_add_sync(0xffffffffu, (unsigned)cnt);
      const int c = (total == 0) ? 0 : ((int64_t)total == rows * cols ? 2 : 1);
      if (lane == t) cls = c;
    }
    if (valid) a.tile_class[base + J] = (uint8_t)cls;
    const uint32_t pb = __ballot_sync(0xffffffffu, cls == 1);
    const uint32_t fb = __ballot_sync(0xffffffffu, cls == 2);
    const uint32_t lt = (1u << lane) - 1u;
    if (cls == 1) a.kv_idx[base + n_part + __popc(pb & lt)] = J;
    if (cls == 2) a.full_idx[base + n_full + __popc(fb & lt)] = J;
    n_part += __popc(pb);
    n_full += __popc(fb);
  }
  for (int k = n_part + lane; k < a.nkv; k += 32) a.kv_idx[base + k] = 0;
  for (int k = n_full + lane; k < a.nkv; k += 32) a.full_idx[base + k] = 0;
  if (lane == 0) {
    a.kv_num[row] = n_part;
    a.full_num[row] = n_full;
  }
}

__global__ void __launch_bounds__(kBuildWarps * 32) classify_cols_kernel(BuildArgs a) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t col = (int64_t)blockIdx.x * kBuildWarps + warp;  // (bm, hm, J)
  if (col >= (int64_t)a.Bm * a.Hm * a.nkv) return;
  const int J = (int)(col % a.nkv);
  const int64_t bmhm = col / a.nkv;
  const uint8_t* cls_base = a.tile_class + bmhm * a.nq * a.nkv + J;
  const int64_t base = col * a.nq;
  int n_part = 0, n_full = 0;
  for (int c0 = 0; c0 < a.nq; c0 += 32) {
    const int I = c0 + lane;
    const int cls = (I < a.nq) ? cls_base[(int64_t)I * a.nkv] : 0;
    const uint32_t pb = __ballot_sync(0xffffffffu, cls == 1);
    const uint32_t fb = __ballot_sync(0xffffffffu, cls == 2);
    const uint32_t lt = (1u << lane) - 1u;
    if (cls == 1) a.q_idx[base + n_part + __popc(pb & lt)] = I;
    if (cls == 2) a.full_q_idx[base + n_full + __popc(fb & lt)] = I;
    n_part += __popc(pb);
    n_full += __popc(fb);
  }
  for (int k = n_part + lane; k < a.nq; k += 32) a.q_idx[base + k] = 0;
  for (int k = n_full + lane; k < a.nq; k += 32) a.full_q_idx[base + k] = 0;
  if (lane == 0) {
    a.q_num[col] = n_part;
    a.full_q_num[col] = n_full;
  }
}

// Counting sort of n items by descending (num + full_num); one block.
// hist has max_count + 1 buckets in dynamic shared memory.
__global__ void __launch_bounds__(1024) order_kernel(const int32_t* num, const int32_t* full_num, int32_t n,
                                                     int32_t max_count, int32_t* order) {
  extern __shared__ int32_t hist[];
  const int nb = max_count + 1;
  for (int k = threadIdx.x; k < nb; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const int c = min(num[r] + full_num[r], max_count);
    atomicAdd(&hist[max_count - c], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int k = 0; k < nb; ++k) {
      const int h = hist[k];
      hist[k] = run;
      run += h;
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const int c = min(num[r] + full_num[r], max_count);
    order[atomicAdd(&hist[max_count - c], 1)] = r;
  }
}

__global__ void identity_order_kernel(int32_t n, int32_t* order) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r < n) order[r] = (int32_t)r;
}

constexpr int kMaxSortBuckets = 12 * 1024;  // 48 KB of shared memory

cudaError_t launch_order(const int32_t* num, const int32_t* full_num, int64_t n, int32_t max_count, int32_t* order,
                         cudaStream_t stream) {
  if (max_count + 1 <= kMaxSortBuckets) {
    order_kernel<<<1, 1024, (size_t)(max_count + 1) * sizeof(int32_t), stream>>>(num, full_num, (int32_t)n,
                                                                                max_count, order);
  } else {
    identity_order_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>((int32_t)n, order);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_build(const BuildArgs& a, cudaStream_t stream) {
  const int tmax = a.nq > a.nkv ? a.nq : a.nkv;
  if (a.mask.has_doc) {
    const int64_t warps = (int64_t)a.Bm * 2 * tmax;
    tile_summary_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(a);
  }
  const int64_t rows = (int64_t)a.Bm * a.Hm * a.nq;
  const int64_t cols = (int64_t)a.Bm * a.Hm * a.nkv;
  classify_rows_kernel<<<(unsigned)((rows + kBuildWarps - 1) / kBuildWarps), kBuildWarps * 32, 0, stream>>>(a);
  classify_cols_kernel<<<(unsigned)((cols + kBuildWarps - 1) / kBuildWarps), kBuildWarps * 32, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_order(a.kv_num, a.full_num, rows, a.nkv, a.row_order, stream);
  if (e != cudaSuccess) return e;
  return launch_order(a.q_num, a.full_q_num, cols, a.nq, a.col_order, stream);
}

}  // namespace fa
