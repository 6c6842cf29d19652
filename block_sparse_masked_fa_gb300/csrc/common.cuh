// common.cuh -- definitions shared by the block-mask builder and the attention
// kernels: the device copy of a mask program and its evaluation.
//
// A mask program (tutorial "FlexAttention in PyTorch", sections "The two
// hooks" and Patterns 1-3) is evaluated 32 key columns at a time: for one
// query row i and columns j0 .. j0+31 every atom yields a 32-bit word whose bit
// c says whether (i, j0 + c) is visible, and AND / OR combine the words.  The
// operand stack is a fixed set of eight registers shifted on push and pop, so
// the evaluation never touches local memory.
#pragma once
#include <climits>
#include <cstdint>

#include "fa.h"

namespace fa {

constexpr uint32_t kStatusTimeout = 1u;  // a bounded wait gave up
constexpr uint32_t kStatusCheck = 2u;    // a device range check failed

// Device copy of a mask program: node kinds by value, parameters as device
// pointers.  `doc` is the (single) SAME_DOC array, row-major [Bm][doc_len].
struct DevMask {
  int32_t n;
  int32_t has_doc;
  int32_t doc_vec_ok;  // doc rows are 16-byte aligned (base and doc_len % 4 == 0)
  int64_t doc_len;
  const int32_t* doc;
  // runs of equal ids: [Bm][run_len] pairs (lo, hi) and per batch row a flag
  // set when that row's ids never decrease (filled by the builder)
  const int32_t* runs;
  const int32_t* sorted;
  int64_t run_len;
  int64_t q_off;  // position of query row 0 (fa_mask_spec::q_offset)
  int32_t op[FA_MAX_MASK_NODES];
  const int32_t* param[FA_MAX_MASK_NODES];
};

// Scalar parameter of node k for batch row bm: W, n_sink or prefix_len[bm].
__device__ __forceinline__ int32_t node_arg(const DevMask& m, int k, int bm) {
  const int op = m.op[k];
  if (op == FA_M_WINDOW || op == FA_M_SINK) return __ldg(m.param[k]);
  if (op == FA_M_PREFIX) return __ldg(m.param[k] + bm);
  return 0;
}

// Bits [0, n) set, n clamped to [0, 32].
__device__ __forceinline__ uint32_t low_bits(int64_t n) {
  return n <= 0 ? 0u : (n >= 32 ? 0xffffffffu : ((1u << (uint32_t)n) - 1u));
}

// Word of the positions x0 .. x0+31 inside [lo, hi).
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int x0) {
  return low_bits((int64_t)hi - x0) & ~low_bits((int64_t)lo - x0);
}

// The run [lo, hi) of position x in batch row bm when that row's ids never
// decrease, so that doc[y] == doc[x] exactly for y in [lo, hi).  Returns false
// (and the caller compares ids one by one) otherwise.
__device__ __forceinline__ bool doc_run(const DevMask& m, int bm, int64_t x, int& lo, int& hi) {
  if (m.runs == nullptr || __ldg(m.sorted + bm) == 0) return false;
  const int2 r = __ldg(reinterpret_cast<const int2*>(m.runs) + (int64_t)bm * m.run_len + x);
  lo = r.x;
  hi = r.y;
  return true;
}

// Visibility word of query row i over key columns j0 .. j0+31.
//  arg[k]    resolved scalar parameter of node k (see node_arg)
//  eq_doc()  word of (doc[j0 + c] == doc[i]) for c = 0..31
template <class EqDoc>
__device__ __forceinline__ uint32_t mask_word(const DevMask& m, const int32_t* arg, int64_t i, int64_t j0,
                                              EqDoc eq_doc) {
  uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0, s5 = 0, s6 = 0, s7 = 0;
#pragma unroll
  for (int k = 0; k < FA_MAX_MASK_NODES; ++k) {
    if (k < m.n) {
      const int op = m.op[k];
      if (op == FA_M_AND || op == FA_M_OR) {
        s0 = (op == FA_M_AND) ? (s1 & s0) : (s1 | s0);
        s1 = s2; s2 = s3; s3 = s4; s4 = s5; s5 = s6; s6 = s7; s7 = 0;
      } else {
        uint32_t w;
        if (op == FA_M_CAUSAL) {
          w = low_bits(i - j0 + 1);                      // j <= i
        } else if (op == FA_M_WINDOW) {
          w = ~low_bits(i - (int64_t)arg[k] + 1 - j0);   // j >= i - W + 1
        } else if (op == FA_M_SINK || op == FA_M_PREFIX) {
          w = low_bits((int64_t)arg[k] - j0);            // j < n
        } else if (op == FA_M_SAME_DOC) {
          w = eq_doc();
        } else {
          w = 0xffffffffu;                               // FA_M_TRUE
        }
        s7 = s6; s6 = s5; s5 = s4; s4 = s3; s3 = s2; s2 = s1; s1 = s0; s0 = w;
      }
    }
  }
  return s0;
}

// Node kinds of a mask program packed four bits each (node k in bits
// [4k, 4k + 4)).  Built once per thread from the kernel argument with constant
// indices, so that the rolled evaluators below read registers only: indexing
// the argument's op[] with a loop counter goes through a generic pointer into
// parameter space, which costs hundreds of cycles per node.
__device__ __forceinline__ uint64_t pack_ops(const DevMask& m) {
  static_assert(FA_MAX_MASK_NODES * 4 <= 64, "node kinds must fit one 64-bit word");
  uint64_t ops = 0;
#pragma unroll
  for (int k = 0; k < FA_MAX_MASK_NODES; ++k)
    if (k < m.n) ops |= (uint64_t)(m.op[k] & 15) << (4 * k);
  return ops;
}

// Same as mask_word, with the node loop kept rolled: small code for the
// attention kernels' partial tiles.
//  n, ops    node count and packed node kinds (pack_ops)
//  arg[k]    resolved scalar parameter of node k for this batch row (node_arg)
template <class EqDoc>
__device__ __forceinline__ uint32_t mask_word_rolled(int n, uint64_t ops, const int32_t* arg, int64_t i,
                                                     int64_t j0, EqDoc eq_doc) {
  uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0, s5 = 0, s6 = 0, s7 = 0;
#pragma unroll 1
  for (int k = 0; k < n; ++k, ops >>= 4) {
    const int op = (int)(ops & 15u);
    if (op == FA_M_AND || op == FA_M_OR) {
      s0 = (op == FA_M_AND) ? (s1 & s0) : (s1 | s0);
      s1 = s2; s2 = s3; s3 = s4; s4 = s5; s5 = s6; s6 = s7; s7 = 0;
    } else {
      uint32_t w;
      if (op == FA_M_CAUSAL) {
        w = low_bits(i - j0 + 1);                          // j <= i
      } else if (op == FA_M_WINDOW) {
        w = ~low_bits(i - (int64_t)arg[k] + 1 - j0);       // j >= i - W + 1
      } else if (op == FA_M_SINK || op == FA_M_PREFIX) {
        w = low_bits((int64_t)arg[k] - j0);                // j < n
      } else if (op == FA_M_SAME_DOC) {
        w = eq_doc();
      } else {
        w = 0xffffffffu;
      }
      s7 = s6; s6 = s5; s5 = s4; s4 = s3; s3 = s2; s2 = s1; s1 = s0; s0 = w;
    }
  }
  return s0;
}

// Transposed visibility word: key column j fixed, query rows i0 .. i0+31
// (bit c is pair (i0 + c, j)); used where a thread owns a key row.
//  eq_doc()  word of (doc[i0 + c] == doc[j]) for c = 0..31
template <class EqDoc>
__device__ __forceinline__ uint32_t mask_word_t_rolled(int n, uint64_t ops, const int32_t* arg, int64_t j,
                                                       int64_t i0, EqDoc eq_doc) {
  uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0, s5 = 0, s6 = 0, s7 = 0;
#pragma unroll 1
  for (int k = 0; k < n; ++k, ops >>= 4) {
    const int op = (int)(ops & 15u);
    if (op == FA_M_AND || op == FA_M_OR) {
      s0 = (op == FA_M_AND) ? (s1 & s0) : (s1 | s0);
      s1 = s2; s2 = s3; s3 = s4; s4 = s5; s5 = s6; s6 = s7; s7 = 0;
    } else {
      uint32_t w;
      if (op == FA_M_CAUSAL) {
        w = ~low_bits(j - i0);                              // i >= j
      } else if (op == FA_M_WINDOW) {
        w = low_bits(j + (int64_t)arg[k] - i0);             // i < j + W
      } else if (op == FA_M_SINK || op == FA_M_PREFIX) {
        w = (j < (int64_t)arg[k]) ? 0xffffffffu : 0u;       // j < n
      } else if (op == FA_M_SAME_DOC) {
        w = eq_doc();
      } else {
        w = 0xffffffffu;
      }
      s7 = s6; s6 = s5; s5 = s4; s4 = s3; s3 = s2; s2 = s1; s1 = s0; s0 = w;
    }
  }
  return s0;
}

// Word of positions y0 .. y0+31 from a row's two visible intervals [s.x, s.y)
// and [s.z, s.w) (fa_block_mask::row_segs, where s.x >= 0).
__device__ __forceinline__ uint32_t seg_word(int4 s, int y0) {
  return range_bits(s.x, s.y, y0) | range_bits(s.z, s.w, y0);
}

}  // namespace fa
