// internal.h -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace fa {

// Runs a setter once per device: function attributes such as the dynamic
// shared-memory limit belong to the device that was current when they were set,
// so a launcher keeps one flag per device index, guarded against host threads
// that launch at the same time.  A failed setter is retried on the next call.
struct PerDeviceOnce {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  bool done[kMaxDevices] = {};

  template <typename F>
  cudaError_t run(F&& setter) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = setter();
    if (e == cudaSuccess) done[dev] = true;
    return e;
  }
};

// One class grid [planes][n_r][n_c] (planes = Bm * Hm) and the lists built
// from it: per row (null row_num: none) and per column (null col_num: none),
// with their work orders.
struct ListJob {
  uint8_t* cls;
  int32_t planes, n_r, n_c;
  int32_t *row_num, *row_idx, *row_full_num, *row_full_idx, *row_order;
  int32_t *col_num, *col_idx, *col_full_num, *col_full_idx, *col_order;
};

struct BuildArgs {
  DevMask mask;
  int32_t Bm, Hm, block, nq, nkv;
  int64_t q_len, kv_len;
  int32_t *kv_num, *kv_idx, *full_num, *full_idx;
  int32_t *q_num, *q_idx, *full_q_num, *full_q_idx;
  int32_t *row_order, *col_order;
  uint8_t* tile_class;
  int32_t* summary;  // [Bm][2][max(nq, nkv)][4]: doc-id min, max, step-0/1 flag per query / key tile
  int32_t* doc_runs;  // [Bm][max(q_len, kv_len)][2] runs, then [Bm] sorted flags
  int32_t* row_segs;  // [Bm][2][max(q_len, kv_len)][4] visible intervals per row / column
  uint32_t* status;
  // Caller-chosen tiles (fa_block_mask_from_kv_blocks), else null: per query-tile
  // row a count and sel_stride indices of PARTIAL (sel_*) and FULL (sel_full_*)
  // tiles, [Bm][Hm][nq] and [Bm][Hm][nq][sel_stride]; they replace classification.
  const int32_t *sel_num, *sel_idx, *sel_full_num, *sel_full_idx;
  int32_t sel_stride;
  // block < 128: the attention kernels' coarser grids, built from tile_class --
  // the forward's rows of 128 query positions over key tiles of fwd_kv_block,
  // the backward's columns of 128 key positions over query tiles of 128
  // (fwd.cls null at block 128)
  ListJob fwd, bwd;
  int32_t fwd_kv_block;
};

// Launches a kernel on `stream` allowed to start while the kernel before it
// drains (programmatic stream serialization); the kernel itself waits for that
// one to complete before touching memory (pdl_wait_then_release).  Used for the
// builder's chain of short kernels and the decode combine; the attention
// kernels, which fill every SM, measured slower launched this way and are
// launched plainly.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_build(const BuildArgs& a, cudaStream_t stream);

// Work description shared by the forward and backward kernels.
struct AttnArgs {
  int32_t B, H, Bm, Hm, nq, nkv, D;
  int32_t q_len, kv_len;
  const int32_t *kv_num, *kv_idx, *full_num, *full_idx;        // per query-tile row
  const int32_t *q_num, *q_idx, *full_q_num, *full_q_idx;      // per key-tile column
  const int32_t *row_order, *col_order;
  float scale;
  int32_t score_op;
  const float* score_param;
  float* param_grad;  // backward only: dL/dslope[H] (ALiBi), dL/dbias[H][bias_len] (RELBIAS), or null
  int32_t bias_len, bias_d0;  // RELBIAS: table length per head, distance of entry 0
  // forward only: paged keys / values -- page of logical key tile J of batch b
  // at page_table[b * nkv + J], pages of 128 rows in [H][n_pages * 128][D] pools; or null
  const int32_t* page_table;
  int32_t n_pages;
  // forward: a buffer its producer warps set to zero while it runs (the dq
  // accumulator of a backward workspace; 16-byte units), or null
  uint4* zero_dst;
  int64_t zero_n16;
  // backward: the dq accumulator is already zero (set so by such a forward)
  int32_t acc_zeroed;
  uint32_t* status;
  DevMask mask;
  const int4* row_segs;  // [Bm][2][seg_len]: see fa_block_mask
  int64_t seg_len;
  int32_t kv_block;  // forward: key positions per listed key tile (128, or 64 below block 128)
  int32_t kv_cap;    // short-query forward: rows per (b, h) of k / v (>= kv_len: a bucketed cache)
};

struct FwdTensors {
  const void *q, *k, *v;
  void* out;
  float* lse;
};

struct BwdTensors {
  const void *q, *k, *v, *out, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* dq_acc;  // fp32 [B, H, q_len, D]
  float* stats;   // fp32 [B, H, nq][2][128]: -LSE * log2(e) and -Delta per query tile
  uint32_t* sched;  // the main kernel's item counter (zeroed by bwd_pre)
};

// Returns a CUDA error, or cudaErrorUnknown with *enc_failed set when a
// tensor map could not be encoded.
cudaError_t launch_forward(const AttnArgs& a, const FwdTensors& t, cudaStream_t stream, bool* enc_failed);
cudaError_t launch_backward(const AttnArgs& a, const BwdTensors& t, cudaStream_t stream, bool* enc_failed);

// Short-query forward: the split of every (b, h)'s key tiles over CTAs on the
// current device and the workspace it needs (partial out and LSE per split),
// and the launch (decode_partial_kernel, then decode_combine_kernel).
cudaError_t decode_plan(int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, int* splits,
                        size_t* ws_bytes);
cudaError_t launch_decode(const AttnArgs& a, const FwdTensors& t, void* workspace, int splits, cudaStream_t stream,
                          bool* enc_failed);

// Device address (current device) of the library-owned scratch of fa_backward_noalloc.
cudaError_t noalloc_scratch(void** ptr);

#ifdef FA_TEST_HOOKS
// Test library only: make the producer of block 0 skip the load (and the
// arrive) of the key tile of its first step, so that the MMA warp's bounded
// wait for it runs out and the kernel takes its give-up path.
cudaError_t test_hook_forward(int on);
cudaError_t test_hook_backward(int on);
#endif

// Tensor-map encoding through the driver entry point (no libcuda link).
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t d0,
                    uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

}  // namespace fa
