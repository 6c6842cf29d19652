// api.cu -- the C ABI declared in include/fa.h: host-side validation, the
// block-mask buffer layout, tensor-map encoding and kernel launches.
// Everything here runs on the host; it never synchronises a stream except in
// fa_get_status and fa_block_mask_summary.
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "internal.h"

namespace fa {
namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kDecodeMaxHeads = 65535;  // the decode grid's second dimension is B * H
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Byte offsets of the block-mask arrays inside the caller's buffer.
struct Layout {
  enum {
    KV_NUM, KV_IDX, FULL_NUM, FULL_IDX, Q_NUM, Q_IDX, FULL_Q_NUM, FULL_Q_IDX, ROW_ORDER, COL_ORDER, TILE_CLASS,
    SUMMARY, DOC_RUNS, ROW_SEGS, STATUS,
    // block < 128 only (empty otherwise): the attention kernels' coarser tiles
    FWD_NUM, FWD_IDX, FWD_FULL_NUM, FWD_FULL_IDX, FWD_ORDER, FWD_CLASS,
    BWD_NUM, BWD_IDX, BWD_FULL_NUM, BWD_FULL_IDX, BWD_ORDER, BWD_CLASS, N
  };
  size_t off[N];
  size_t total;
  int64_t nq, nkv;
  int64_t fwd_nq, fwd_nkv, bwd_nq, bwd_nkv;  // 0 at block 128
};

constexpr int kFwdSmallKvBlock = 64;  // the forward's key tile below block 128

fa_status make_layout(int32_t Bm, int32_t Hm, int64_t q_len, int64_t kv_len, int32_t block, Layout* L) {
  if (Bm < 1 || Hm < 1 || q_len < 1 || kv_len < 1) return FA_ERR_SHAPE;
  if (block < 16 || block > 128 || (block & (block - 1)) != 0) return FA_ERR_UNSUPPORTED;
  if (q_len > (int64_t)INT32_MAX - 256 || kv_len > (int64_t)INT32_MAX - 256) return FA_ERR_SHAPE;
  const int64_t nq = (q_len + block - 1) / block, nkv = (kv_len + block - 1) / block;
  const int64_t rows = (int64_t)Bm * Hm * nq, cols = (int64_t)Bm * Hm * nkv;
  const int64_t tiles = rows * nkv;
  if (tiles > (int64_t)INT32_MAX || rows > (int64_t)INT32_MAX / 2 || cols > (int64_t)INT32_MAX / 2)
    return FA_ERR_SHAPE;
  const bool coarse = block < 128;
  const int64_t fnq = coarse ? (q_len + 127) / 128 : 0, fnkv = coarse ? (kv_len + kFwdSmallKvBlock - 1) / kFwdSmallKvBlock : 0;
  const int64_t bnq = fnq, bnkv = coarse ? (kv_len + 127) / 128 : 0;
  const size_t planes = (size_t)Bm * Hm;
  const size_t sizes[Layout::N] = {
      (size_t)rows * 4,  (size_t)tiles * 4, (size_t)rows * 4, (size_t)tiles * 4,
      (size_t)cols * 4,  (size_t)tiles * 4, (size_t)cols * 4, (size_t)tiles * 4,
      (size_t)rows * 4,  (size_t)cols * 4,  (size_t)tiles,
      (size_t)Bm * 2 * (size_t)(nq > nkv ? nq : nkv) * 4 * 4,
      (size_t)Bm * (size_t)(q_len > kv_len ? q_len : kv_len) * 8 + (size_t)Bm * 4,
      (size_t)Bm * 2 * (size_t)(q_len > kv_len ? q_len : kv_len) * 16,
      4,
      planes * fnq * 4, planes * fnq * fnkv * 4, planes * fnq * 4, planes * fnq * fnkv * 4, planes * fnq * 4,
      planes * fnq * fnkv,
      planes * bnkv * 4, planes * bnkv * bnq * 4, planes * bnkv * 4, planes * bnkv * bnq * 4, planes * bnkv * 4,
      planes * bnq * bnkv};
  size_t at = 0;
  for (int k = 0; k < Layout::N; ++k) {
    L->off[k] = at;
    at += align_up(sizes[k]);
  }
  L->total = at;
  L->nq = nq;
  L->nkv = nkv;
  L->fwd_nq = fnq;
  L->fwd_nkv = fnkv;
  L->bwd_nq = bnq;
  L->bwd_nkv = bnkv;
  return FA_OK;
}

// Checks a mask program and fills its device copy.
fa_status check_mask(const fa_mask_spec* spec, int64_t q_len, int64_t kv_len, DevMask* dm) {
  if (spec == nullptr) return FA_ERR_INVALID_ARG;
  if (spec->n < 1 || spec->n > FA_MAX_MASK_NODES) return FA_ERR_INVALID_ARG;
  std::memset(dm, 0, sizeof(*dm));
  dm->n = spec->n;
  int depth = 0;
  const int32_t* doc = nullptr;
  for (int k = 0; k < spec->n; ++k) {
    const int op = spec->node[k].op;
    const int32_t* prm = spec->node[k].param;
    switch (op) {
      case FA_M_TRUE:
      case FA_M_CAUSAL:
        depth += 1;
        break;
      case FA_M_WINDOW:
      case FA_M_SINK:
      case FA_M_PREFIX:
        if (prm == nullptr || !aligned4(prm)) return FA_ERR_INVALID_ARG;
        depth += 1;
        break;
      case FA_M_SAME_DOC:
        if (prm == nullptr || !aligned4(prm)) return FA_ERR_INVALID_ARG;
        if (doc != nullptr && doc != prm) return FA_ERR_INVALID_ARG;  // one doc array per program
        doc = prm;
        depth += 1;
        break;
      case FA_M_AND:
      case FA_M_OR:
        if (depth < 2) return FA_ERR_INVALID_ARG;
        depth -= 1;
        break;
      default:
        return FA_ERR_INVALID_ARG;
    }
    if (depth > FA_MAX_MASK_STACK) return FA_ERR_INVALID_ARG;
    dm->op[k] = op;
    dm->param[k] = prm;
  }
  if (depth != 1) return FA_ERR_INVALID_ARG;
  // every query row's position lies below max(q_len, kv_len), where the
  // document ids and their run table are defined
  const int64_t span = q_len > kv_len ? q_len : kv_len;
  if (spec->q_offset < 0 || spec->q_offset > span - q_len) return FA_ERR_INVALID_ARG;
  dm->q_off = spec->q_offset;
  if (doc != nullptr) {
    const int64_t need = q_len > kv_len ? q_len : kv_len;
    if (spec->doc_len < need) return FA_ERR_SHAPE;
    dm->has_doc = 1;
    dm->doc = doc;
    dm->doc_len = spec->doc_len;
    dm->doc_vec_ok = aligned16(doc) && (spec->doc_len % 4 == 0);
  }
  return FA_OK;
}

// ---- driver entry point for tensor-map encoding (the library does not link libcuda)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

fa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

enum AttnKind { kForward, kForwardPagedOrDecode, kDecode, kBackward };

// Shared shape checks of fa_forward / fa_backward.
fa_status check_attn(int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                     const fa_score_spec* score, float* scale, AttnKind kind) {
  const bool backward = kind == kBackward;
  if (bm == nullptr) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || q_len < 1 || kv_len < 1) return FA_ERR_SHAPE;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (bm->block != 128) {  // the kernels walk the coarser lists the builder derived
    if (kind == kForwardPagedOrDecode || kind == kDecode || bm->from_blocks) return FA_ERR_UNSUPPORTED;
    if (bm->block > 128 || bm->fwd_kv_block != kFwdSmallKvBlock) return FA_ERR_INVALID_ARG;
    if (backward ? (bm->bwd_q_num_blocks == nullptr || bm->bwd_col_order == nullptr)
                 : (bm->fwd_kv_num_blocks == nullptr || bm->fwd_row_order == nullptr))
      return FA_ERR_INVALID_ARG;
  }
  // the short-query forward may run on a block mask built for a longer (bucketed) cache
  if (bm->q_len != q_len || (kind == kDecode ? bm->kv_len < kv_len : bm->kv_len != kv_len)) return FA_ERR_SHAPE;
  if (!(bm->Bm == 1 || bm->Bm == B) || !(bm->Hm == 1 || bm->Hm == H)) return FA_ERR_SHAPE;
  if ((int64_t)B * H * ((q_len + 127) / 128) > (int64_t)INT32_MAX) return FA_ERR_SHAPE;
  if ((int64_t)B * H * ((kv_len + 127) / 128) > (int64_t)INT32_MAX) return FA_ERR_SHAPE;
  if (bm->status == nullptr || bm->row_order == nullptr) return FA_ERR_INVALID_ARG;
  if (score != nullptr) {
    if (score->op < FA_S_NONE || score->op > FA_S_RELBIAS) return FA_ERR_INVALID_ARG;
    if (score->op != FA_S_NONE && (score->param == nullptr || !aligned4(score->param))) return FA_ERR_INVALID_ARG;
    if (score->op == FA_S_RELBIAS && (score->bias_len < 1 || score->bias_len > (1 << 24) ||
                                      score->bias_d0 < -(1 << 30) || score->bias_d0 > (1 << 30)))
      return FA_ERR_INVALID_ARG;
    if (backward && score->param_grad != nullptr) {
      if (score->op != FA_S_ALIBI && score->op != FA_S_RELBIAS) return FA_ERR_UNSUPPORTED;
      if (!aligned4(score->param_grad)) return FA_ERR_ALIGNMENT;
    }
  }
  if (!(*scale >= 0.f) || std::isinf(*scale)) return FA_ERR_INVALID_ARG;
  if (*scale == 0.f) *scale = 1.0f / std::sqrt((float)D);
  return FA_OK;
}

AttnArgs attn_args(int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                   const fa_score_spec* score, float scale, DevMask dm, bool backward) {
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = B;
  a.H = H;
  a.Bm = bm->Bm;
  a.Hm = bm->Hm;
  a.nq = bm->nq;
  a.nkv = bm->nkv;
  a.D = D;
  a.q_len = (int32_t)q_len;
  a.kv_len = (int32_t)kv_len;
  a.kv_num = bm->kv_num_blocks;
  a.kv_idx = bm->kv_indices;
  a.full_num = bm->full_kv_num_blocks;
  a.full_idx = bm->full_kv_indices;
  a.q_num = bm->q_num_blocks;
  a.q_idx = bm->q_indices;
  a.full_q_num = bm->full_q_num_blocks;
  a.full_q_idx = bm->full_q_indices;
  a.row_order = bm->row_order;
  a.col_order = bm->col_order;
  a.scale = scale;
  a.score_op = score ? score->op : FA_S_NONE;
  a.score_param = score ? score->param : nullptr;
  a.param_grad = (backward && score) ? score->param_grad : nullptr;
  if (score != nullptr && score->op == FA_S_RELBIAS) {
    a.bias_len = score->bias_len;
    a.bias_d0 = score->bias_d0;
  }
  a.status = bm->status;
  a.mask = dm;
  a.kv_block = 128;
  a.kv_cap = (int32_t)kv_len;
  if (bm->block != 128 && !backward) {  // the forward's 128 x 64 tiles
    a.nq = bm->fwd_nq;
    a.nkv = bm->fwd_nkv;
    a.kv_block = bm->fwd_kv_block;
    a.kv_num = bm->fwd_kv_num_blocks;
    a.kv_idx = bm->fwd_kv_indices;
    a.full_num = bm->fwd_full_kv_num_blocks;
    a.full_idx = bm->fwd_full_kv_indices;
    a.row_order = bm->fwd_row_order;
    a.q_num = a.q_idx = a.full_q_num = a.full_q_idx = a.col_order = nullptr;
  } else if (bm->block != 128) {  // the backward's 128 x 128 tiles
    a.nq = bm->bwd_nq;
    a.nkv = bm->bwd_nkv;
    a.q_num = bm->bwd_q_num_blocks;
    a.q_idx = bm->bwd_q_indices;
    a.full_q_num = bm->bwd_full_q_num_blocks;
    a.full_q_idx = bm->bwd_full_q_indices;
    a.col_order = bm->bwd_col_order;
    a.kv_num = a.kv_idx = a.full_num = a.full_idx = a.row_order = nullptr;
  }
  a.row_segs = reinterpret_cast<const int4*>(bm->row_segs);
  a.seg_len = bm->q_len > bm->kv_len ? bm->q_len : bm->kv_len;
  if (dm.has_doc && bm->doc_runs != nullptr) {
    const int64_t run_len = bm->q_len > bm->kv_len ? bm->q_len : bm->kv_len;
    a.mask.runs = bm->doc_runs;
    a.mask.sorted = bm->doc_runs + 2 * (int64_t)bm->Bm * run_len;
    a.mask.run_len = run_len;
  }
  return a;
}

}  // namespace

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t d0,
                    uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * elem_bytes, d0 * d1 * elem_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared body of fa_create_block_mask and fa_block_mask_from_kv_blocks: lays
// out `buffer`, fills `bm` and queues the builder (with the caller's tile lists
// in place of classification when `sel` is set).
static fa_status build_block_mask(const fa_mask_spec* spec, int32_t Bm, int32_t Hm, int64_t q_len, int64_t kv_len,
                                  int32_t block, void* buffer, size_t buffer_bytes, fa_block_mask* bm,
                                  const BuildArgs* sel, cudaStream_t stream) {
  if (bm == nullptr || buffer == nullptr) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(buffer) & (kAlign - 1)) != 0) return FA_ERR_ALIGNMENT;
  Layout L;
  fa_status st = make_layout(Bm, Hm, q_len, kv_len, block, &L);
  if (st != FA_OK) return st;
  if (buffer_bytes < L.total) return FA_ERR_WORKSPACE;
  DevMask dm;
  st = check_mask(spec, q_len, kv_len, &dm);
  if (st != FA_OK) return st;

  uint8_t* base = static_cast<uint8_t*>(buffer);
  auto i32 = [&](int k) { return reinterpret_cast<int32_t*>(base + L.off[k]); };
  std::memset(bm, 0, sizeof(*bm));
  bm->Bm = Bm;
  bm->Hm = Hm;
  bm->block = block;
  bm->nq = (int32_t)L.nq;
  bm->nkv = (int32_t)L.nkv;
  bm->q_len = q_len;
  bm->kv_len = kv_len;
  bm->kv_num_blocks = i32(Layout::KV_NUM);
  bm->kv_indices = i32(Layout::KV_IDX);
  bm->full_kv_num_blocks = i32(Layout::FULL_NUM);
  bm->full_kv_indices = i32(Layout::FULL_IDX);
  bm->q_num_blocks = i32(Layout::Q_NUM);
  bm->q_indices = i32(Layout::Q_IDX);
  bm->full_q_num_blocks = i32(Layout::FULL_Q_NUM);
  bm->full_q_indices = i32(Layout::FULL_Q_IDX);
  bm->row_order = i32(Layout::ROW_ORDER);
  bm->col_order = i32(Layout::COL_ORDER);
  bm->tile_class = base + L.off[Layout::TILE_CLASS];
  bm->tile_summary = i32(Layout::SUMMARY);
  bm->doc_runs = i32(Layout::DOC_RUNS);
  bm->row_segs = i32(Layout::ROW_SEGS);
  bm->status = reinterpret_cast<uint32_t*>(base + L.off[Layout::STATUS]);
  bm->spec = *spec;
  bm->from_blocks = sel != nullptr ? 1 : 0;
  if (block < 128) {
    bm->fwd_kv_block = kFwdSmallKvBlock;
    bm->fwd_nq = (int32_t)L.fwd_nq;
    bm->fwd_nkv = (int32_t)L.fwd_nkv;
    bm->bwd_nq = (int32_t)L.bwd_nq;
    bm->bwd_nkv = (int32_t)L.bwd_nkv;
    bm->fwd_kv_num_blocks = i32(Layout::FWD_NUM);
    bm->fwd_kv_indices = i32(Layout::FWD_IDX);
    bm->fwd_full_kv_num_blocks = i32(Layout::FWD_FULL_NUM);
    bm->fwd_full_kv_indices = i32(Layout::FWD_FULL_IDX);
    bm->fwd_row_order = i32(Layout::FWD_ORDER);
    bm->fwd_tile_class = base + L.off[Layout::FWD_CLASS];
    bm->bwd_q_num_blocks = i32(Layout::BWD_NUM);
    bm->bwd_q_indices = i32(Layout::BWD_IDX);
    bm->bwd_full_q_num_blocks = i32(Layout::BWD_FULL_NUM);
    bm->bwd_full_q_indices = i32(Layout::BWD_FULL_IDX);
    bm->bwd_col_order = i32(Layout::BWD_ORDER);
    bm->bwd_tile_class = base + L.off[Layout::BWD_CLASS];
  }

  cudaError_t e = cudaMemsetAsync(bm->status, 0, 4, stream);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  BuildArgs a;
  std::memset(&a, 0, sizeof(a));
  a.mask = dm;
  a.Bm = Bm;
  a.Hm = Hm;
  a.block = block;
  a.nq = bm->nq;
  a.nkv = bm->nkv;
  a.q_len = q_len;
  a.kv_len = kv_len;
  a.kv_num = bm->kv_num_blocks;
  a.kv_idx = bm->kv_indices;
  a.full_num = bm->full_kv_num_blocks;
  a.full_idx = bm->full_kv_indices;
  a.q_num = bm->q_num_blocks;
  a.q_idx = bm->q_indices;
  a.full_q_num = bm->full_q_num_blocks;
  a.full_q_idx = bm->full_q_indices;
  a.row_order = bm->row_order;
  a.col_order = bm->col_order;
  a.tile_class = bm->tile_class;
  a.summary = bm->tile_summary;
  a.doc_runs = bm->doc_runs;
  a.row_segs = bm->row_segs;
  a.status = bm->status;
  if (block < 128) {
    a.fwd_kv_block = bm->fwd_kv_block;
    a.fwd.cls = bm->fwd_tile_class;
    a.fwd.planes = Bm * Hm;
    a.fwd.n_r = bm->fwd_nq;
    a.fwd.n_c = bm->fwd_nkv;
    a.fwd.row_num = bm->fwd_kv_num_blocks;
    a.fwd.row_idx = bm->fwd_kv_indices;
    a.fwd.row_full_num = bm->fwd_full_kv_num_blocks;
    a.fwd.row_full_idx = bm->fwd_full_kv_indices;
    a.fwd.row_order = bm->fwd_row_order;
    a.bwd.cls = bm->bwd_tile_class;
    a.bwd.planes = Bm * Hm;
    a.bwd.n_r = bm->bwd_nq;
    a.bwd.n_c = bm->bwd_nkv;
    a.bwd.col_num = bm->bwd_q_num_blocks;
    a.bwd.col_idx = bm->bwd_q_indices;
    a.bwd.col_full_num = bm->bwd_full_q_num_blocks;
    a.bwd.col_full_idx = bm->bwd_full_q_indices;
    a.bwd.col_order = bm->bwd_col_order;
  }
  if (sel != nullptr) {
    a.sel_num = sel->sel_num;
    a.sel_idx = sel->sel_idx;
    a.sel_full_num = sel->sel_full_num;
    a.sel_full_idx = sel->sel_full_idx;
    a.sel_stride = sel->sel_stride;
  }
  if (dm.has_doc) {  // classify reads the run table that the builder fills first
    const int64_t run_len = q_len > kv_len ? q_len : kv_len;
    a.mask.runs = bm->doc_runs;
    a.mask.sorted = bm->doc_runs + 2 * (int64_t)Bm * run_len;
    a.mask.run_len = run_len;
  }
  return cuda_status(launch_build(a, stream));
}

}  // namespace fa

using namespace fa;

extern "C" {

int32_t fa_version(void) { return 100; }

#ifdef FA_TEST_HOOKS
// Exported by the test library only (never by the product build): which = 0
// clears both hooks, 1 starves the forward's first key-tile load, 2 the
// backward's (see test_hook_forward in internal.h).
fa_status fa_test_hook(int32_t which) {
  if (which < 0 || which > 2) return FA_ERR_INVALID_ARG;
  if (fa::test_hook_forward(which == 1) != cudaSuccess || fa::test_hook_backward(which == 2) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}
#endif

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_SHAPE: return "bad or inconsistent shape";
    case FA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    case FA_ERR_DEVICE_CHECK: return "device range check failed";
    case FA_ERR_WORKSPACE: return "buffer too small";
  }
  return "unknown status";
}

fa_status fa_block_mask_bytes(int32_t Bm, int32_t Hm, int64_t q_len, int64_t kv_len, int32_t block, size_t* bytes) {
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  Layout L;
  const fa_status st = make_layout(Bm, Hm, q_len, kv_len, block, &L);
  if (st != FA_OK) return st;
  *bytes = L.total;
  return FA_OK;
}

fa_status fa_create_block_mask(const fa_mask_spec* spec, int32_t Bm, int32_t Hm, int64_t q_len, int64_t kv_len,
                               int32_t block, void* buffer, size_t buffer_bytes, fa_block_mask* bm,
                               cudaStream_t stream) {
  return build_block_mask(spec, Bm, Hm, q_len, kv_len, block, buffer, buffer_bytes, bm, nullptr, stream);
}

fa_status fa_block_mask_from_kv_blocks(const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                       const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                       int32_t idx_stride, const fa_mask_spec* spec, int32_t Bm, int32_t Hm,
                                       int64_t q_len, int64_t kv_len, int32_t block, void* buffer,
                                       size_t buffer_bytes, fa_block_mask* bm, cudaStream_t stream) {
  if (kv_num_blocks == nullptr || kv_indices == nullptr) return FA_ERR_INVALID_ARG;
  if ((full_kv_num_blocks == nullptr) != (full_kv_indices == nullptr)) return FA_ERR_INVALID_ARG;
  if (!aligned4(kv_num_blocks) || !aligned4(kv_indices) || !aligned4(full_kv_num_blocks) ||
      !aligned4(full_kv_indices))
    return FA_ERR_ALIGNMENT;
  if (idx_stride < 1) return FA_ERR_SHAPE;
  fa_mask_spec all;  // no program: every pair of a listed PARTIAL tile is visible
  if (spec == nullptr) {
    std::memset(&all, 0, sizeof(all));
    all.n = 1;
    all.node[0].op = FA_M_TRUE;
    spec = &all;
  }
  BuildArgs sel;
  std::memset(&sel, 0, sizeof(sel));
  sel.sel_num = kv_num_blocks;
  sel.sel_idx = kv_indices;
  sel.sel_full_num = full_kv_num_blocks;
  sel.sel_full_idx = full_kv_indices;
  sel.sel_stride = idx_stride;
  return build_block_mask(spec, Bm, Hm, q_len, kv_len, block, buffer, buffer_bytes, bm, &sel, stream);
}

fa_status fa_forward(const void* q, const void* k, const void* v, int32_t B, int32_t H, int64_t q_len,
                     int64_t kv_len, int32_t D, const fa_block_mask* bm, const fa_score_spec* score, float scale,
                     void* out, float* lse, cudaStream_t stream) {
  return fa_forward_paged(q, k, v, nullptr, 0, B, H, q_len, kv_len, D, bm, score, scale, out, lse, stream);
}

fa_status fa_forward_paged(const void* q, const void* k, const void* v, const int32_t* page_table, int32_t n_pages,
                           int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                           const fa_score_spec* score, float scale, void* out, float* lse, cudaStream_t stream) {
  if (!q || !k || !v || !out || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(lse)) return FA_ERR_ALIGNMENT;
  if (page_table != nullptr) {  // fa_forward passes none
    if (!aligned4(page_table)) return FA_ERR_ALIGNMENT;
    if (n_pages < 1 || (int64_t)n_pages * 128 > (int64_t)INT32_MAX) return FA_ERR_SHAPE;
  }
  fa_status st = check_attn(B, H, q_len, kv_len, D, bm, score, &scale,
                            page_table != nullptr ? kForwardPagedOrDecode : kForward);
  if (st != FA_OK) return st;
  DevMask dm;
  st = check_mask(&bm->spec, q_len, kv_len, &dm);
  if (st != FA_OK) return st;
  AttnArgs a = attn_args(B, H, q_len, kv_len, D, bm, score, scale, dm, false);
  a.page_table = page_table;
  a.n_pages = page_table != nullptr ? n_pages : 0;
  FwdTensors t{q, k, v, out, lse};
  bool enc_failed = false;
  const cudaError_t e = launch_forward(a, t, stream, &enc_failed);
  if (enc_failed) return FA_ERR_CUDA;
  return cuda_status(e);
}

fa_status fa_forward_decode_workspace_bytes(int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                                            size_t* bytes) {
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || q_len < 1 || kv_len < 1) return FA_ERR_SHAPE;
  if (q_len > FA_DECODE_MAX_Q || (D != 64 && D != 128)) return FA_ERR_UNSUPPORTED;
  if ((int64_t)B * H > kDecodeMaxHeads) return FA_ERR_UNSUPPORTED;  // one grid row per (b, h)
  if (kv_len > (int64_t)INT32_MAX - 256) return FA_ERR_SHAPE;
  int splits = 0;
  size_t need = 0;
  if (decode_plan(B, H, q_len, kv_len, D, &splits, &need) != cudaSuccess) return FA_ERR_CUDA;
  *bytes = need;
  return FA_OK;
}

fa_status fa_forward_decode(const void* q, const void* k, const void* v, const int32_t* page_table, int32_t n_pages,
                            int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                            const fa_score_spec* score, float scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !out || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(lse) || !aligned16(workspace))
    return FA_ERR_ALIGNMENT;
  if (page_table != nullptr) {
    if (!aligned4(page_table)) return FA_ERR_ALIGNMENT;
    if (n_pages < 1 || (int64_t)n_pages * 128 > (int64_t)INT32_MAX) return FA_ERR_SHAPE;
  }
  if (q_len < 1 || q_len > FA_DECODE_MAX_Q) return q_len < 1 ? FA_ERR_SHAPE : FA_ERR_UNSUPPORTED;
  if ((int64_t)B * H > kDecodeMaxHeads) return FA_ERR_UNSUPPORTED;
  fa_status st = check_attn(B, H, q_len, kv_len, D, bm, score, &scale, kDecode);
  if (st != FA_OK) return st;
  size_t need = 0;
  int splits = 0;
  if (decode_plan(B, H, q_len, kv_len, D, &splits, &need) != cudaSuccess) return FA_ERR_CUDA;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  DevMask dm;
  st = check_mask(&bm->spec, q_len, kv_len, &dm);
  if (st != FA_OK) return st;
  AttnArgs a = attn_args(B, H, q_len, kv_len, D, bm, score, scale, dm, false);
  a.page_table = page_table;
  a.n_pages = page_table != nullptr ? n_pages : 0;
  a.kv_cap = (int32_t)bm->kv_len;  // k / v rows per (b, h): the block mask's (bucketed) length
  FwdTensors t{q, k, v, out, lse};
  bool enc_failed = false;
  const cudaError_t e = launch_decode(a, t, workspace, splits, stream, &enc_failed);
  if (enc_failed) return FA_ERR_CUDA;
  return cuda_status(e);
}

fa_status fa_forward_prepare_backward(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                                      int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                                      const fa_score_spec* score, float scale, void* out, float* lse,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !out || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(lse) || !aligned16(workspace))
    return FA_ERR_ALIGNMENT;
  fa_status st = check_attn(B, H, q_len, kv_len, D, bm, score, &scale, kForward);
  if (st != FA_OK) return st;
  size_t need = 0;
  st = fa_backward_workspace_bytes(B, H, q_len, D, &need);
  if (st != FA_OK) return st;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  DevMask dm;
  st = check_mask(&bm->spec, q_len, kv_len, &dm);
  if (st != FA_OK) return st;
  AttnArgs a = attn_args(B, H, q_len, kv_len, D, bm, score, scale, dm, false);
  a.zero_dst = static_cast<uint4*>(workspace);  // the dq accumulator: the workspace's first rows * D * 4 bytes
  a.zero_n16 = (int64_t)B * H * q_len * D * 4 / 16;
  FwdTensors t{q, k, v, out, lse};
  bool enc_failed = false;
  const cudaError_t e = launch_forward(a, t, stream, &enc_failed);
  if (enc_failed) return FA_ERR_CUDA;
  return cuda_status(e);
}

fa_status fa_backward_workspace_bytes(int32_t B, int32_t H, int64_t q_len, int32_t D, size_t* bytes) {
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || q_len < 1) return FA_ERR_SHAPE;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const size_t rows = (size_t)B * H * (size_t)q_len;
  const size_t tiles = (size_t)B * H * (size_t)((q_len + 127) / 128);
  *bytes = align_up(rows * D * 4) + align_up(tiles * 256 * 4) + align_up(4);
  return FA_OK;
}

// fa_backward and fa_backward_prepared: acc_zeroed takes the workspace's dq
// accumulator as already zero
static fa_status backward_ws(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                      const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, bool acc_zeroed, cudaStream_t stream) {
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || !aligned4(lse))
    return FA_ERR_ALIGNMENT;
  fa_status st = check_attn(B, H, q_len, kv_len, D, bm, score, &scale, kBackward);
  if (st != FA_OK) return st;
  size_t need = 0;
  st = fa_backward_workspace_bytes(B, H, q_len, D, &need);
  if (st != FA_OK) return st;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  DevMask dm;
  st = check_mask(&bm->spec, q_len, kv_len, &dm);
  if (st != FA_OK) return st;
  AttnArgs a = attn_args(B, H, q_len, kv_len, D, bm, score, scale, dm, true);
  a.acc_zeroed = acc_zeroed ? 1 : 0;
  const size_t rows = (size_t)B * H * (size_t)q_len;
  BwdTensors t;
  t.q = q;
  t.k = k;
  t.v = v;
  t.out = out;
  t.dout = dout;
  t.lse = lse;
  t.dq = dq;
  t.dk = dk;
  t.dv = dv;
  t.dq_acc = static_cast<float*>(workspace);
  t.stats = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align_up(rows * D * 4));
  t.sched = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(t.stats) +
                                        align_up((size_t)B * H * (size_t)((q_len + 127) / 128) * 256 * 4));
  bool enc_failed = false;
  const cudaError_t e = launch_backward(a, t, stream, &enc_failed);
  if (enc_failed) return FA_ERR_CUDA;
  return cuda_status(e);
}

fa_status fa_backward(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                      const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return backward_ws(q, k, v, out, lse, dout, B, H, q_len, kv_len, D, bm, score, scale, dq, dk, dv, workspace,
                     workspace_bytes, false, stream);
}

fa_status fa_backward_prepared(const void* q, const void* k, const void* v, const void* out, const float* lse,
                               const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                               const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq, void* dk,
                               void* dv, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return backward_ws(q, k, v, out, lse, dout, B, H, q_len, kv_len, D, bm, score, scale, dq, dk, dv, workspace,
                     workspace_bytes, true, stream);
}

fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                              const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                              const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq, void* dk,
                              void* dv, cudaStream_t stream) {
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned4(lse))
    return FA_ERR_ALIGNMENT;
  fa_status st = check_attn(B, H, q_len, kv_len, D, bm, score, &scale, kBackward);
  if (st != FA_OK) return st;
  size_t need = 0;
  st = fa_backward_workspace_bytes(B, H, q_len, D, &need);
  if (st != FA_OK) return st;
  if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;  // too large for the static scratch
  DevMask dm;
  st = check_mask(&bm->spec, q_len, kv_len, &dm);
  if (st != FA_OK) return st;
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return FA_ERR_CUDA;
  const AttnArgs a = attn_args(B, H, q_len, kv_len, D, bm, score, scale, dm, true);
  const size_t rows = (size_t)B * H * (size_t)q_len;
  BwdTensors t;
  t.q = q;
  t.k = k;
  t.v = v;
  t.out = out;
  t.dout = dout;
  t.lse = lse;
  t.dq = dq;
  t.dk = dk;
  t.dv = dv;
  t.dq_acc = static_cast<float*>(scratch);
  t.stats = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + align_up(rows * D * 4));
  t.sched = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(t.stats) +
                                        align_up((size_t)B * H * (size_t)((q_len + 127) / 128) * 256 * 4));
  bool enc_failed = false;
  const cudaError_t e = launch_backward(a, t, stream, &enc_failed);
  if (enc_failed) return FA_ERR_CUDA;
  return cuda_status(e);
}

fa_status fa_get_status(const fa_block_mask* bm, int32_t clear, cudaStream_t stream) {
  if (bm == nullptr || bm->status == nullptr) return FA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, bm->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (clear && word != 0 && cudaMemset(bm->status, 0, 4) != cudaSuccess) return FA_ERR_CUDA;
  if (word & kStatusTimeout) return FA_ERR_TIMEOUT;
  if (word & kStatusCheck) return FA_ERR_DEVICE_CHECK;
  return FA_OK;
}

fa_status fa_block_mask_summary(const fa_block_mask* bm, int64_t counts[3], cudaStream_t stream) {
  if (bm == nullptr || counts == nullptr || bm->tile_class == nullptr) return FA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  const size_t tiles = (size_t)bm->Bm * bm->Hm * (size_t)bm->nq * (size_t)bm->nkv;
  std::vector<uint8_t> cls(tiles);
  if (cudaMemcpy(cls.data(), bm->tile_class, tiles, cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  counts[0] = counts[1] = counts[2] = 0;
  for (uint8_t c : cls) counts[c < 3 ? c : 0] += 1;
  return FA_OK;
}

}  // extern "C"
