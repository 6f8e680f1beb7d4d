// Host side of the C ABI declared in include/flce.h: argument validation,
// workspace layout, TMA descriptor encoding and the launch sequence.  No
// allocation and no synchronisation happen here; every kernel goes on the
// caller's stream.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "flce_internal.h"

namespace flce {

int64_t ce_cta_capacity(int dtype, bool vector_path);
int64_t ce_vector_elems(int dtype, bool vector_path);

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr size_t kAlign = 256;
// Default chunk: the largest multiple of 256 tokens whose bf16 logits fit in
// 2 GiB (8192 tokens at V = 128256, 4096 at V = 256000).  Larger chunks halve
// the fp32 grad_weight read-modify-write passes and give the long grad_H
// products more tiles; the scratch stays bounded by the chunk.
constexpr int64_t kDefaultChunkBudget = int64_t(2) << 30;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- profiler
struct Profiler {
  bool enabled = false;
  int capacity = 0;
  int count = 0;
  bool open = false;
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> ids;
} g_prof;

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] with row pitch `pitch_elems`, read in
// 64 x 64 boxes with the 128-byte swizzle; out-of-range elements read as 0.
bool make_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t pitch_elems,
              CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems * 2)};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, type, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- layouts
struct FlceLayout {
  int64_t chunk, num_chunks, vp, nvt;  // nvt: 256-column vocabulary tiles
  int64_t npart;                       // per-row LSE partials: one per part_cols(forward_epi_warps) columns
  int gh_slices;  // most K slices of a split grad_H (1: never split)
  size_t header, zbuf, partials, tgt_logit, row_lse, row_scale, row_tgt, loss_rows, gh_part, total;
  size_t cvt_h, cvt_w, cvt_b;  // fp32 operands: their bf16 copies (0 bytes otherwise)
  int64_t z_plane;             // split fp32 operands: elements between the two chunk-logit planes (else 0)
};

// grad_H tiles (256 x 512, K = V) fewer than the SM pairs leave pairs idle
// for the longest products of the backward launch: their K range is then
// split into slices, as many as fill the pairs, each at least 8 k blocks
// (512 of the vocabulary) long.
constexpr int kGemmMaxPairs = 128;  // sizes the partial-sum buffer for any GPU up to 256 SMs
int gh_slices(int64_t rows, int64_t H, int64_t V, int pairs) {
  const int64_t base = ceil_div(rows, 2 * kBM) * ceil_div(H, 2 * kBN);
  if (base <= 0 || base >= pairs) return 1;
  const int64_t most = std::max<int64_t>(1, ceil_div(V, kBK) / 8);
  return static_cast<int>(std::min<int64_t>(ceil_div(pairs, base), most));
}

int64_t default_chunk(int64_t N, int64_t V) {
  int64_t c = kDefaultChunkBudget / (V * 2);
  c = c / 256 * 256;
  if (c < 256) c = 256;
  if (c > 16384) c = 16384;
  if (N > 0 && c > N) c = N;
  return c;
}

bool flce_layout(int64_t N, int64_t H, int64_t V, int64_t chunk, int reduction, FlceLayout* L,
                 int dtype = FLCE_DTYPE_BF16) {
  if (N < 0 || H < 8 || V < 1 || chunk < 0 || reduction < 0 || reduction > 2) return false;
  if (N >= (int64_t(1) << 31) || V >= (int64_t(1) << 31) || H >= (int64_t(1) << 24)) return false;
  L->chunk = chunk == 0 ? default_chunk(N, V) : chunk;
  if (N > 0 && L->chunk > N) L->chunk = N;
  if (L->chunk < 1) L->chunk = 1;
  L->num_chunks = N > 0 ? ceil_div(N, L->chunk) : 0;
  L->vp = round_up(static_cast<size_t>(V), 8);
  L->nvt = ceil_div(V, kBN);
  size_t off = 0;
  L->header = off;
  off = round_up(off + sizeof(WorkspaceHeader) + sizeof(unsigned int) * 2 * (L->num_chunks + 1), kAlign);
  // split fp32 operands (FLCE_DTYPE_FP32): the chunk logits as two planes of
  // 16-bit halves, and hi + lo bf16 planes of hidden and weight; the bias is
  // read in fp32.  Rounded fp32 operands: one bf16 copy of each.
  const bool split = dtype == FLCE_DTYPE_FP32;
  const bool rounded = dtype == FLCE_DTYPE_FP32_ROUNDED;
  const size_t planes = split ? 2 : 1;
  // LSE partials per row: one per column range of a forward epilogue warp
  L->npart = ceil_div(V, part_cols(forward_epi_warps(H, split ? 3 : 1)));
  L->zbuf = off;
  L->z_plane = split ? L->chunk * static_cast<int64_t>(L->vp) : 0;
  off = round_up(off + planes * static_cast<size_t>(L->chunk) * L->vp * 2, kAlign);
  L->partials = off;
  // the per-tile partials of the forward epilogue; after row_finalize the same
  // bytes take the grad-logits pass's per-row-block bias column sums
  off = round_up(off + std::max(static_cast<size_t>(L->chunk) * L->npart * sizeof(float4),
                                static_cast<size_t>(ceil_div(L->chunk, kGlBiasRows)) * L->vp * sizeof(float)),
                 kAlign);
  L->tgt_logit = off;
  off = round_up(off + static_cast<size_t>(L->chunk) * 4, kAlign);
  L->row_lse = off;
  off = round_up(off + static_cast<size_t>(L->chunk) * 4, kAlign);
  L->row_scale = off;
  off = round_up(off + static_cast<size_t>(L->chunk) * 4, kAlign);
  L->row_tgt = off;
  off = round_up(off + static_cast<size_t>(L->chunk) * 4, kAlign);
  L->loss_rows = off;
  off = round_up(off + (reduction == FLCE_REDUCTION_NONE ? 0 : static_cast<size_t>(N) * 4), kAlign);
  L->gh_slices = gh_slices(L->chunk, H, V, kGemmMaxPairs);
  L->gh_part = off;
  off = round_up(off + (L->gh_slices > 1 ? static_cast<size_t>(L->gh_slices) * L->chunk * H * 4 : 0), kAlign);
  const size_t copies = split ? 2 : (rounded ? 1 : 0);
  L->cvt_h = off;
  off = round_up(off + copies * static_cast<size_t>(N) * H * 2, kAlign);
  L->cvt_w = off;
  off = round_up(off + copies * static_cast<size_t>(V) * H * 2, kAlign);
  L->cvt_b = off;
  off = round_up(off + (rounded ? static_cast<size_t>(L->vp) * 2 : 0), kAlign);
  L->total = off;
  return true;
}

struct CeLayout {
  size_t header, loss_rows, flags, total;
};

bool ce_layout(int64_t N, int64_t V, int dtype, int reduction, CeLayout* L) {
  if (N < 0 || V < 1 || (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP32 && dtype != FLCE_DTYPE_FP16) ||
      reduction < 0 || reduction > 2)
    return false;
  L->header = 0;
  L->loss_rows = round_up(sizeof(WorkspaceHeader) + 16, kAlign);
  L->flags = round_up(L->loss_rows + static_cast<size_t>(N) * 4, kAlign);
  L->total = round_up(L->flags + sizeof(unsigned long long), kAlign);  // the tagged arrival counter
  return true;
}

// A 40-bit value no recent call of this process used: the single-launch CE
// form tags its arrival counter with it (the word it finds in the workspace
// is some earlier call's, or whatever the memory held).
unsigned long long next_ce_nonce() {
  static std::atomic<unsigned long long> counter{
      0x9E3779B97F4A7C15ull ^
      static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count())};
  return (counter.fetch_add(1, std::memory_order_relaxed) + 1) & ((1ull << 40) - 1);
}

#define FLCE_TRY_CUDA(expr)                  \
  do {                                       \
    if ((expr) != cudaSuccess) return FLCE_ERR_CUDA; \
  } while (0)

}  // namespace

void prof_begin(cudaStream_t s, int kernel_id) {
  if (!g_prof.enabled || g_prof.count >= g_prof.capacity) return;
  cudaEventRecord(g_prof.start[g_prof.count], s);
  g_prof.ids[g_prof.count] = kernel_id;
  g_prof.open = true;
}

void prof_end(cudaStream_t s) {
  if (!g_prof.enabled || !g_prof.open) return;
  cudaEventRecord(g_prof.stop[g_prof.count], s);
  g_prof.count++;
  g_prof.open = false;
}

}  // namespace flce

using namespace flce;

extern "C" {

const char* flce_status_string(flce_status_t s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG: bad argument (null pointer, size or enum)";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED: unsupported dtype or shape";
    case FLCE_ERR_WORKSPACE: return "FLCE_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA: a CUDA call or kernel launch failed";
    case FLCE_ERR_TARGET_RANGE: return "FLCE_ERR_TARGET_RANGE: a target outside [0, V) that is not ignore_index";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT: a pipeline wait exceeded its time limit";
    case FLCE_ERR_MISALIGNED: return "FLCE_ERR_MISALIGNED: a pointer breaks its alignment requirement";
  }
  return "FLCE_UNKNOWN_STATUS";
}

int flce_version(void) { return kVersion; }

int64_t flce_default_chunk(int64_t N, int64_t H, int64_t V) {
  (void)H;
  if (V < 1) return 0;
  return default_chunk(N, V);
}

size_t flce_workspace_size(int64_t N, int64_t H, int64_t V, int64_t chunk, int reduction) {
  FlceLayout L;
  if (!flce_layout(N, H, V, chunk, reduction, &L)) return 0;
  return L.total;
}

size_t flce_workspace_size_typed(int dtype, int64_t N, int64_t H, int64_t V, int64_t chunk, int reduction) {
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP16 && dtype != FLCE_DTYPE_FP32 &&
      dtype != FLCE_DTYPE_FP32_ROUNDED)
    return 0;
  FlceLayout L;
  if (!flce_layout(N, H, V, chunk, reduction, &L, dtype)) return 0;
  return L.total;
}

flce_status_t flce_fwd_bwd(const void* hidden, const void* weight, const void* bias, const int64_t* target,
                           int64_t N, int64_t H, int64_t V, int64_t ignore_index, int reduction,
                           int64_t chunk, float grad_scale, const float* grad_out_none, float* loss,
                           void* grad_hidden, float* grad_weight, float* grad_bias, int accumulate,
                           int32_t* n_valid_out, float* lse_out, float* target_logit_out, void* workspace,
                           size_t workspace_bytes, int32_t* status_dev, flce_stream_t stream) {
  return flce_fwd_bwd_typed(FLCE_DTYPE_BF16, hidden, weight, bias, target, N, H, V, ignore_index, reduction, chunk,
                            grad_scale, grad_out_none, loss, grad_hidden, grad_weight, grad_bias, accumulate,
                            n_valid_out, lse_out, target_logit_out, workspace, workspace_bytes, status_dev, stream);
}

flce_status_t flce_fwd_bwd_typed(int dtype, const void* hidden, const void* weight, const void* bias,
                                 const int64_t* target, int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                                 int reduction, int64_t chunk, float grad_scale, const float* grad_out_none,
                                 float* loss, void* grad_hidden, float* grad_weight, float* grad_bias,
                                 int accumulate, int32_t* n_valid_out, float* lse_out, float* target_logit_out,
                                 void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                 flce_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  FlceLayout L;
  if (N < 0 || V < 1 || H < 1 || chunk < 0 || reduction < 0 || reduction > 2) return FLCE_ERR_INVALID_ARG;
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP16 && dtype != FLCE_DTYPE_FP32 &&
      dtype != FLCE_DTYPE_FP32_ROUNDED)
    return FLCE_ERR_UNSUPPORTED;
  const bool fp16 = dtype == FLCE_DTYPE_FP16;
  const bool split = dtype == FLCE_DTYPE_FP32;            // hi + lo bf16 planes, three products
  const bool rounded = dtype == FLCE_DTYPE_FP32_ROUNDED;  // one bf16 rounding
  const bool fp32 = split || rounded;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!flce_layout(N, H, V, chunk, reduction, &L, dtype)) return FLCE_ERR_INVALID_ARG;
  if (loss == nullptr || weight == nullptr) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (hidden == nullptr || target == nullptr)) return FLCE_ERR_INVALID_ARG;
  if (grad_bias != nullptr && bias == nullptr) return FLCE_ERR_INVALID_ARG;
  if (grad_out_none != nullptr && reduction != FLCE_REDUCTION_NONE) return FLCE_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return FLCE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(bias, 16) || !aligned(grad_hidden, 16) ||
      !aligned(grad_weight, 16) || !aligned(target, 8) || !aligned(loss, 4) || !aligned(grad_bias, 4))
    return FLCE_ERR_MISALIGNED;
  if (workspace == nullptr || !aligned(workspace, kAlign) || workspace_bytes < L.total) return FLCE_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  int* status = status_dev != nullptr ? status_dev : &hdr->status;
  uint16_t* zbuf = reinterpret_cast<uint16_t*>(ws + L.zbuf);
  float4* partials = reinterpret_cast<float4*>(ws + L.partials);
  float* tgt_logit = reinterpret_cast<float*>(ws + L.tgt_logit);
  float* row_lse = reinterpret_cast<float*>(ws + L.row_lse);
  float* row_scale = reinterpret_cast<float*>(ws + L.row_scale);
  int* row_tgt = reinterpret_cast<int*>(ws + L.row_tgt);
  float* loss_rows = reduction == FLCE_REDUCTION_NONE ? loss : reinterpret_cast<float*>(ws + L.loss_rows);
  const uint64_t timeout = g_timeout_ns.load();

  const size_t hdr_bytes = sizeof(WorkspaceHeader) + sizeof(unsigned int) * 2 * (L.num_chunks + 1);
  FLCE_TRY_CUDA(cudaMemsetAsync(hdr, 0, hdr_bytes, stream));
  FLCE_TRY_CUDA(launch_count_targets(target, N, V, ignore_index, hdr, 0, 0, status, n_valid_out,
                                     (grad_bias != nullptr && !accumulate) ? grad_bias : nullptr,
                                     (grad_bias != nullptr && !accumulate) ? V : 0, grad_out_none, stream));
  if (N == 0) {
    if (grad_weight != nullptr && !accumulate) FLCE_TRY_CUDA(launch_zero(grad_weight, V * H, stream));
    if (reduction != FLCE_REDUCTION_NONE)
      FLCE_TRY_CUDA(launch_loss_reduce(loss_rows, 0, reduction, &hdr->n_valid, loss, stream, false));
    return FLCE_OK;
  }

  CUtensorMap tm_h2, tm_w2, tm_z2;  // split: the lo planes
  if (split) {
    // fp32 operands split into bf16 hi + lo planes once per call; the
    // products are hi.hi + hi.lo + lo.hi (grad_hidden written in fp32)
    uint16_t* h_hi = reinterpret_cast<uint16_t*>(ws + L.cvt_h);
    uint16_t* h_lo = h_hi + N * H;
    uint16_t* w_hi = reinterpret_cast<uint16_t*>(ws + L.cvt_w);
    uint16_t* w_lo = w_hi + V * H;
    FLCE_TRY_CUDA(launch_f32_split_bf16(static_cast<const float*>(hidden), h_hi, h_lo, N * H, stream));
    FLCE_TRY_CUDA(launch_f32_split_bf16(static_cast<const float*>(weight), w_hi, w_lo, V * H, stream));
    if (!make_map(&tm_h2, h_lo, H, N, H) || !make_map(&tm_w2, w_lo, H, V, H)) return FLCE_ERR_CUDA;
    hidden = h_hi;
    weight = w_hi;
  } else if (rounded) {
    // fp32 operands: the tensor cores take their bf16 roundings, copied once
    // per call into the workspace (grad_hidden is still written in fp32)
    uint16_t* h16 = reinterpret_cast<uint16_t*>(ws + L.cvt_h);
    uint16_t* w16 = reinterpret_cast<uint16_t*>(ws + L.cvt_w);
    FLCE_TRY_CUDA(launch_f32_to_bf16(static_cast<const float*>(hidden), h16, N * H, stream));
    FLCE_TRY_CUDA(launch_f32_to_bf16(static_cast<const float*>(weight), w16, V * H, stream));
    hidden = h16;
    weight = w16;
    if (bias != nullptr) {
      uint16_t* b16 = reinterpret_cast<uint16_t*>(ws + L.cvt_b);
      FLCE_TRY_CUDA(launch_f32_to_bf16(static_cast<const float*>(bias), b16, V, stream));
      bias = b16;
    }
  }

  CUtensorMap tm_h, tm_w, tm_z;
  const CUtensorMapDataType mtype = fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&tm_h, hidden, H, N, H, mtype) || !make_map(&tm_w, weight, H, V, H, mtype)) return FLCE_ERR_CUDA;
  const int sms = device_sm_count();
  const float* gmax = (reduction == FLCE_REDUCTION_NONE && grad_out_none != nullptr) ? &hdr->gmax : nullptr;
  const bool want_grads = grad_hidden != nullptr || grad_weight != nullptr || grad_bias != nullptr;

  for (int64_t k = 0; k < L.num_chunks; ++k) {
    const int64_t row0 = k * L.chunk;
    const int c_len = static_cast<int>(std::min<int64_t>(L.chunk, N - row0));
    if (!make_map(&tm_z, zbuf, V, c_len, L.vp, mtype)) return FLCE_ERR_CUDA;
    if (split && !make_map(&tm_z2, zbuf + L.z_plane, V, c_len, L.vp)) return FLCE_ERR_CUDA;

    GemmParams g = {};
    g.row0 = row0;
    g.c_len = c_len;
    g.H = static_cast<int>(H);
    g.V = static_cast<int>(V);
    g.f_num_m = static_cast<int>(ceil_div(c_len, kBM));
    g.f_kblocks = static_cast<int>(ceil_div(H, kBK));
    g.bias = split ? nullptr : static_cast<const uint16_t*>(bias);
    g.bias_f32 = split ? static_cast<const float*>(bias) : nullptr;
    g.nseg = split ? 3 : 1;
    g.z_plane = L.z_plane;
    g.target = target;
    g.zbuf = zbuf;
    g.ldz = L.vp;
    g.partials = partials;
    g.epi_warps = forward_epi_warps(H, g.nseg);
    g.nvt = static_cast<int>(L.npart);  // the layout sized them for this warp count
    g.tgt_logit = tgt_logit;
    g.grad_hidden = fp32 ? nullptr : static_cast<uint16_t*>(grad_hidden);
    g.grad_hidden_f32 = fp32 ? static_cast<float*>(grad_hidden) : nullptr;
    g.grad_weight = grad_weight;
    g.gw_store = (k == 0 && !accumulate) ? 1 : 0;
    g.status = status;
    g.timeout_ns = timeout;
    g.in_fp16 = fp16 ? 1 : 0;
    g.n_valid = &hdr->n_valid;
    g.gmax = gmax;
    g.reduction = reduction;
    g.grad_scale = grad_scale;

    const int tile_m = 2 * kBM;  // CTA-pair tiles: 256 rows
    g.f_num_m = static_cast<int>(ceil_div(c_len, tile_m));
    g.num_tiles = static_cast<int>(g.f_num_m * L.nvt);
    g.tile_counter = &hdr->tile_counters[2 * k];
    FLCE_TRY_CUDA(launch_gemm2(kModeForward, tm_h, tm_w, tm_z, g, 2 * std::min(sms / 2, g.num_tiles), stream,
                               split ? &tm_h2 : nullptr, split ? &tm_w2 : nullptr, split ? &tm_z2 : nullptr));

    RowParams r = {};
    r.row0 = row0;
    r.c_len = c_len;
    r.N = N;
    r.V = V;
    r.ignore_index = ignore_index;
    r.reduction = reduction;
    r.grad_scale = grad_scale;
    r.grad_out = grad_out_none;
    r.target = target;
    r.partials = partials;
    r.nvt = g.nvt;
    r.tgt_logit = tgt_logit;
    r.n_valid = &hdr->n_valid;
    r.row_lse = row_lse;
    r.row_scale = row_scale;
    r.row_tgt = row_tgt;
    r.loss_rows = loss_rows;
    r.lse_out = lse_out;
    r.tl_out = target_logit_out;
    r.status = status;
    r.zbuf = zbuf;
    r.ldz = L.vp;
    r.grad_bias = grad_bias;
    r.bias_part = reinterpret_cast<float*>(ws + L.partials);
    r.z_fp16 = fp16 ? 1 : 0;
    r.z_plane = L.z_plane;
    r.gmax = gmax;
    FLCE_TRY_CUDA(launch_row_finalize(r, stream));
    if (!want_grads) continue;
    FLCE_TRY_CUDA(launch_grad_logits(r, stream));

    g.h_num_m = static_cast<int>(ceil_div(c_len, tile_m));
    g.h_kblocks = static_cast<int>(ceil_div(V, kBK));
    // grad_H in 256 x 512 tiles, split along K when they are too few
    g.h_base = grad_hidden != nullptr ? static_cast<int>(g.h_num_m * ceil_div(H, 2 * kBN)) : 0;
    g.h_split = g.h_base > 0 ? std::min(gh_slices(c_len, H, V, sms / 2), L.gh_slices) : 1;
    g.h_kbs = static_cast<int>(ceil_div(g.h_kblocks, g.h_split));
    g.h_split = static_cast<int>(ceil_div(g.h_kblocks, g.h_kbs));  // no empty slice
    g.h_tiles = g.h_base * g.h_split;
    g.gh_part = g.h_split > 1 ? reinterpret_cast<float*>(ws + L.gh_part) : nullptr;
    g.gh_part_ld = L.chunk * H;
    g.w_num_n = static_cast<int>(ceil_div(H, kBN));
    g.w_kblocks = static_cast<int>(ceil_div(c_len, kBK));
    const int w_tiles = grad_weight != nullptr ? static_cast<int>(ceil_div(V, tile_m) * g.w_num_n) : 0;
    g.num_tiles = g.h_tiles + w_tiles;
    g.tile_counter = &hdr->tile_counters[2 * k + 1];
    if (g.num_tiles > 0)
      FLCE_TRY_CUDA(launch_gemm2(kModeBackward, tm_h, tm_w, tm_z, g, 2 * std::min(sms / 2, g.num_tiles), stream,
                                 split ? &tm_h2 : nullptr, split ? &tm_w2 : nullptr, split ? &tm_z2 : nullptr));
    if (g.h_tiles > 0 && g.h_split > 1)
      FLCE_TRY_CUDA(launch_gh_reduce(g.gh_part, g.h_split, g.gh_part_ld, c_len, static_cast<int>(H), row0,
                                     fp32 ? nullptr : static_cast<uint16_t*>(grad_hidden), fp16 ? 1 : 0,
                                     fp32 ? static_cast<float*>(grad_hidden) : nullptr, stream));
  }
  if (reduction != FLCE_REDUCTION_NONE)
    FLCE_TRY_CUDA(launch_loss_reduce(loss_rows, N, reduction, &hdr->n_valid, loss, stream, false));
  return FLCE_OK;
}

size_t ce_workspace_size(int64_t N, int64_t V, int dtype, int reduction) {
  CeLayout L;
  if (!ce_layout(N, V, dtype, reduction, &L)) return 0;
  return L.total;
}

flce_status_t ce_fwd_bwd(const void* logits, int dtype, void* grad_logits, const int64_t* target, int64_t N,
                         int64_t V, int64_t ignore_index, int reduction, float grad_scale,
                         const float* grad_out_none, float* loss, void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, flce_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP32 && dtype != FLCE_DTYPE_FP16) return FLCE_ERR_UNSUPPORTED;
  CeLayout L;
  if (!ce_layout(N, V, dtype, reduction, &L)) return FLCE_ERR_INVALID_ARG;
  if (loss == nullptr || (N > 0 && (logits == nullptr || target == nullptr))) return FLCE_ERR_INVALID_ARG;
  if (grad_out_none != nullptr && reduction != FLCE_REDUCTION_NONE) return FLCE_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 31) / 8) return FLCE_ERR_UNSUPPORTED;
  const size_t esz = dtype == FLCE_DTYPE_FP32 ? 4 : 2;
  if (!aligned(logits, esz) || !aligned(grad_logits, esz) || !aligned(target, 8) || !aligned(loss, 4))
    return FLCE_ERR_MISALIGNED;
  if (grad_logits != nullptr && grad_logits != logits) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(grad_logits);
    const uintptr_t bytes = static_cast<uintptr_t>(N) * V * esz;
    if (a < b + bytes && b < a + bytes) return FLCE_ERR_INVALID_ARG;  // partial overlap
  }
  if (workspace == nullptr || !aligned(workspace, kAlign) || workspace_bytes < L.total) return FLCE_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  int* status = status_dev != nullptr ? status_dev : &hdr->status;
  float* loss_rows = reduction == FLCE_REDUCTION_NONE ? loss : reinterpret_cast<float*>(ws + L.loss_rows);

  const bool ptrs16 = aligned(logits, 16) && (grad_logits == nullptr || aligned(grad_logits, 16));
  const bool vec = (static_cast<size_t>(V) * esz) % 16 == 0 && ptrs16;
  if (N > 0 && N <= kCeSelfCountMaxRows && ce_rows_single_launch_ok(V, dtype, vec, ptrs16)) {
    // one launch: the row kernel counts the targets itself and finds the CTA
    // that adds the loss partials by flags, so nothing needs zeroing first
    CeParams p = {};
    p.logits = logits;
    p.grad = grad_logits;
    p.target = target;
    p.N = N;
    p.V = V;
    p.ignore_index = ignore_index;
    p.reduction = reduction;
    p.grad_scale = grad_scale;
    p.grad_out = grad_out_none;
    p.loss_rows = loss_rows;
    // the status word: the caller's, or the workspace's own, which CTA 0
    // clears when it starts (the other CTAs only write it after a 2 s wait)
    p.status = status;
    p.clear_status = status_dev == nullptr ? 1 : 0;
    p.cluster = 1;
    p.seg_len = V;
    p.loss_out = reduction != FLCE_REDUCTION_NONE ? loss : nullptr;
    p.self_count = 1;
    p.done_flags = reinterpret_cast<unsigned long long*>(ws + L.flags);
    p.nonce = next_ce_nonce();
    FLCE_TRY_CUDA(launch_ce_rows(p, dtype, vec, ptrs16, false, stream));
    return FLCE_OK;
  }
  if (N <= kCountSingleBlockMax) {
    // one block zeroes the header and counts; the CE kernel overlaps it (PDL)
    FLCE_TRY_CUDA(launch_count_targets(target, N, V, ignore_index, hdr, 0, 1, status, nullptr, nullptr, 0, nullptr, stream));
  } else {
    FLCE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WorkspaceHeader) + 16, stream));
    FLCE_TRY_CUDA(launch_count_targets(target, N, V, ignore_index, hdr, 0, 0, status, nullptr, nullptr, 0, nullptr, stream));
  }
  if (N > 0) {
    const int64_t cap = ce_cta_capacity(dtype, vec);
    const int64_t epv = ce_vector_elems(dtype, vec);
    int64_t cl = ceil_div(V, cap);
    if (cl > 8) cl = 8;
    if (cl < 1) cl = 1;
    int64_t seg = ceil_div(V, cl);
    seg = ceil_div(seg, epv) * epv;
    cl = ceil_div(V, seg);
    CeParams p = {};
    p.logits = logits;
    p.grad = grad_logits;
    p.target = target;
    p.N = N;
    p.V = V;
    p.ignore_index = ignore_index;
    p.reduction = reduction;
    p.grad_scale = grad_scale;
    p.grad_out = grad_out_none;
    p.loss_rows = loss_rows;
    p.n_valid = &hdr->n_valid;
    p.status = status;
    p.cluster = static_cast<int>(cl);
    p.seg_len = seg;
    p.loss_out = reduction != FLCE_REDUCTION_NONE ? loss : nullptr;  // fused final reduction
    p.ticket = reinterpret_cast<unsigned int*>(&hdr->pad[1]);
    FLCE_TRY_CUDA(launch_ce_rows(p, dtype, vec, ptrs16, true, stream));
  } else if (reduction != FLCE_REDUCTION_NONE) {
    FLCE_TRY_CUDA(launch_loss_reduce(loss_rows, 0, reduction, &hdr->n_valid, loss, stream, false));
  }
  return FLCE_OK;
}

// ------------------------------------------------------------ vocabulary shards

size_t flce_vp_workspace_size(int64_t C, int64_t H, int64_t V_shard) {
  if (C < 1 || H < 8 || V_shard < 1 || C >= (int64_t(1) << 31) || V_shard >= (int64_t(1) << 31)) return 0;
  FlceLayout L;
  if (!flce_layout(C, H, V_shard, C, FLCE_REDUCTION_NONE, &L)) return 0;
  return L.total;
}

flce_status_t flce_vp_forward(const void* hidden, const void* weight_shard, const void* bias_shard,
                              const int64_t* target, int64_t C, int64_t H, int64_t V_shard, int64_t vocab_offset,
                              int64_t ignore_index, float* lse_shard, float* lse16_shard,
                              float* target_logit_shard, void* workspace, size_t workspace_bytes,
                              int32_t* status_dev, flce_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (C < 1 || V_shard < 1 || H < 8 || vocab_offset < 0) return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  FlceLayout L;
  if (!flce_layout(C, H, V_shard, C, FLCE_REDUCTION_NONE, &L)) return FLCE_ERR_INVALID_ARG;
  if (hidden == nullptr || weight_shard == nullptr || target == nullptr || lse_shard == nullptr ||
      lse16_shard == nullptr || target_logit_shard == nullptr)
    return FLCE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(weight_shard, 16) || !aligned(bias_shard, 16) || !aligned(target, 8))
    return FLCE_ERR_MISALIGNED;
  if (workspace == nullptr || !aligned(workspace, kAlign) || workspace_bytes < L.total) return FLCE_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  int* status = status_dev != nullptr ? status_dev : &hdr->status;
  FLCE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WorkspaceHeader) + 4 * sizeof(unsigned int), stream));
  CUtensorMap tm_h, tm_w, tm_z;
  if (!make_map(&tm_h, hidden, H, C, H) || !make_map(&tm_w, weight_shard, H, V_shard, H) ||
      !make_map(&tm_z, ws + L.zbuf, V_shard, C, L.vp))
    return FLCE_ERR_CUDA;
  const int tile_m = 2 * kBM;
  GemmParams g = {};
  g.row0 = 0;
  g.c_len = static_cast<int>(C);
  g.H = static_cast<int>(H);
  g.V = static_cast<int>(V_shard);
  g.f_num_m = static_cast<int>(ceil_div(C, tile_m));
  g.f_kblocks = static_cast<int>(ceil_div(H, kBK));
  g.bias = static_cast<const uint16_t*>(bias_shard);
  g.target = target;
  g.v_offset = vocab_offset;
  g.zbuf = reinterpret_cast<uint16_t*>(ws + L.zbuf);
  g.ldz = L.vp;
  g.partials = reinterpret_cast<float4*>(ws + L.partials);
  g.epi_warps = forward_epi_warps(H, 1);
  g.nvt = static_cast<int>(L.npart);
  g.tgt_logit = reinterpret_cast<float*>(ws + L.tgt_logit);
  g.status = status;
  g.timeout_ns = g_timeout_ns.load();
  g.num_tiles = static_cast<int>(g.f_num_m * L.nvt);
  g.tile_counter = &hdr->tile_counters[0];
  const int sms = device_sm_count();
  FLCE_TRY_CUDA(launch_gemm2(kModeForward, tm_h, tm_w, tm_z, g, 2 * std::min(sms / 2, g.num_tiles), stream));
  RowParams r = {};
  r.row0 = 0;
  r.c_len = static_cast<int>(C);
  r.N = C;
  r.V = V_shard;
  r.ignore_index = ignore_index;
  r.target = target;
  r.partials = g.partials;
  r.nvt = g.nvt;
  r.tgt_logit = g.tgt_logit;
  r.v_offset = vocab_offset;
  r.status = status;
  FLCE_TRY_CUDA(launch_vp_finalize(r, lse_shard, lse16_shard, target_logit_shard, stream));
  return FLCE_OK;
}

flce_status_t flce_vp_backward(const void* hidden, const void* weight_shard, const int64_t* target, int64_t C,
                               int64_t H, int64_t V_shard, int64_t vocab_offset, int64_t ignore_index,
                               const float* lse16, const float* row_scale, float* grad_hidden_partial,
                               float* grad_weight_shard, float* grad_bias_shard, int accumulate, void* workspace,
                               size_t workspace_bytes, int32_t* status_dev, flce_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (C < 1 || V_shard < 1 || H < 8 || vocab_offset < 0 || (accumulate != 0 && accumulate != 1))
    return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  FlceLayout L;
  if (!flce_layout(C, H, V_shard, C, FLCE_REDUCTION_NONE, &L)) return FLCE_ERR_INVALID_ARG;
  if (hidden == nullptr || weight_shard == nullptr || target == nullptr || lse16 == nullptr || row_scale == nullptr)
    return FLCE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(weight_shard, 16) || !aligned(target, 8) ||
      !aligned(grad_hidden_partial, 16) || !aligned(grad_weight_shard, 16) || !aligned(grad_bias_shard, 4))
    return FLCE_ERR_MISALIGNED;
  if (workspace == nullptr || !aligned(workspace, kAlign) || workspace_bytes < L.total) return FLCE_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  int* status = status_dev != nullptr ? status_dev : &hdr->status;
  FLCE_TRY_CUDA(cudaMemsetAsync(&hdr->tile_counters[1], 0, sizeof(unsigned int), stream));
  if (grad_bias_shard != nullptr && !accumulate) FLCE_TRY_CUDA(launch_zero(grad_bias_shard, V_shard, stream));
  RowParams r = {};
  r.row0 = 0;
  r.c_len = static_cast<int>(C);
  r.N = C;
  r.V = V_shard;
  r.ignore_index = ignore_index;
  r.target = target;
  r.row_lse = const_cast<float*>(lse16);
  r.row_scale = const_cast<float*>(row_scale);
  r.row_tgt = nullptr;
  r.v_offset = vocab_offset;
  r.status = status;
  r.zbuf = reinterpret_cast<uint16_t*>(ws + L.zbuf);
  r.ldz = L.vp;
  r.grad_bias = grad_bias_shard;
  r.bias_part = reinterpret_cast<float*>(ws + L.partials);
  FLCE_TRY_CUDA(launch_grad_logits(r, stream));
  if (grad_hidden_partial == nullptr && grad_weight_shard == nullptr) return FLCE_OK;
  CUtensorMap tm_h, tm_w, tm_z;
  if (!make_map(&tm_h, hidden, H, C, H) || !make_map(&tm_w, weight_shard, H, V_shard, H) ||
      !make_map(&tm_z, ws + L.zbuf, V_shard, C, L.vp))
    return FLCE_ERR_CUDA;
  const int tile_m = 2 * kBM;
  GemmParams g = {};
  g.row0 = 0;
  g.c_len = static_cast<int>(C);
  g.H = static_cast<int>(H);
  g.V = static_cast<int>(V_shard);
  g.target = target;
  g.v_offset = vocab_offset;
  g.zbuf = r.zbuf;
  g.ldz = L.vp;
  g.grad_hidden_f32 = grad_hidden_partial;
  g.grad_weight = grad_weight_shard;
  g.gw_store = accumulate ? 0 : 1;
  g.status = status;
  g.timeout_ns = g_timeout_ns.load();
  g.h_num_m = static_cast<int>(ceil_div(C, tile_m));
  g.h_kblocks = static_cast<int>(ceil_div(V_shard, kBK));
  const int sms = device_sm_count();
  g.h_base = grad_hidden_partial != nullptr ? static_cast<int>(g.h_num_m * ceil_div(H, 2 * kBN)) : 0;
  g.h_split = g.h_base > 0 ? std::min(gh_slices(C, H, V_shard, sms / 2), L.gh_slices) : 1;
  g.h_kbs = static_cast<int>(ceil_div(g.h_kblocks, g.h_split));
  g.h_split = static_cast<int>(ceil_div(g.h_kblocks, g.h_kbs));
  g.h_tiles = g.h_base * g.h_split;
  g.gh_part = g.h_split > 1 ? reinterpret_cast<float*>(ws + L.gh_part) : nullptr;
  g.gh_part_ld = L.chunk * H;
  g.w_num_n = static_cast<int>(ceil_div(H, kBN));
  g.w_kblocks = static_cast<int>(ceil_div(C, kBK));
  const int w_tiles = grad_weight_shard != nullptr ? static_cast<int>(ceil_div(V_shard, tile_m) * g.w_num_n) : 0;
  g.num_tiles = g.h_tiles + w_tiles;
  g.tile_counter = &hdr->tile_counters[1];
  FLCE_TRY_CUDA(launch_gemm2(kModeBackward, tm_h, tm_w, tm_z, g, 2 * std::min(sms / 2, g.num_tiles), stream));
  if (g.h_tiles > 0 && g.h_split > 1)
    FLCE_TRY_CUDA(launch_gh_reduce(g.gh_part, g.h_split, g.gh_part_ld, static_cast<int>(C), static_cast<int>(H), 0,
                                   nullptr, 0, grad_hidden_partial, stream));
  return FLCE_OK;
}

flce_status_t ce_vp_partials(const void* logits, int dtype, const int64_t* target, int64_t N, int64_t V_shard,
                             int64_t vocab_offset, int64_t ignore_index, float* lse_shard, float* target_logit_shard,
                             int32_t* status_dev, flce_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP32 && dtype != FLCE_DTYPE_FP16) return FLCE_ERR_UNSUPPORTED;
  if (N < 0 || V_shard < 1 || vocab_offset < 0) return FLCE_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 31) / 8) return FLCE_ERR_UNSUPPORTED;
  if (N > 0 && (logits == nullptr || target == nullptr || lse_shard == nullptr || target_logit_shard == nullptr))
    return FLCE_ERR_INVALID_ARG;
  const size_t esz = dtype == FLCE_DTYPE_FP32 ? 4 : 2;
  if (!aligned(logits, esz) || !aligned(target, 8) || !aligned(lse_shard, 4) || !aligned(target_logit_shard, 4))
    return FLCE_ERR_MISALIGNED;
  if (N == 0) return FLCE_OK;
  const bool ptrs16 = aligned(logits, 16);
  const bool vec = (static_cast<size_t>(V_shard) * esz) % 16 == 0 && ptrs16;
  if (vp_partials_rows_fits(dtype, V_shard, vec)) {
    FLCE_TRY_CUDA(launch_vp_partials_rows(logits, dtype, target, N, V_shard, vocab_offset, ignore_index, lse_shard,
                                          target_logit_shard, stream));
    return FLCE_OK;
  }
  const int64_t cap = ce_cta_capacity(dtype, vec);
  const int64_t epv = ce_vector_elems(dtype, vec);
  int64_t cl = ceil_div(V_shard, cap);
  cl = cl > 8 ? 8 : (cl < 1 ? 1 : cl);
  int64_t seg = ceil_div(ceil_div(V_shard, cl), epv) * epv;
  cl = ceil_div(V_shard, seg);
  CeParams p = {};
  p.logits = logits;
  p.grad = nullptr;
  p.target = target;
  p.N = N;
  p.V = V_shard;
  p.ignore_index = ignore_index;
  p.reduction = FLCE_REDUCTION_SUM;  // no scale is formed in this mode
  p.grad_scale = 1.f;
  p.status = status_dev;
  p.cluster = static_cast<int>(cl);
  p.seg_len = seg;
  p.lse_out = lse_shard;
  p.zt_out = target_logit_shard;
  p.v_offset = vocab_offset;
  FLCE_TRY_CUDA(launch_ce_rows(p, dtype, vec, ptrs16, false, stream));
  return FLCE_OK;
}

flce_status_t ce_vp_backward(const void* logits, int dtype, void* grad_logits, const int64_t* target, int64_t N,
                             int64_t V_shard, int64_t vocab_offset, int64_t ignore_index, const float* lse,
                             const float* row_scale, int32_t* status_dev, flce_stream_t stream_) {
  (void)status_dev;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP32 && dtype != FLCE_DTYPE_FP16) return FLCE_ERR_UNSUPPORTED;
  if (N < 0 || V_shard < 1 || vocab_offset < 0) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (logits == nullptr || grad_logits == nullptr || target == nullptr || lse == nullptr ||
                row_scale == nullptr))
    return FLCE_ERR_INVALID_ARG;
  const size_t esz = dtype == FLCE_DTYPE_FP32 ? 4 : 2;
  if (!aligned(logits, esz) || !aligned(grad_logits, esz) || !aligned(target, 8)) return FLCE_ERR_MISALIGNED;
  if (grad_logits != logits) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(grad_logits);
    const uintptr_t bytes = static_cast<uintptr_t>(N) * V_shard * esz;
    if (a < b + bytes && b < a + bytes) return FLCE_ERR_INVALID_ARG;
  }
  FLCE_TRY_CUDA(launch_ce_vp_grad(logits, grad_logits, dtype, target, N, V_shard, vocab_offset, ignore_index, lse,
                                  row_scale, stream));
  return FLCE_OK;
}

void flce_set_wait_timeout_ns(uint64_t timeout_ns) {
  g_timeout_ns.store(timeout_ns > 0 ? timeout_ns : 1);
}

flce_status_t flce_selftest_wait_timeout(int32_t* status_dev, uint64_t timeout_ns, flce_stream_t stream) {
  if (status_dev == nullptr || !aligned(status_dev, 4)) return FLCE_ERR_INVALID_ARG;
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FLCE_ERR_INVALID_ARG;
  return launch_wait_selftest(status_dev, timeout_ns, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FLCE_OK
             : FLCE_ERR_CUDA;
}

const char* flce_kernel_name(int id) {
  switch (id) {
    case FLCE_KERNEL_COUNT_TARGETS: return "count_targets";
    case FLCE_KERNEL_GEMM_FWD: return "gemm_forward";
    case FLCE_KERNEL_ROW_FINALIZE: return "row_finalize";
    case FLCE_KERNEL_GRAD_LOGITS: return "grad_logits";
    case FLCE_KERNEL_GEMM_BWD: return "gemm_backward";
    case FLCE_KERNEL_LOSS_REDUCE: return "loss_reduce";
    case FLCE_KERNEL_CE_ROWS: return "ce_rows";
    case FLCE_KERNEL_ZERO: return "zero";
    case FLCE_KERNEL_BIAS_REDUCE: return "bias_reduce";
    case FLCE_KERNEL_GH_REDUCE: return "gh_reduce";
  }
  return "unknown";
}

flce_status_t flce_profile_enable(int capacity) {
  if (capacity <= 0) return FLCE_ERR_INVALID_ARG;
  if (static_cast<int>(g_prof.start.size()) < capacity) {
    while (static_cast<int>(g_prof.start.size()) < capacity) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess) return FLCE_ERR_CUDA;
      if (cudaEventCreate(&b) != cudaSuccess) return FLCE_ERR_CUDA;
      g_prof.start.push_back(a);
      g_prof.stop.push_back(b);
      g_prof.ids.push_back(-1);
    }
  }
  g_prof.capacity = capacity;
  g_prof.count = 0;
  g_prof.open = false;
  g_prof.enabled = true;
  return FLCE_OK;
}

void flce_profile_disable(void) { g_prof.enabled = false; }

int flce_profile_read(int* kernel_ids, float* ms, int max) {
  int n = 0;
  for (int i = 0; i < g_prof.count && n < max; ++i) {
    float t = 0.f;
    if (cudaEventSynchronize(g_prof.stop[i]) != cudaSuccess) break;
    if (cudaEventElapsedTime(&t, g_prof.start[i], g_prof.stop[i]) != cudaSuccess) break;
    kernel_ids[n] = g_prof.ids[i];
    ms[n] = t;
    ++n;
  }
  g_prof.count = 0;
  return n;
}

}  // extern "C"
