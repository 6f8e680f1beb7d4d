// Internal declarations shared by the kernels and the host layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/flce.h"

namespace flce {

// ---------------------------------------------------------------- GEMM tiles
constexpr int kBM = 128;          // tile rows (tensor-memory lanes)
constexpr int kBN = 256;          // tile columns (fp32 accumulator columns)
constexpr int kBK = 64;           // k per pipeline stage (128 bytes of bf16)
// Warps that drain the accumulators: 4 (one per TMEM lane quarter) or 8 (two
// per quarter, each taking half of a tile's columns), chosen per launch.
// part_cols: columns of a tile one epilogue warp drains, and so of one LSE
// partial (256 or 128).
constexpr int part_cols(int epi_warps) { return kBN / (epi_warps / 4); }
// Forward launches use 8 epilogue warps when the k loop is short (H * nseg
// below 4096), where draining a tile takes longer than its MMAs.
inline int forward_epi_warps(int64_t H, int nseg) { return H * (nseg > 1 ? nseg : 1) < 4096 ? 8 : 4; }
constexpr int kTmemCols = 2 * kBN;  // two accumulators (double buffering)
constexpr int kTileRing = 8;      // scheduler ring of tile ids
constexpr int kBoxBytes = 64 * 64 * 2;             // one TMA box: 64 x 64 bf16

enum GemmMode { kModeForward = 0, kModeBackward = 1 };

struct GemmParams {
  // chunk geometry
  int64_t row0;      // first token of the chunk
  int c_len;         // tokens in the chunk
  int H, V;
  int num_tiles;     // total tiles of the launch
  // forward tiles: M = chunk tokens, N = vocabulary, K = H
  int f_num_m, f_kblocks;
  // backward tiles: grad_H (M = chunk tokens, N = H, K = V), then
  // grad_W (M = vocabulary, N = H, K = chunk tokens)
  int h_tiles, h_num_m, h_kblocks;
  int w_num_n, w_kblocks;
  // grad_H split along K (the vocabulary) when its tiles are fewer than the
  // SM pairs: h_tiles = h_base * h_split tiles, slice s taking k blocks
  // [s h_kbs, (s + 1) h_kbs); each slice writes fp32 partial sums to
  // gh_part [h_split][chunk rows][H] (slice stride gh_part_ld elements),
  // added in slice order by gh_reduce afterwards.  h_split 1: direct stores
  int h_base, h_split, h_kbs;
  float* gh_part;
  int64_t gh_part_ld;
  // forward epilogue
  const uint16_t* bias;     // bf16 [V] or null
  const int64_t* target;    // [N]
  int64_t v_offset;         // global id of this weight's first vocabulary row (0 unless sharded)
  uint16_t* zbuf;           // bf16 [c_len, ldz] chunk logits
  int64_t ldz;
  float4* partials;         // [c_len, nvt]: (max, sum exp(z - max), same over bf16(z), 0) per part_cols columns
  int nvt;                  // partials per row: ceil(V / part_cols(epi_warps))
  int epi_warps;            // 4 or 8 (forward_epi_warps); backward launches use 4
  float* tgt_logit;         // [c_len]
  // operands: 0 bf16, 1 fp16 (hidden, weight, bias, chunk logits, grad_hidden)
  int in_fp16;
  // fp32 operands split into bf16 hi + lo planes (nseg = 3; else 1 or 0):
  // every product is hi.hi + hi.lo + lo.hi, three segments of the k loop,
  // each reading the hi or lo map of an operand; the chunk logits are
  // stored as two planes z_plane elements apart (the upper and lower halves
  // of their fp32 bits) and their gradient comes back as bf16 hi + lo
  // planes at the same places; the bias is added in fp32 from bias_f32
  int nseg;
  int64_t z_plane;
  const float* bias_f32;
  // fp16 only: dZ is stored divided by the uniform part of the row scale
  // (see uniform_scale), which the backward epilogue multiplies back in
  const int* n_valid;
  const float* gmax;
  int reduction;
  float grad_scale;
  // backward epilogue
  uint16_t* grad_hidden;    // bf16 [N, H] or null
  float* grad_hidden_f32;   // fp32 [N, H] instead of grad_hidden (a shard's partial), or null
  float* grad_weight;       // fp32 [V, H] or null
  int gw_store;             // 1: overwrite grad_weight tiles, 0: add to them
  // scheduling / failure
  unsigned int* tile_counter;
  int* status;
  uint64_t timeout_ns;
};

struct RowParams {
  int64_t row0;
  int c_len;
  int64_t N, V;
  int64_t ignore_index;
  int reduction;
  float grad_scale;
  const float* grad_out;    // [N] or null
  const int64_t* target;
  const float4* partials;
  int nvt;
  const float* tgt_logit;
  const int* n_valid;
  float* row_lse;           // [c_len]: log-sum-exp of the bf16 logits (softmax of dZ)
  float* row_scale;         // [c_len]: 0 for ignored rows
  int* row_tgt;             // [c_len]: target column or -1; null: derived from target - v_offset
  int64_t v_offset;         // global id of the first vocabulary column (0 unless sharded)
  float* loss_rows;         // [N] (workspace, or the loss output for NONE)
  float* lse_out;           // [N] or null
  float* tl_out;            // [N] or null
  int* status;
  // grad-logits pass
  uint16_t* zbuf;           // chunk logits, bf16 or (z_fp16) fp16
  int64_t ldz;
  float* grad_bias;         // [V] or null
  // with grad_bias: the column sums of each block of gl_rows rows go to
  // bias_part [ceil(c_len / gl_rows), ldz] (fp32), then one thread per column
  // adds them to grad_bias in block order (deterministic)
  float* bias_part;
  int gl_rows;
  int z_fp16;
  // split fp32 operands: the chunk logits are two planes z_plane elements
  // apart (upper and lower halves of their fp32 bits); dZ goes back to the
  // same places as bf16 hi + lo planes.  0: one 16-bit plane
  int64_t z_plane;
  const float* gmax;        // fp16: max |grad_out| over valid rows (reduction none)
};

// Rows per block of the grad-logits pass when it also sums the bias gradient.
constexpr int kGlBiasRows = 128;

struct CeParams {
  const void* logits;
  void* grad;               // may alias logits, or null
  const int64_t* target;
  int64_t N, V;
  int64_t ignore_index;
  int reduction;
  float grad_scale;
  const float* grad_out;
  float* loss_rows;         // [N]
  const int* n_valid;
  int* status;
  int cluster;              // CTAs per row
  int64_t seg_len;          // elements per CTA segment (multiple of the vector width)
  float* loss_out;          // sum / mean: the last CTA writes the reduced loss here (null: no reduction)
  unsigned int* ticket;     // zeroed counter used to find the last CTA
  float* lse_out;           // partials mode (vocabulary shard): per-row LSE here, no gradient
  float* zt_out;            // partials mode: target logit if the target is in this shard, else 0
  int64_t v_offset;         // global id of this shard's first column
  // single-launch form (no count kernel, nothing zeroed beforehand): every CTA
  // counts the valid targets itself, and the last CTA to finish is found by
  // an arrival counter tagged with this call's nonce, instead of a zeroed
  // ticket
  int self_count;
  unsigned long long* done_flags;  // the tagged arrival counter (one word), or null: use `ticket`
  unsigned long long nonce;        // below 2^40, different from every earlier call's on this memory
  int clear_status;                // CTA 0 zeroes *status when it starts (the workspace's own word)
};

// The tagged arrival counter: the low kTagCountBits bits of the 64-bit word
// count, the bits above hold the call's nonce.
constexpr int kTagCountBits = 24;

// Most rows the single-launch CE form takes (each CTA reads every target).
constexpr int64_t kCeSelfCountMaxRows = 16384;
// Most CTAs the single-launch form's arrival counter can count.
constexpr int kCeMaxFlags = 1 << 20;

// fp16 operands: the part of every row's gradient scale that is the same for
// all rows (mean: g / n_valid; sum: g; none: g * max |grad_out|, or g).  The
// chunk's dZ is stored in fp16 divided by it, so its entries stay within
// [-1, 1] instead of underflowing, and the backward products multiply it back.
__device__ __forceinline__ float uniform_scale(int reduction, float grad_scale, const int* n_valid,
                                              const float* gmax) {
  if (reduction == FLCE_REDUCTION_MEAN) {
    const int nv = *n_valid;
    return nv > 0 ? grad_scale / static_cast<float>(nv) : 0.f;
  }
  if (reduction == FLCE_REDUCTION_SUM || gmax == nullptr) return grad_scale;
  return grad_scale * *gmax;
}

// Header at the start of every workspace.
struct WorkspaceHeader {
  int status;
  int n_valid;
  int pad[2];               // [0]: count kernel block ticket, [1]: CE kernel block ticket
  float gmax;               // max |grad_out| over valid rows, when asked for
  int pad2;
  double loss_sum;
  unsigned int tile_counters[];  // two per chunk
};

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.
// zero_header: one block zeroes the header itself (status when it is the
// header's own, counts, tickets and `num_counters` tile counters) before
// counting, so no memset is needed; otherwise the caller zeroes the header.
constexpr int64_t kCountSingleBlockMax = 65536;
// grad_out (optional): also leaves max |grad_out| over the valid rows in hdr->gmax.
cudaError_t launch_count_targets(const int64_t* target, int64_t N, int64_t V, int64_t ignore_index,
                                 WorkspaceHeader* hdr, int num_counters, int zero_header,
                                 int* status, int32_t* n_valid_out, float* zero_a, int64_t zero_a_n,
                                 const float* grad_out, cudaStream_t s);
// tm_h2 / tm_w2 / tm_z2: the lo planes of split fp32 operands (p.nseg = 3), else null
cudaError_t launch_gemm2(int mode, const CUtensorMap& tm_h, const CUtensorMap& tm_w,
                         const CUtensorMap& tm_z, const GemmParams& p, int grid, cudaStream_t s,
                         const CUtensorMap* tm_h2 = nullptr, const CUtensorMap* tm_w2 = nullptr,
                         const CUtensorMap* tm_z2 = nullptr);
cudaError_t launch_row_finalize(const RowParams& p, cudaStream_t s);
cudaError_t launch_grad_logits(const RowParams& p, cudaStream_t s);
cudaError_t launch_vp_finalize(const RowParams& p, float* lse_out, float* lse16_out, float* zt_out,
                               cudaStream_t s);
cudaError_t launch_ce_vp_grad(const void* logits, void* grad, int dtype, const int64_t* target, int64_t N,
                              int64_t V, int64_t v_offset, int64_t ignore_index, const float* lse,
                              const float* row_scale, cudaStream_t s);
cudaError_t launch_loss_reduce(const float* loss_rows, int64_t N, int reduction, const int* n_valid,
                               float* loss, cudaStream_t s, bool pdl);
cudaError_t launch_zero(float* p, int64_t n, cudaStream_t s);
cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t s);
cudaError_t launch_f32_split_bf16(const float* in, uint16_t* hi, uint16_t* lo, int64_t n, cudaStream_t s);
// grad_H rows [row0, row0 + rows) (H columns) from the split-K partial sums
// part [slices][rows][H] (slice stride `ld` elements), added in slice order:
// out16 (bf16, or fp16 when f16) or out32 (fp32), whichever is not null.
cudaError_t launch_gh_reduce(const float* part, int slices, int64_t ld, int rows, int H, int64_t row0,
                             uint16_t* out16, int f16, float* out32, cudaStream_t s);
// vector_path: rows are whole 16-byte vectors and both pointers 16-byte
// aligned; aligned_ptrs: both pointers 16-byte aligned (rows of any length).
bool vp_partials_rows_fits(int dtype, int64_t V, bool vector_path);
cudaError_t launch_vp_partials_rows(const void* logits, int dtype, const int64_t* target, int64_t N, int64_t V,
                                    int64_t v_offset, int64_t ignore_index, float* lse_out, float* zt_out,
                                    cudaStream_t s);
cudaError_t launch_ce_rows(const CeParams& p, int dtype, bool vector_path, bool aligned_ptrs, bool pdl,
                           cudaStream_t s);
// Whether rows of V elements go to a form that supports the single launch
// (the row-ring or streaming kernel).
bool ce_rows_single_launch_ok(int64_t V, int dtype, bool vector_path, bool aligned_ptrs);
cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s);

int device_sm_count();

// ---------------------------------------------------------------- profiler
void prof_begin(cudaStream_t s, int kernel_id);
void prof_end(cudaStream_t s);

}  // namespace flce
