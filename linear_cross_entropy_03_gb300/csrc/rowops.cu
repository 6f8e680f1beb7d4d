// Memory-bound row kernels of the fused linear cross entropy.
//
//  count_targets   number of valid targets over all N rows (the mean's
//                  denominator, which must be known before any chunk's
//                  gradient is formed) and the target range check.
//  row_finalize    per chunk row: combine the per-vocabulary-tile (max, sum of
//                  exp) partials into the log-sum-exp, the row loss and the
//                  row's gradient scale.
//  grad_logits     per chunk: dZ = scale * (softmax - onehot) written in place
//                  over the chunk's bf16 logits, plus the bias gradient as
//                  column sums (torchtune post "Peak Performance, Minimized
//                  Memory ...", Figure 1, step 3; liger-kernel README
//                  "Kernels", CrossEntropy item).
//  loss_reduce     sum (or mean) of the per-row losses in a fixed order.
#include <cuda_fp16.h>
#include <math.h>

#include "ptx.cuh"

namespace flce {
namespace {

constexpr int kCountThreads = 1024;

__global__ void __launch_bounds__(kCountThreads)
    count_targets_kernel(const int64_t* __restrict__ target, int64_t N, int64_t V, int64_t ignore_index,
                         WorkspaceHeader* hdr, int* status, int32_t* n_valid_out, float* zero_a,
                         int64_t zero_a_n, int zero_header, int num_counters, const float* grad_out) {
  grid_dependents_launch();
  if (zero_header) {  // single block: clear the header first
    if (threadIdx.x == 0) {
      if (status == &hdr->status) hdr->status = 0;
      hdr->pad[0] = 0;
      hdr->pad[1] = 0;
      hdr->gmax = 0.f;
      hdr->loss_sum = 0.0;
    }
    for (int i = threadIdx.x; i < num_counters; i += blockDim.x) hdr->tile_counters[i] = 0u;
    __syncthreads();
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_a_n; i += stride)
    zero_a[i] = 0.f;
  int cnt = 0;
  bool bad = false;
  float gm = 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < N; i += stride) {
    const int64_t t = target[i];
    if (t != ignore_index) {
      if (t >= 0 && t < V) {
        ++cnt;
        if (grad_out != nullptr) gm = fmaxf(gm, fabsf(grad_out[i]));
      } else {
        bad = true;
      }
    }
  }
  if (grad_out != nullptr) {  // non-negative floats order like their bit patterns
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
    if ((threadIdx.x & 31) == 0 && gm > 0.f) atomicMax(reinterpret_cast<int*>(&hdr->gmax), __float_as_int(gm));
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, FLCE_STATUS_BIT_TARGET_RANGE);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  __shared__ int s_cnt[kCountThreads / 32];
  __shared__ bool s_last;
  if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += s_cnt[w];
    if (zero_header) {
      hdr->n_valid = total;
      if (n_valid_out != nullptr) *n_valid_out = total;
    } else {
      atomicAdd(&hdr->n_valid, total);
      __threadfence();
      const unsigned int ticket = atomicAdd(reinterpret_cast<unsigned int*>(&hdr->pad[0]), 1u);
      s_last = ticket == gridDim.x - 1;
    }
  }
  if (zero_header) return;
  __syncthreads();
  if (s_last && threadIdx.x == 0 && n_valid_out != nullptr) {
    __threadfence();
    *n_valid_out = atomicAdd(&hdr->n_valid, 0);
  }
}

constexpr int kFinalizeWarps = 8;

__global__ void __launch_bounds__(32 * kFinalizeWarps) row_finalize_kernel(const RowParams p) {
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kFinalizeWarps + warp;
  if (r >= p.c_len) return;
  const int64_t n = p.row0 + r;
  const float4* pr = p.partials + static_cast<int64_t>(r) * p.nvt;
  float m = -INFINITY;
  for (int i = lane; i < p.nvt; i += 32) m = fmaxf(m, pr[i].x);
  m = warp_max(m);
  float s32 = 0.f, s16 = 0.f;
  for (int i = lane; i < p.nvt; i += 32) {
    const float4 q = pr[i];
    const float e = __expf(q.x - m);
    s32 += q.y * e;
    s16 += q.z * e;
  }
  s32 = warp_sum(s32);
  s16 = warp_sum(s16);
  if (lane == 0) {
    // The loss uses the log-sum-exp of the fp32 logits; the gradient's
    // softmax is normalised over the bf16 logits it is formed from, so each
    // dZ row sums to zero.
    const float lse = m + logf(s32);
    const float lse_bf16 = m + logf(s16);
    const int64_t t = p.target[n];
    const bool in_range = t >= 0 && t < p.V;
    const bool valid = t != p.ignore_index && in_range;
    if (t != p.ignore_index && !in_range) atomicOr(p.status, FLCE_STATUS_BIT_TARGET_RANGE);
    const float zt = valid ? p.tgt_logit[r] : 0.f;
    const float loss = valid ? lse - zt : 0.f;
    float scale = 0.f;
    if (valid) {
      if (p.reduction == FLCE_REDUCTION_MEAN)
        scale = p.grad_scale / static_cast<float>(*p.n_valid);
      else if (p.reduction == FLCE_REDUCTION_SUM)
        scale = p.grad_scale;
      else
        scale = p.grad_scale * (p.grad_out != nullptr ? p.grad_out[n] : 1.f);
    }
    p.row_lse[r] = lse_bf16;
    p.row_scale[r] = scale;
    p.row_tgt[r] = valid ? static_cast<int>(t) : -1;
    p.loss_rows[n] = loss;
    if (p.lse_out != nullptr) p.lse_out[n] = lse;
    if (p.tl_out != nullptr) p.tl_out[n] = zt;
  }
}

constexpr int kGlThreads = 256;
constexpr int kGlCols = kGlThreads * 8;  // one 16-byte vector of bf16 per thread
constexpr int kGlRows = 32;              // rows per block without the bias gradient
constexpr int kGlUnroll = 4;
static_assert(kGlBiasRows >= kGlRows && kGlBiasRows % kGlUnroll == 0, "grad-logits row blocks");

// F16: fp16 chunk logits; dZ is stored divided by the rows' common scale
// (uniform_scale), which the backward products multiply back in.  SPLIT:
// exact fp32 chunk logits in two planes, dZ written back as bf16 hi + lo.
template <bool F16>
__device__ __forceinline__ float z_lo(uint32_t w) {
  return F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))) : bf16_lo(w);
}
template <bool F16>
__device__ __forceinline__ float z_hi(uint32_t w) {
  return F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))) : bf16_hi(w);
}
template <bool F16>
__device__ __forceinline__ uint32_t z_pack(float lo, float hi) {
  if (F16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  return pack_bf16x2(lo, hi);
}

// d rounded to bf16 (nearest even) and the rounded remainder: d = hi + lo to
// about 2^-16 of |d|.
__device__ __forceinline__ void split_bf16(float d0, float d1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(d0, d1);
  lo = pack_bf16x2(d0 - bf16_lo(hi), d1 - bf16_hi(hi));
}

template <bool F16, bool SPLIT>
__global__ void __launch_bounds__(kGlThreads) grad_logits_kernel(const RowParams p) {
  __shared__ float s_lse[kGlBiasRows], s_scale[kGlBiasRows];
  __shared__ int s_tgt[kGlBiasRows];
  grid_dependency_wait();
  const int r0 = blockIdx.y * p.gl_rows;
  const int rows = min(p.gl_rows, p.c_len - r0);
  for (int i = threadIdx.x; i < rows; i += kGlThreads) {
    s_lse[i] = p.row_lse[r0 + i];
    s_scale[i] = p.row_scale[r0 + i];
    if (p.row_tgt != nullptr) {
      s_tgt[i] = p.row_tgt[r0 + i];
    } else {  // vocabulary shard: the target's column here, or -1 if another shard holds it
      const int64_t tg = p.target[p.row0 + r0 + i];
      const int64_t tl = tg - p.v_offset;
      s_tgt[i] = (tg != p.ignore_index && tl >= 0 && tl < p.V) ? static_cast<int>(tl) : -1;
    }
  }
  __syncthreads();
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kGlCols + threadIdx.x * 8;
  if (v0 >= p.V) return;
  const int nval = p.V - v0 < 8 ? static_cast<int>(p.V - v0) : 8;
  float store_mul = 1.f;
  if (F16) {
    const float u = uniform_scale(p.reduction, p.grad_scale, p.n_valid, p.gmax);
    store_mul = u != 0.f ? 1.f / u : 0.f;
  }
  float cs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) cs[j] = 0.f;
  uint16_t* base = p.zbuf + static_cast<int64_t>(r0) * p.ldz + v0;
  for (int rr = 0; rr < rows; rr += kGlUnroll) {
    uint4 in[kGlUnroll], in_lo[SPLIT ? kGlUnroll : 1];
#pragma unroll
    for (int u = 0; u < kGlUnroll; ++u) {
      const bool live = rr + u < rows && s_scale[rr + u] != 0.f;
      const uint16_t* src = base + static_cast<int64_t>(rr + u) * p.ldz;
      in[u] = live ? __ldcs(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
      if (SPLIT) in_lo[u] = live ? __ldcs(reinterpret_cast<const uint4*>(src + p.z_plane)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kGlUnroll; ++u) {
      const int r = rr + u;
      if (r >= rows) break;
      uint4* dst = reinterpret_cast<uint4*>(base + static_cast<int64_t>(r) * p.ldz);
      uint4* dst_lo = SPLIT ? reinterpret_cast<uint4*>(base + static_cast<int64_t>(r) * p.ldz + p.z_plane) : nullptr;
      const int t = s_tgt[r];  // -1: no target column in this block of the vocabulary
      if (s_scale[r] == 0.f) {  // ignored row (or zero upstream gradient): exact zeros
        __stcs(dst, make_uint4(0, 0, 0, 0));
        if (SPLIT) __stcs(dst_lo, make_uint4(0, 0, 0, 0));
        continue;
      }
      const float lse = s_lse[r], sc = s_scale[r];
      const uint32_t w[4] = {in[u].x, in[u].y, in[u].z, in[u].w};
      float d[8];
      if (SPLIT) {  // the exact fp32 logits from their two halves
        const uint32_t wl[4] = {in_lo[SPLIT ? u : 0].x, in_lo[SPLIT ? u : 0].y, in_lo[SPLIT ? u : 0].z,
                                in_lo[SPLIT ? u : 0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          d[2 * i] = __uint_as_float(__byte_perm(wl[i], w[i], 0x5410));
          d[2 * i + 1] = __uint_as_float(__byte_perm(wl[i], w[i], 0x7632));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          d[2 * i] = z_lo<F16>(w[i]);
          d[2 * i + 1] = z_hi<F16>(w[i]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float onehot = (v0 + j == t) ? 1.f : 0.f;
        d[j] = sc * (__expf(d[j] - lse) - onehot);
        if (j < nval) cs[j] += d[j];
      }
      uint4 o;
      if (SPLIT) {
        uint4 ol;
        split_bf16(d[0], d[1], o.x, ol.x);
        split_bf16(d[2], d[3], o.y, ol.y);
        split_bf16(d[4], d[5], o.z, ol.z);
        split_bf16(d[6], d[7], o.w, ol.w);
        __stcs(dst_lo, ol);
      } else {
        o.x = z_pack<F16>(store_mul * d[0], store_mul * d[1]);
        o.y = z_pack<F16>(store_mul * d[2], store_mul * d[3]);
        o.z = z_pack<F16>(store_mul * d[4], store_mul * d[5]);
        o.w = z_pack<F16>(store_mul * d[6], store_mul * d[7]);
      }
      __stcs(dst, o);
    }
  }
  if (p.grad_bias != nullptr) {  // this block's column sums; bias_reduce adds the blocks in order
    float* dst = p.bias_part + static_cast<int64_t>(blockIdx.y) * p.ldz + v0;
    if (nval == 8) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(cs[0], cs[1], cs[2], cs[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(cs[4], cs[5], cs[6], cs[7]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < nval) dst[j] = cs[j];
    }
  }
}

// grad_bias[v] += sum over row blocks b (in order) of part[b, v]: one thread
// per column, so the sum's order is fixed and the result the same every run.
__global__ void __launch_bounds__(256) bias_reduce_kernel(const float* __restrict__ part, int blocks, int64_t ld,
                                                          int64_t V, float* __restrict__ grad_bias) {
  const int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (v >= V) return;
  float acc = 0.f;
  for (int b = 0; b < blocks; ++b) acc += part[static_cast<int64_t>(b) * ld + v];
  grad_bias[v] += acc;
}

// Per-row partials of one vocabulary shard after its forward products:
// LSE over the shard's fp32 logits, LSE over their bf16 roundings, and the
// target logit when the target lies in the shard (else 0).
__global__ void __launch_bounds__(32 * kFinalizeWarps)
    vp_finalize_kernel(const RowParams p, float* lse_out, float* lse16_out, float* zt_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kFinalizeWarps + warp;
  if (r >= p.c_len) return;
  const float4* pr = p.partials + static_cast<int64_t>(r) * p.nvt;
  float m = -INFINITY;
  for (int i = lane; i < p.nvt; i += 32) m = fmaxf(m, pr[i].x);
  m = warp_max(m);
  float s32 = 0.f, s16 = 0.f;
  for (int i = lane; i < p.nvt; i += 32) {
    const float4 q = pr[i];
    const float e = __expf(q.x - m);
    s32 += q.y * e;
    s16 += q.z * e;
  }
  s32 = warp_sum(s32);
  s16 = warp_sum(s16);
  if (lane == 0) {
    const int64_t n = p.row0 + r;
    const int64_t tg = p.target[n];
    const int64_t tl = tg - p.v_offset;
    const bool here = tg != p.ignore_index && tl >= 0 && tl < p.V;
    lse_out[n] = m + logf(s32);
    lse16_out[n] = m + logf(s16);
    zt_out[n] = here ? p.tgt_logit[r] : 0.f;
  }
}

// Gradient of the cross entropy on one vocabulary shard of materialised
// logits, given the row LSE over the whole vocabulary and the row scale:
// dZ = scale * (exp(z - lse) - [column == target]), written in place or to a
// separate buffer; rows with scale 0 get exact zeros.
__device__ __forceinline__ float load_as_f(const uint16_t* p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }
__device__ __forceinline__ float load_as_f(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float load_as_f(const float* p) { return *p; }
__device__ __forceinline__ void store_f(uint16_t* p, float v) { *p = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu); }
__device__ __forceinline__ void store_f(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void store_f(float* p, float v) { *p = v; }

template <typename T>
__global__ void __launch_bounds__(256)
    ce_vp_grad_kernel(const T* __restrict__ logits, T* grad, const int64_t* __restrict__ target, int64_t N, int64_t V,
                      int64_t v_offset, int64_t ignore_index, const float* __restrict__ lse,
                      const float* __restrict__ row_scale) {
  for (int64_t row = blockIdx.y; row < N; row += gridDim.y) {
  const int64_t tg = target[row];
  const int64_t tl = tg - v_offset;
  const int64_t t = (tg != ignore_index && tl >= 0 && tl < V) ? tl : -1;
  const float sc = row_scale[row];
  const float l = lse[row];
  const T* x = logits + row * V;
  T* g = grad + row * V;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < V;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float z = load_as_f(x + v);
    const float d = sc == 0.f ? 0.f : sc * (__expf(z - l) - (v == t ? 1.f : 0.f));
    store_f(g + v, d);
  }
  }
}

// The same with 16-byte vectors (rows of a multiple of 16 bytes, 16-byte
// aligned): one vector per thread and step, grid (vectors of a row, rows).
// Packed fp32x2 arithmetic: exp(z - lse) as ex2 of one fused multiply-add,
// times the row scale; the target element's onehot is taken off in the one
// vector that holds it.
__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8], uint16_t) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[2 * q] = bf16_lo(w[q]);
    x[2 * q + 1] = bf16_hi(w[q]);
  }
}
__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8], __half) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __half22float2(h[q]);
    x[2 * q] = f.x;
    x[2 * q + 1] = f.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8], uint16_t) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8], __half) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2 h = __floats2half2_rn(x[2 * q], x[2 * q + 1]);
    w[q] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(256)
    ce_vp_grad_vec_kernel(const T* __restrict__ logits, T* grad, const int64_t* __restrict__ target, int64_t N,
                          int64_t V, int64_t v_offset, int64_t ignore_index, const float* __restrict__ lse,
                          const float* __restrict__ row_scale) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr float kL2e = 1.4426950408889634f;
  const int64_t nvec = V / EPV;
  for (int64_t row = blockIdx.y; row < N; row += gridDim.y) {
    const int64_t tg = target[row];
    const int64_t tl = tg - v_offset;
    const int64_t t = (tg != ignore_index && tl >= 0 && tl < V) ? tl : -1;
    const int64_t tvec = t >= 0 ? t / EPV : -1;  // the vector holding the target, and its element
    const int tel = t >= 0 ? static_cast<int>(t % EPV) : 0;
    const float sc = row_scale[row];
    const float nl = -lse[row] * kL2e;
    const uint4* x = reinterpret_cast<const uint4*>(logits + row * V);
    uint4* g = reinterpret_cast<uint4*>(grad + row * V);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (sc == 0.f) {  // an ignored row (or grad_out 0): zero gradient
        __stcs(g + i, make_uint4(0, 0, 0, 0));
        continue;
      }
      const uint4 u = __ldcs(x + i);
      float z[8];
      if constexpr (EPV == 8) {
        unpack8(u, z, T());
      } else {
        z[0] = __uint_as_float(u.x);
        z[1] = __uint_as_float(u.y);
        z[2] = __uint_as_float(u.z);
        z[3] = __uint_as_float(u.w);
      }
      const float2 l2e = make_float2(kL2e, kL2e), nl2 = make_float2(nl, nl), sc2 = make_float2(sc, sc);
#pragma unroll
      for (int q = 0; q < EPV / 2; ++q) {
        const float2 a = __ffma2_rn(make_float2(z[2 * q], z[2 * q + 1]), l2e, nl2);
        const float2 d = __fmul2_rn(make_float2(ex2_approx(a.x), ex2_approx(a.y)), sc2);
        z[2 * q] = d.x;
        z[2 * q + 1] = d.y;
      }
      if (i == tvec) {
#pragma unroll
        for (int k = 0; k < EPV; ++k)
          if (k == tel) z[k] -= sc;
      }
      if constexpr (EPV == 8) {
        __stcs(g + i, pack8(z, T()));
      } else {
        __stcs(g + i, make_uint4(__float_as_uint(z[0]), __float_as_uint(z[1]), __float_as_uint(z[2]),
                                 __float_as_uint(z[3])));
      }
    }
  }
}

// fp32 -> bf16 (round to nearest even), 8 elements per thread and step,
// scalar tail; in and out 16-byte aligned.
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* __restrict__ in, uint16_t* __restrict__ out,
                                                          int64_t n) {
  const int64_t n8 = n / 8;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += step) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(in) + 2 * i);
    const float4 b = __ldcs(reinterpret_cast<const float4*>(in) + 2 * i + 1);
    reinterpret_cast<uint4*>(out)[i] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
  for (int64_t i = n8 * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step)
    out[i] = static_cast<uint16_t>(pack_bf16x2(in[i], 0.f) & 0xFFFFu);
}

// fp32 -> bf16 hi + lo planes: hi = x rounded to bf16 (nearest even), lo =
// (x - hi) rounded likewise, so hi + lo equals x to about 2^-16 of |x|.
// 8 elements per thread and step, scalar tail; pointers 16-byte aligned.
__global__ void __launch_bounds__(256) f32_split_bf16_kernel(const float* __restrict__ in, uint16_t* __restrict__ hi,
                                                             uint16_t* __restrict__ lo, int64_t n) {
  const int64_t n8 = n / 8;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += step) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(in) + 2 * i);
    const float4 b = __ldcs(reinterpret_cast<const float4*>(in) + 2 * i + 1);
    uint4 h, l;
    split_bf16(a.x, a.y, h.x, l.x);
    split_bf16(a.z, a.w, h.y, l.y);
    split_bf16(b.x, b.y, h.z, l.z);
    split_bf16(b.z, b.w, h.w, l.w);
    reinterpret_cast<uint4*>(hi)[i] = h;
    reinterpret_cast<uint4*>(lo)[i] = l;
  }
  for (int64_t i = n8 * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step) {
    uint32_t h, l;
    split_bf16(in[i], 0.f, h, l);
    hi[i] = static_cast<uint16_t>(h & 0xFFFFu);
    lo[i] = static_cast<uint16_t>(l & 0xFFFFu);
  }
}

// grad_H from the split-K partial sums: 8 consecutive columns per thread and
// step (H % 8 == 0), slices added in order (deterministic).
__global__ void __launch_bounds__(256) gh_reduce_kernel(const float* __restrict__ part, int slices, int64_t ld,
                                                        int rows, int H, int64_t row0, uint16_t* out16, int f16,
                                                        float* out32) {
  const int64_t n8 = static_cast<int64_t>(rows) * H / 8;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += step) {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int s = 0;
    for (; s + 4 <= slices; s += 4) {  // four slices' loads in flight, added in slice order
      float4 x[4], y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4* src = reinterpret_cast<const float4*>(part + (s + k) * ld) + 2 * i;
        x[k] = __ldcs(src);
        y[k] = __ldcs(src + 1);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a[0] += x[k].x; a[1] += x[k].y; a[2] += x[k].z; a[3] += x[k].w;
        a[4] += y[k].x; a[5] += y[k].y; a[6] += y[k].z; a[7] += y[k].w;
      }
    }
    for (; s < slices; ++s) {
      const float4* src = reinterpret_cast<const float4*>(part + s * ld) + 2 * i;
      const float4 x = __ldcs(src), y = __ldcs(src + 1);
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
      a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    }
    const int64_t o = row0 * H + 8 * i;  // rows of the chunk lie row0 rows into the output
    if (out32 != nullptr) {
      reinterpret_cast<float4*>(out32 + o)[0] = make_float4(a[0], a[1], a[2], a[3]);
      reinterpret_cast<float4*>(out32 + o)[1] = make_float4(a[4], a[5], a[6], a[7]);
    } else if (f16) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 h = __floats2half2_rn(a[2 * q], a[2 * q + 1]);
        w[q] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(out16 + o) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      *reinterpret_cast<uint4*>(out16 + o) =
          make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
    }
  }
}

constexpr int kReduceThreads = 1024;

__global__ void __launch_bounds__(kReduceThreads)
    loss_reduce_kernel(const float* __restrict__ loss_rows, int64_t N, int reduction,
                       const int* n_valid, float* loss) {
  grid_dependency_wait();
  // each thread: a compensated fp32 sum of its rows in index order; then two
  // fixed shuffle trees (warp, then block).  Deterministic, and accurate to
  // about 1e-6 relative for any N (fp32 throughout: fp64 is slow here)
  float sum = 0.f, comp = 0.f;
  for (int64_t i = threadIdx.x; i < N; i += kReduceThreads) {
    const float y = loss_rows[i] - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  }
  float acc = sum - comp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ float s_acc[kReduceThreads / 32];
  if ((threadIdx.x & 31) == 0) s_acc[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float total = s_acc[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    if (threadIdx.x == 0) {
      if (reduction == FLCE_REDUCTION_MEAN) {
        const int nv = *n_valid;
        loss[0] = nv > 0 ? total / static_cast<float>(nv) : __int_as_float(0x7fc00000);
      } else {
        loss[0] = total;
      }
    }
  }
}

__global__ void zero_kernel(float* p, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    p[i] = 0.f;
}

// One thread waits on a barrier nothing will ever arrive on.
__global__ void wait_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_addr(&bar), 1);
  fence_barrier_init();
  const WaitCtl ctl{&abort_flag, status, timeout_ns};
  if (mbar_wait(smem_addr(&bar), 0, ctl)) atomicOr(status, 0x100);  // cannot happen
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 132;
  }
  return cached[dev];
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_count_targets(const int64_t* target, int64_t N, int64_t V, int64_t ignore_index,
                                 WorkspaceHeader* hdr, int num_counters, int zero_header,
                                 int* status, int32_t* n_valid_out, float* zero_a, int64_t zero_a_n,
                                 const float* grad_out, cudaStream_t s) {
  const int64_t work = N > zero_a_n ? N : zero_a_n;
  int blocks = static_cast<int>((work + kCountThreads * 4 - 1) / (kCountThreads * 4));
  blocks = blocks < 1 ? 1 : (blocks > sm_count() ? sm_count() : blocks);
  if (zero_header) blocks = 1;
  prof_begin(s, FLCE_KERNEL_COUNT_TARGETS);
  count_targets_kernel<<<blocks, kCountThreads, 0, s>>>(target, N, V, ignore_index, hdr, status, n_valid_out,
                                                       zero_a, zero_a_n, zero_header, num_counters, grad_out);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

cudaError_t launch_row_finalize(const RowParams& p, cudaStream_t s) {
  const int blocks = (p.c_len + kFinalizeWarps - 1) / kFinalizeWarps;
  prof_begin(s, FLCE_KERNEL_ROW_FINALIZE);
  RowParams pc = p;
  void* args[] = {&pc};
  const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(row_finalize_kernel), dim3(blocks),
                                   dim3(32 * kFinalizeWarps), args, s, false);
  prof_end(s);
  return e;
}

cudaError_t launch_grad_logits(const RowParams& p, cudaStream_t s) {
  RowParams pc = p;
  pc.gl_rows = p.grad_bias != nullptr ? kGlBiasRows : kGlRows;
  const int row_blocks = (p.c_len + pc.gl_rows - 1) / pc.gl_rows;
  const dim3 grid(static_cast<unsigned>((p.V + kGlCols - 1) / kGlCols), static_cast<unsigned>(row_blocks));
  prof_begin(s, FLCE_KERNEL_GRAD_LOGITS);
  void* args[] = {&pc};
  const void* fn = p.z_fp16    ? reinterpret_cast<const void*>(grad_logits_kernel<true, false>)
                   : p.z_plane ? reinterpret_cast<const void*>(grad_logits_kernel<false, true>)
                               : reinterpret_cast<const void*>(grad_logits_kernel<false, false>);
  cudaError_t e = launch_pdl(fn, grid, dim3(kGlThreads), args, s, false);
  prof_end(s);
  if (e != cudaSuccess || p.grad_bias == nullptr) return e;
  prof_begin(s, FLCE_KERNEL_BIAS_REDUCE);
  bias_reduce_kernel<<<static_cast<unsigned>((p.V + 255) / 256), 256, 0, s>>>(p.bias_part, row_blocks, p.ldz, p.V,
                                                                            p.grad_bias);
  e = cudaGetLastError();
  prof_end(s);
  return e;
}

cudaError_t launch_vp_finalize(const RowParams& p, float* lse_out, float* lse16_out, float* zt_out,
                               cudaStream_t s) {
  const int blocks = (p.c_len + kFinalizeWarps - 1) / kFinalizeWarps;
  prof_begin(s, FLCE_KERNEL_ROW_FINALIZE);
  vp_finalize_kernel<<<blocks, 32 * kFinalizeWarps, 0, s>>>(p, lse_out, lse16_out, zt_out);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

cudaError_t launch_ce_vp_grad(const void* logits, void* grad, int dtype, const int64_t* target, int64_t N,
                              int64_t V, int64_t v_offset, int64_t ignore_index, const float* lse,
                              const float* row_scale, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  const size_t esz = dtype == FLCE_DTYPE_FP32 ? 4 : 2;
  const bool vec = (static_cast<size_t>(V) * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(grad) % 16 == 0;
  if (vec) {
    const int64_t nvec = static_cast<int64_t>(V) * esz / 16;
    int64_t bx = (nvec + 255) / 256;
    if (bx > 64) bx = 64;
    const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(N < 65535 ? N : 65535));
    prof_begin(s, FLCE_KERNEL_CE_ROWS);
    if (dtype == FLCE_DTYPE_BF16)
      ce_vp_grad_vec_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(logits),
                                                            static_cast<uint16_t*>(grad), target, N, V, v_offset,
                                                            ignore_index, lse, row_scale);
    else if (dtype == FLCE_DTYPE_FP16)
      ce_vp_grad_vec_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(logits),
                                                          static_cast<__half*>(grad), target, N, V, v_offset,
                                                          ignore_index, lse, row_scale);
    else
      ce_vp_grad_vec_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(logits), static_cast<float*>(grad),
                                                         target, N, V, v_offset, ignore_index, lse, row_scale);
    const cudaError_t e = cudaGetLastError();
    prof_end(s);
    return e;
  }
  int64_t bx = (V + 255) / 256;
  if (bx > 64) bx = 64;
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(N < 65535 ? N : 65535));
  prof_begin(s, FLCE_KERNEL_CE_ROWS);
  if (dtype == FLCE_DTYPE_BF16)
    ce_vp_grad_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(logits),
                                                      static_cast<uint16_t*>(grad), target, N, V, v_offset,
                                                      ignore_index, lse, row_scale);
  else if (dtype == FLCE_DTYPE_FP16)
    ce_vp_grad_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(logits), static_cast<__half*>(grad),
                                                    target, N, V, v_offset, ignore_index, lse, row_scale);
  else
    ce_vp_grad_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(logits), static_cast<float*>(grad),
                                                   target, N, V, v_offset, ignore_index, lse, row_scale);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n / 8 + 255) / 256;
  const int64_t cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  f32_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_f32_split_bf16(const float* in, uint16_t* hi, uint16_t* lo, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n / 8 + 255) / 256;
  const int64_t cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  f32_split_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(in, hi, lo, n);
  return cudaGetLastError();
}

cudaError_t launch_gh_reduce(const float* part, int slices, int64_t ld, int rows, int H, int64_t row0,
                             uint16_t* out16, int f16, float* out32, cudaStream_t s) {
  const int64_t n8 = static_cast<int64_t>(rows) * H / 8;
  if (n8 <= 0) return cudaSuccess;
  int64_t blocks = (n8 + 255) / 256;
  const int64_t cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  prof_begin(s, FLCE_KERNEL_GH_REDUCE);
  gh_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(part, slices, ld, rows, H, row0, out16, f16, out32);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

cudaError_t launch_loss_reduce(const float* loss_rows, int64_t N, int reduction, const int* n_valid,
                               float* loss, cudaStream_t s, bool pdl) {
  prof_begin(s, FLCE_KERNEL_LOSS_REDUCE);
  void* args[] = {&loss_rows, &N, &reduction, &n_valid, &loss};
  const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(loss_reduce_kernel), dim3(1),
                                   dim3(kReduceThreads), args, s, pdl);
  prof_end(s);
  return e;
}

cudaError_t launch_zero(float* p, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int blocks = static_cast<int>((n + 256 * 8 - 1) / (256 * 8));
  blocks = blocks > 4 * sm_count() ? 4 * sm_count() : blocks;
  prof_begin(s, FLCE_KERNEL_ZERO);
  zero_kernel<<<blocks, 256, 0, s>>>(p, n);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

int device_sm_count() { return sm_count(); }

}  // namespace flce
