// Cross entropy on materialised logits [N, V] (bf16, fp16 or fp32): loss and
// the logits gradient in one pass over the bytes (liger-kernel 0.0.1 ->
// 0.1.1 PyPI diff, README "Kernels", CrossEntropy item: loss and gradient
// computed together, the gradient optionally replacing the input; DeepSpeed
// PR #8540 "Changes": FP32/FP16/BF16 logits).
//
// HBM-bound; three forms by row length, all reading every logit from DRAM
// once and writing its gradient once:
//  - rows up to 72 KB: the row ring -- persistent 1024-thread CTAs, one per
//    SM, whole rows brought into a shared-memory ring by TMA bulk copies,
//    two 512-thread groups taking alternate rows, each row held in registers
//    from max to gradient store;
//  - longer rows: the streaming form -- persistent 512-thread CTAs, a first
//    pass with an online (max, sum of exp) per thread, a second pass that
//    re-reads the row from L2 and writes the gradient;
//  - pointers that are not 16-byte aligned: one thread-block cluster per
//    row, each CTA a segment in registers, the row's partials combined
//    through distributed shared memory (segments longer than the registers
//    hold read twice).
// Rows that are not a whole number of 16-byte vectors use the first two
// forms through their 16-byte-aligned covering range.  For sum / mean one
// CTA adds the per-CTA loss partials in a fixed order (deterministic).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace flce {
namespace {

constexpr int kCeThreads = 256;
constexpr int kCeVecs = 4;  // vectors held per thread
constexpr int kCeWarps = kCeThreads / 32;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<uint16_t>(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ uint16_t from_f<uint16_t>(float v) {
  return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// EPV consecutive elements (EPV * sizeof(T) == 16 on the vector path).
template <typename T, int EPV>
struct Packet {
  T v[EPV];
};

template <typename T, int EPV>
__device__ __forceinline__ void load_packet(Packet<T, EPV>& pk, const T* src) {
  if constexpr (EPV * sizeof(T) == 16) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(src));
    *reinterpret_cast<uint4*>(pk.v) = u;
  } else {
#pragma unroll
    for (int k = 0; k < EPV; ++k) pk.v[k] = src[k];
  }
}

template <typename T, int EPV>
__device__ __forceinline__ void store_packet(T* dst, const Packet<T, EPV>& pk) {
  if constexpr (EPV * sizeof(T) == 16) {
    __stcs(reinterpret_cast<uint4*>(dst), *reinterpret_cast<const uint4*>(pk.v));
  } else {
#pragma unroll
    for (int k = 0; k < EPV; ++k) dst[k] = pk.v[k];
  }
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Gradient of one packet, written back into the packet; returns the target
// logit if the packet holds the target (else leaves zt unchanged).
template <typename T, int EPV>
__device__ __forceinline__ void grad_packet(Packet<T, EPV>& pk, int64_t e, int64_t t, bool valid, float scale,
                                            float lse, float& zt, bool& found) {
#pragma unroll
  for (int k = 0; k < EPV; ++k) {
    const float z = to_f<T>(pk.v[k]);
    const bool hit = valid && (e + k == t);
    if (hit) {
      zt = z;
      found = true;
    }
    const float d = valid ? scale * (__expf(z - lse) - (hit ? 1.f : 0.f)) : 0.f;
    pk.v[k] = from_f<T>(d);
  }
}

template <typename T, int EPV>
__device__ __forceinline__ void find_target(const Packet<T, EPV>& pk, int64_t e, int64_t t, float& zt,
                                            bool& found) {
#pragma unroll
  for (int k = 0; k < EPV; ++k)
    if (e + k == t) {
      zt = to_f<T>(pk.v[k]);
      found = true;
    }
}

template <typename T, int EPV>
__global__ void __launch_bounds__(kCeThreads) ce_rows_kernel(const CeParams p) {
  __shared__ float s_max[kCeWarps], s_sum[kCeWarps];
  __shared__ float2 part;  // this CTA's (max, sum of exp), read by the whole cluster
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = p.cluster;
  const int seg = cl > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
  const int64_t row = blockIdx.x / cl;
  const int64_t seg_start = seg * p.seg_len;
  const int64_t seg_end = min(p.V, seg_start + p.seg_len);
  const T* x = static_cast<const T*>(p.logits) + row * p.V;
  T* g = p.grad != nullptr ? static_cast<T*>(p.grad) + row * p.V : nullptr;
  constexpr int64_t kCap = static_cast<int64_t>(kCeThreads) * kCeVecs * EPV;
  const bool in_regs = seg_end - seg_start <= kCap;

  Packet<T, EPV> buf[kCeVecs];
  float m_thr = -INFINITY, s_thr = 0.f;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kCeVecs; ++i) {
      const int64_t e = seg_start + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
      if (e < seg_end) load_packet<T, EPV>(buf[i], x + e);
    }
#pragma unroll
    for (int i = 0; i < kCeVecs; ++i) {
      const int64_t e = seg_start + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
#pragma unroll
      for (int k = 0; k < EPV; ++k)
        if (e + k < seg_end) m_thr = fmaxf(m_thr, to_f<T>(buf[i].v[k]));
    }
  } else {
    // streaming pass 1: online (max, sum of exp) per thread
    for (int64_t b = seg_start; b < seg_end; b += kCap) {
#pragma unroll
      for (int i = 0; i < kCeVecs; ++i) {
        const int64_t e = b + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
        if (e < seg_end) {
          Packet<T, EPV> pk;
          load_packet<T, EPV>(pk, x + e);
          float pm = -INFINITY;
#pragma unroll
          for (int k = 0; k < EPV; ++k)
            if (e + k < seg_end) pm = fmaxf(pm, to_f<T>(pk.v[k]));
          const float mn = fmaxf(m_thr, pm);
          if (mn > -INFINITY) {
            s_thr *= __expf(m_thr - mn);
#pragma unroll
            for (int k = 0; k < EPV; ++k)
              if (e + k < seg_end) s_thr += __expf(to_f<T>(pk.v[k]) - mn);
            m_thr = mn;
          }
        }
      }
    }
  }

  // CTA max
  {
    const float wm = warp_max(m_thr);
    if (lane == 0) s_max[warp] = wm;
  }
  __syncthreads();
  float m_cta = s_max[0];
#pragma unroll
  for (int w = 1; w < kCeWarps; ++w) m_cta = fmaxf(m_cta, s_max[w]);

  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kCeVecs; ++i) {
      const int64_t e = seg_start + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
#pragma unroll
      for (int k = 0; k < EPV; ++k)
        if (e + k < seg_end) s_thr += __expf(to_f<T>(buf[i].v[k]) - m_cta);
    }
  } else {
    s_thr = m_thr > -INFINITY ? s_thr * __expf(m_thr - m_cta) : 0.f;
  }
  {
    const float ws = warp_sum(s_thr);
    if (lane == 0) s_sum[warp] = ws;
  }
  __syncthreads();

  float lse;
  if (cl > 1) {
    if (threadIdx.x == 0) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kCeWarps; ++w) s += s_sum[w];
      part = make_float2(m_cta, s);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    float2 q = make_float2(-INFINITY, 0.f);
    if (lane < cl) q = *cg::this_cluster().map_shared_rank(&part, lane);
    const float M = warp_max(q.x);
    const float S = warp_sum(q.x > -INFINITY ? q.y * __expf(q.x - M) : 0.f);
    lse = M + logf(S);
    cluster_arrive_relaxed();  // done with the other CTAs' shared memory
  } else {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kCeWarps; ++w) s += s_sum[w];
    lse = m_cta + logf(s);
  }

  const int64_t tg = p.target[row];
  const int64_t t = tg - p.v_offset;  // the target's column in these logits
  const bool valid = tg != p.ignore_index && t >= 0 && t < p.V;
  grid_dependency_wait();  // n_valid (and the zeroed ticket) come from the preceding count kernel
  float scale = 0.f;
  if (valid) {
    if (p.reduction == FLCE_REDUCTION_MEAN)
      scale = p.grad_scale / static_cast<float>(*p.n_valid);
    else if (p.reduction == FLCE_REDUCTION_SUM)
      scale = p.grad_scale;
    else
      scale = p.grad_scale * (p.grad_out != nullptr ? p.grad_out[row] : 1.f);
  }

  float zt = 0.f;
  bool found = false;  // this thread holds the target logit
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kCeVecs; ++i) {
      const int64_t e = seg_start + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
      if (e < seg_end) {
        if (g == nullptr) {
          find_target<T, EPV>(buf[i], e, valid ? t : -1, zt, found);
        } else {
          grad_packet<T, EPV>(buf[i], e, t, valid, scale, lse, zt, found);
          if (e + EPV <= seg_end) {
            store_packet<T, EPV>(g + e, buf[i]);
          } else {
#pragma unroll
            for (int k = 0; k < EPV; ++k)
              if (e + k < seg_end) g[e + k] = buf[i].v[k];
          }
        }
      }
    }
  } else {
    for (int64_t b = seg_start; b < seg_end; b += kCap) {
#pragma unroll
      for (int i = 0; i < kCeVecs; ++i) {
        const int64_t e = b + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
        if (e < seg_end) {
          Packet<T, EPV> pk;
          load_packet<T, EPV>(pk, x + e);
          if (g == nullptr) {
            find_target<T, EPV>(pk, e, valid ? t : -1, zt, found);
          } else {
            grad_packet<T, EPV>(pk, e, t, valid, scale, lse, zt, found);
            if (e + EPV <= seg_end) {
              store_packet<T, EPV>(g + e, pk);
            } else {
#pragma unroll
              for (int k = 0; k < EPV; ++k)
                if (e + k < seg_end) g[e + k] = pk.v[k];
            }
          }
        }
      }
    }
  }
  if (p.lse_out != nullptr) {  // partials of a vocabulary shard
    if (found) p.zt_out[row] = zt;
    if (seg == 0 && threadIdx.x == 0) {
      p.lse_out[row] = lse;
      if (!valid) p.zt_out[row] = 0.f;
    }
  } else {
    if (found) p.loss_rows[row] = lse - zt;
    if (!valid && seg == 0 && threadIdx.x == 0) p.loss_rows[row] = 0.f;
  }

  if (p.loss_out != nullptr) {
    // sum / mean: the last CTA to finish adds the row losses in a fixed order
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned int ticket = atomicAdd(p.ticket, 1u);
      s_last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      double acc = 0.0;
      for (int64_t i = threadIdx.x; i < p.N; i += kCeThreads) acc += static_cast<double>(__ldcg(p.loss_rows + i));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      __shared__ double s_acc[kCeWarps];
      if (lane == 0) s_acc[warp] = acc;
      __syncthreads();
      if (threadIdx.x == 0) {
        double total = 0.0;
#pragma unroll
        for (int w = 0; w < kCeWarps; ++w) total += s_acc[w];
        if (p.reduction == FLCE_REDUCTION_MEAN) {
          const int nv = *p.n_valid;
          p.loss_out[0] = nv > 0 ? static_cast<float>(total / nv) : __int_as_float(0x7fc00000);
        } else {
          p.loss_out[0] = static_cast<float>(total);
        }
      }
    }
  }
  if (cl > 1) cluster_wait_acquire();  // the other CTAs have finished reading `part`
}

// ---------------------------------------------------------------------------
// Row-ring form, for rows that fit in shared memory (V * sizeof(T) <= 72 KB,
// 16-byte aligned rows): one persistent 1024-thread CTA per SM takes rows
// blockIdx.x, blockIdx.x + gridDim.x, ...; one thread keeps `depth` whole-row
// TMA bulk loads in flight in a shared-memory ring, so the SM streams without
// pause.  Each row is copied from the ring into registers, reduced, and its
// gradient written from the registers with 16-byte stores.
constexpr int kRingThreads = 1024;
constexpr int kRingMaxDepth = 4;
constexpr int64_t kRingSmemBudget = 220 * 1024;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Packet helpers of the row-ring form: a 16-byte vector of 8 bf16 / fp16 or 4 fp32.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T>
__device__ __forceinline__ float vec_max(const uint4& v);
template <>
__device__ __forceinline__ float vec_max<float>(const uint4& v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// bf16: the max of bf16 values is one of them, so it is taken exactly in one
// running packed bf16x2 maximum, converted once at the end.
template <int VPT>
__device__ __forceinline__ float vec_max_all_bf16(const uint4 (&v)[VPT], int limit, int step) {
  __nv_bfloat162 m = __float2bfloat162_rn(-INFINITY);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (i * step < limit) {
      const __nv_bfloat162* w = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
      m = __hmax2(m, __hmax2(__hmax2(w[0], w[1]), __hmax2(w[2], w[3])));
    }
  }
  return fmaxf(__low2float(m), __high2float(m));
}
// fp16: the same running packed maximum in half2
template <int VPT>
__device__ __forceinline__ float vec_max_all_f16(const uint4 (&v)[VPT], int limit, int step) {
  __half2 m = __float2half2_rn(-INFINITY);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (i * step < limit) {
      const __half2* w = reinterpret_cast<const __half2*>(&v[i]);
      m = __hmax2(m, __hmax2(__hmax2(w[0], w[1]), __hmax2(w[2], w[3])));
    }
  }
  return fmaxf(__low2float(m), __high2float(m));
}

// Max over the vectors i of v with i * step < limit.
template <typename T, int VPT>
__device__ __forceinline__ float vec_max_all(const uint4 (&v)[VPT], int limit, int step) {
  if constexpr (std::is_same<T, uint16_t>::value) {
    return vec_max_all_bf16<VPT>(v, limit, step);
  } else if constexpr (std::is_same<T, __half>::value) {
    return vec_max_all_f16<VPT>(v, limit, step);
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
      if (i * step < limit) m = fmaxf(m, vec_max<T>(v[i]));
    return m;
  }
}

// Replaces every element z by exp(z - m) and adds the exponentials into the
// two lanes of `acc`; nmL = -m * log2 e in both lanes.  Packed fp32x2
// arithmetic: one FMA and one add per two elements.
template <typename T>
__device__ __forceinline__ void vec_exp_acc(uint4& v, float2 nmL, float2& acc);
template <>
__device__ __forceinline__ void vec_exp_acc<uint16_t>(uint4& v, float2 nmL, float2& acc) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
  const float2 l2e = make_float2(kLog2e, kLog2e);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 a = __ffma2_rn(make_float2(bf16_lo(w[q]), bf16_hi(w[q])), l2e, nmL);
    const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    acc = __fadd2_rn(acc, e);
    w[q] = pack_bf16x2(e.x, e.y);
  }
}
template <>
__device__ __forceinline__ void vec_exp_acc<__half>(uint4& v, float2 nmL, float2& acc) {
  __half2* w = reinterpret_cast<__half2*>(&v);
  const float2 l2e = make_float2(kLog2e, kLog2e);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 a = __ffma2_rn(__half22float2(w[q]), l2e, nmL);
    const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    acc = __fadd2_rn(acc, e);
    w[q] = __floats2half2_rn(e.x, e.y);
  }
}
template <>
__device__ __forceinline__ void vec_exp_acc<float>(uint4& v, float2 nmL, float2& acc) {
  float2* f = reinterpret_cast<float2*>(&v);
  const float2 l2e = make_float2(kLog2e, kLog2e);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float2 a = __ffma2_rn(f[q], l2e, nmL);
    f[q] = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    acc = __fadd2_rn(acc, f[q]);
  }
}

template <typename T>
__device__ __forceinline__ void vec_scale(uint4& v, float factor);
// bf16 data: exp(z - max) is held in bf16 and the gradient is one packed
// multiply per two elements (the result is stored in bf16 anyway; the factor
// and the product are each rounded once; bf16 has fp32's exponent range).
template <>
__device__ __forceinline__ void vec_scale<uint16_t>(uint4& v, float factor) {
  __nv_bfloat162* w = reinterpret_cast<__nv_bfloat162*>(&v);
  const __nv_bfloat162 f = __float2bfloat162_rn(factor);
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = __hmul2(w[q], f);
}
template <>
__device__ __forceinline__ void vec_scale<__half>(uint4& v, float factor) {
  // packed fp16 multiplies; a factor below fp16's normal range is applied as
  // (factor * 2^15) then an exact 2^-15, so the factor itself never flushes
  const bool tiny = fabsf(factor) < 6.103515625e-05f;
  const __half2 f1 = __float2half2_rn(tiny ? factor * 32768.f : factor);
  const __half2 f2 = __float2half2_rn(tiny ? 1.f / 32768.f : 1.f);
  __half2* w = reinterpret_cast<__half2*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = __hmul2(__hmul2(w[q], f1), f2);
}
template <>
__device__ __forceinline__ void vec_scale<float>(uint4& v, float factor) {
  float2* f = reinterpret_cast<float2*>(&v);
  const float2 f2 = make_float2(factor, factor);
#pragma unroll
  for (int q = 0; q < 2; ++q) f[q] = __fmul2_rn(f[q], f2);
}

// A vector of -inf in the element type.
template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec();
template <>
__device__ __forceinline__ uint4 neg_inf_vec<uint16_t>() {
  return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
}
template <>
__device__ __forceinline__ uint4 neg_inf_vec<__half>() {
  return make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);
}
template <>
__device__ __forceinline__ uint4 neg_inf_vec<float>() {
  return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}

// Rows whose byte length is not a multiple of 16 (an odd vocabulary size):
// TMA copies the 16-byte-aligned range that covers the row (offsets from the
// 16-byte-aligned tensor start), never past the tensor's last whole 16
// bytes; the elements of the neighbouring rows in its first and last vector
// are masked to -inf and never stored.
struct RowSpan {
  uint64_t a0;  // first byte of the covering range
  int nvr;      // vectors in the covering range
  int nld;      // of them, loaded by TMA: nvr, or nvr - 1 at the tensor's end
  int lead;     // elements of the previous row in vector 0
  int tail;     // this row's elements in vector nvr - 1 (1 .. elements per vector)
};

template <typename T>
__device__ __forceinline__ RowSpan row_span(int64_t row, uint64_t row_bytes, uint64_t tail_limit) {
  const uint64_t sb = static_cast<uint64_t>(row) * row_bytes, eb = sb + row_bytes;
  const uint64_t a0 = sb & ~15ull, a1 = (eb + 15) & ~15ull;
  RowSpan r;
  r.a0 = a0;
  r.nvr = static_cast<int>((a1 - a0) >> 4);
  r.nld = static_cast<int>(((a1 < tail_limit ? a1 : tail_limit) - a0) >> 4);
  r.lead = static_cast<int>((sb & 15) / sizeof(T));
  r.tail = (eb & 15) != 0 ? static_cast<int>((eb & 15) / sizeof(T)) : 16 / static_cast<int>(sizeof(T));
  return r;
}

// Elements of v outside [lo, hi) become -inf.
template <typename T>
__device__ __forceinline__ void mask_outside(uint4& v, int lo, int hi) {
  const uint4 ninf = neg_inf_vec<T>();
  T* e = reinterpret_cast<T*>(&v);
  const T* ni = reinterpret_cast<const T*>(&ninf);
#pragma unroll
  for (int k = 0; k < 16 / static_cast<int>(sizeof(T)); ++k)
    if (k < lo || k >= hi) e[k] = ni[k];
}

// The first n elements of a vector read one by one from global memory (the
// tensor's last, partial 16 bytes), the rest -inf.
template <typename T>
__device__ __forceinline__ uint4 load_first_elems(const T* src, int n) {
  uint4 v = neg_inf_vec<T>();
  T* e = reinterpret_cast<T*>(&v);
#pragma unroll
  for (int k = 0; k < 16 / static_cast<int>(sizeof(T)); ++k)
    if (k < n) e[k] = src[k];
  return v;
}

// Stores elements [lo, hi) of v one by one.
template <typename T>
__device__ __forceinline__ void store_elems(T* dst, const uint4& v, int lo, int hi) {
  const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
  for (int k = 0; k < 16 / static_cast<int>(sizeof(T)); ++k)
    if (k >= lo && k < hi) dst[k] = e[k];
}

// Barrier of one thread group (named barrier `id`, `count` threads) that also
// returns whether any of its threads passed cond = true.
__device__ __forceinline__ bool group_sync_or(uint32_t id, uint32_t count, bool cond) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(cond)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Single-launch form: the number of valid targets over all N rows, counted
// by the whole CTA (every CTA does the same), and the out-of-range flag
// (raised by CTA 0).  t_first is target[threadIdx.x] (or anything past N),
// loaded by the caller before it requested the first rows, so that load is
// ahead of them in the memory queue.  All threads of the CTA must call it.
__device__ int cta_count_valid(const CeParams& p, int64_t t_first) {
  if (p.N <= blockDim.x) {  // one target per thread at most: one counting barrier
    bool valid = false, bad = false;
    if (threadIdx.x < p.N && t_first != p.ignore_index) {
      valid = t_first >= 0 && t_first < p.V;
      bad = !valid;
    }
    const int total = __syncthreads_count(valid);
    if (__syncthreads_or(bad) && blockIdx.x == 0 && threadIdx.x == 0 && p.status != nullptr)
      atomicOr(p.status, FLCE_STATUS_BIT_TARGET_RANGE);
    return total;
  }
  __shared__ int s_count;
  if (threadIdx.x == 0) s_count = 0;
  __syncthreads();
  int count = 0;
  bool bad = false;
  // independent loads (up to N / blockDim.x per thread), then one reduction
#pragma unroll 4
  for (int64_t i = threadIdx.x; i < p.N; i += blockDim.x) {
    const int64_t t = i == threadIdx.x ? t_first : __ldg(p.target + i);
    if (t != p.ignore_index) {
      const bool in_range = t >= 0 && t < p.V;
      count += in_range;
      bad |= !in_range;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) count += __shfl_xor_sync(0xffffffffu, count, o);
  if ((threadIdx.x & 31) == 0 && count > 0) atomicAdd(&s_count, count);
  if (__syncthreads_or(bad) && blockIdx.x == 0 && threadIdx.x == 0 && p.status != nullptr)
    atomicOr(p.status, FLCE_STATUS_BIT_TARGET_RANGE);
  return s_count;
}

// Single-launch form: the arrival counter that finds the last CTA needs no
// zeroing beforehand.  Its 64-bit word holds (call nonce, CTAs arrived).  A
// CTA adds 1 and reads back the old word; if it carries this call's tag, its
// count is the CTA's draw.  Otherwise the word is still an older call's (or
// whatever the memory held): the CTA replaces it by (nonce, 1) with a
// compare-and-swap, its draw being 0, unless another CTA installed the tag
// first, in which case it adds again.  No CTA ever waits for another to make
// progress, so nothing assumes that the grid's CTAs run at the same time.
// CTA 0 installs the tag (count 0) when it starts, so that the arrivals
// normally take one atomic each.  The CAS loop only repeats when another CTA
// changed the word meanwhile, at most once per CTA of the call; its bound is
// a safeguard (status timeout bit, and a draw past every valid count).
__device__ __forceinline__ unsigned long long tag_of(unsigned long long nonce) { return nonce << kTagCountBits; }

// `old` is the value atomicAdd(word, 1) returned.
__device__ unsigned int tagged_draw(unsigned long long* word, unsigned long long nonce, unsigned long long old,
                                    int* status) {
  const unsigned long long tag = tag_of(nonce);
  const unsigned long long mask = (1ull << kTagCountBits) - 1;
  if ((old & ~mask) == tag) return static_cast<unsigned int>(old & mask);
  unsigned long long cur = old + 1;  // the word after this CTA's add
  for (int i = 0; i < (1 << 20); ++i) {
    if ((cur & ~mask) == tag) return static_cast<unsigned int>(atomicAdd(word, 1ull) & mask);
    const unsigned long long prev = atomicCAS(word, cur, tag | 1ull);
    if (prev == cur) return 0u;
    cur = prev;
  }
  if (status != nullptr) atomicOr(status, FLCE_STATUS_BIT_TIMEOUT);
  return static_cast<unsigned int>(mask);
}

// Puts this call's tag on the word (count 0) unless it is there already: one
// read and one compare-and-swap whose result is not waited for.  If the swap
// fails, another CTA changed the word first: either it installed the tag, or
// its add hit the old tag and it installs the tag itself (tagged_draw).
__device__ __forceinline__ void tagged_install(unsigned long long* word, unsigned long long nonce) {
  const unsigned long long tag = tag_of(nonce);
  const unsigned long long cur = ld_relaxed_u64(word);
  if ((cur & ~((1ull << kTagCountBits) - 1)) != tag) atomicCAS(word, cur, tag);
}

// Sum / mean: the CTA's loss partial goes to loss_rows[blockIdx.x] and the
// last CTA to arrive adds all partials (lane order, then a fixed shuffle
// tree, so the sum does not depend on which CTA it is) and writes loss_out.
// Arrivals are counted on the zeroed ticket, or in the single-launch form
// on the tagged counter.  Called by every thread after the CTA's
// partial is final; warp 0 does the work.
__device__ void ce_finish_loss(const CeParams& p, float part, int nv) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int grid = static_cast<int>(gridDim.x);
  unsigned int arrived = 0;
  if (lane == 0) {
    p.loss_rows[blockIdx.x] = part;
    __threadfence();
    arrived = p.done_flags == nullptr
                  ? atomicAdd(p.ticket, 1u) + 1u
                  : tagged_draw(p.done_flags, p.nonce, atomicAdd(p.done_flags, 1ull), p.status) + 1u;
  }
  if (__shfl_sync(0xffffffffu, arrived, 0) != static_cast<unsigned int>(grid)) return;
  __threadfence();
  // the lane's partials are loaded together (one memory latency, not one per
  // load), then added in index order (a missing one adds an exact 0)
  constexpr int kBatch = 8;
  float a = 0.f;
  for (int i0 = lane; i0 < grid; i0 += 32 * kBatch) {
    float x[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) x[k] = i0 + 32 * k < grid ? ld_relaxed_f32(p.loss_rows + i0 + 32 * k) : 0.f;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) a += x[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
  if (lane == 0) {
    if (p.reduction == FLCE_REDUCTION_MEAN)
      p.loss_out[0] = nv > 0 ? a / static_cast<float>(nv) : __int_as_float(0x7fc00000);
    else
      p.loss_out[0] = a;
  }
}

// Bytes between the ring's row buffers: a row, or for unaligned rows the
// 16-byte-aligned range that covers it (at most 30 bytes more).
__host__ __device__ constexpr uint32_t ring_buffer_stride(uint32_t row_bytes, bool unaligned) {
  return unaligned ? (row_bytes + 32u + 127u) & ~127u : (row_bytes + 127u) & ~127u;
}

// Two independent groups of kGroupThreads threads share the CTA's ring and
// take alternate rows, each synchronising on its own named barrier, so one
// group's reductions and stores overlap the other's waits.
constexpr int kRingGroups = 2;
constexpr int kGroupThreads = kRingThreads / kRingGroups;
constexpr int kGroupWarps = kGroupThreads / 32;

// The row ring's barriers.  Buffer b has two, and its use u (the u-th load
// into it) completes phase u / 2 of barrier full[2 b + u % 2].  With an odd
// ring depth consecutive uses of a buffer go to different groups, so a group
// may start waiting for use u while use u - 1 (the other group's) is still
// landing; on a single barrier the parity of that wait could not tell the
// two phases apart and the wait would pass early.  On alternating barriers
// the previous phase of the one waited on is use u - 2, which this same
// group has already consumed.
__device__ __forceinline__ uint32_t ring_bar(const uint64_t* full, int bi, int use) {
  return smem_addr(&full[2 * bi + (use & 1)]);
}
__device__ __forceinline__ uint32_t ring_parity(int use) { return static_cast<uint32_t>((use >> 1) & 1); }

template <typename T, int VPT, bool UNAL>
__global__ void __launch_bounds__(kRingThreads, 1) ce_rows_ring_kernel(const CeParams p, int depth) {
  constexpr int EPV = 16 / sizeof(T);
  extern __shared__ __align__(128) uint8_t ring_smem[];
  __shared__ uint64_t full[2 * kRingMaxDepth];  // two per buffer, alternating by use (ring_bar)
  __shared__ int s_issued[kRingMaxDepth];  // loads issued into each buffer so far
  __shared__ float2 s_part[kRingGroups][2][kGroupWarps];  // per warp (max, sum of exp(z - max))
  __shared__ int s_abort;
  __shared__ float s_gsum[kRingGroups], s_gcomp[kRingGroups];  // per group: compensated sum of its row losses
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / kGroupWarps, gwarp = warp % kGroupWarps;
  const int gtid = threadIdx.x % kGroupThreads;
  const uint32_t bar_id = 1 + grp;
  const uint32_t row_bytes = static_cast<uint32_t>(p.V * sizeof(T));
  const uint32_t buf_stride = ring_buffer_stride(row_bytes, UNAL);
  const uint64_t tail_limit = (static_cast<uint64_t>(p.N) * row_bytes) & ~15ull;  // unaligned rows only
  // row ids fit in 32 bits: the host accepts N < 2^28
  const int stride = gridDim.x;
  const int n_rows = static_cast<int>(p.N);
  const int mine = n_rows > static_cast<int>(blockIdx.x) ? (n_rows - 1 - static_cast<int>(blockIdx.x)) / stride + 1 : 0;
  const uint32_t ring_base = smem_addr(ring_smem);
  const int nvec = static_cast<int>(row_bytes / 16);

  if (threadIdx.x == 0) {
    for (int i = 0; i < depth; ++i) {
      mbar_init(smem_addr(&full[2 * i]), 1);
      mbar_init(smem_addr(&full[2 * i + 1]), 1);
      s_issued[i] = 0;
    }
    s_abort = 0;
    for (int q = 0; q < kRingGroups; ++q) s_gsum[q] = s_gcomp[q] = 0.f;
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtl ctl{&s_abort, p.status, 2000000000ull};
  // the first row of each group is requested at once, the rest of the ring
  // once group 0's first row has landed: the first rows of all SMs then
  // share the DRAM bandwidth with fewer other requests and arrive sooner
  const int first = depth < kRingGroups ? depth : kRingGroups;
  // issues row `row` into buffer `bi`; the count is raised first, so a drain
  // that sees it waits for this copy
  auto issue = [&](int bi, int row) {
    volatile int* cnt = s_issued;
    const int use = cnt[bi];
    cnt[bi] = use + 1;
    const uint32_t bar = ring_bar(full, bi, use);
    if constexpr (UNAL) {
      const RowSpan sp = row_span<T>(row, row_bytes, tail_limit);
      const uint32_t bytes = static_cast<uint32_t>(sp.nld) * 16u;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_load(ring_base + bi * buf_stride, static_cast<const uint8_t*>(p.logits) + sp.a0, bytes, bar);
    } else {
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_load(ring_base + bi * buf_stride, static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.V,
                row_bytes, bar);
    }
  };
  // waits (bounded) for the latest copy issued into every buffer (an earlier
  // use of a buffer was consumed before the latest was issued)
  auto drain = [&]() {
    volatile int* cnt = s_issued;
    for (int bi = 0; bi < depth; ++bi) {
      const int c = cnt[bi];
      if (c > 0) mbar_wait_drain(ring_bar(full, bi, c - 1), ring_parity(c - 1), 2000000000ull);
    }
  };
  const int64_t t_first = p.self_count && threadIdx.x < p.N ? __ldg(p.target + threadIdx.x) : 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < first && i < mine; ++i) issue(i, blockIdx.x + i * stride);
    if (blockIdx.x == 0 && p.done_flags != nullptr) tagged_install(p.done_flags, p.nonce);
    if (blockIdx.x == 0 && p.clear_status) *p.status = 0;  // before this CTA flags anything
  }
  const bool full_rows = !UNAL && nvec == VPT * kGroupThreads;  // no vector past the row's end
  int nv = 1;
  if (p.self_count) {
    nv = cta_count_valid(p, t_first);  // while the first rows load
  } else {
    grid_dependency_wait();  // n_valid and the zeroed ticket come from the count kernel
    if (p.reduction == FLCE_REDUCTION_MEAN) nv = *p.n_valid;
  }
  // gradient scale of a valid row (times grad_out[row] for reduction none)
  const float base_scale = p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(nv) : p.grad_scale;

  // this group's rows: j = grp, grp + 2, ...; a row's scalars are loaded
  // before its data is waited for
  int iter = 0;
  int b = grp, use = 0;  // j % depth and j / depth, kept up to date without divisions
  while (b >= depth) {
    b -= depth;
    ++use;
  }
  for (int j = grp; j < mine; j += kRingGroups, ++iter) {
    if (j != grp) {
      b += kRingGroups;
      while (b >= depth) {
        b -= depth;
        ++use;
      }
    }
    const int row = blockIdx.x + j * stride;
    const int64_t t = __ldg(p.target + row);
    const float go = p.grad_out != nullptr ? __ldg(p.grad_out + row) : 1.f;
    // on a timeout the row is computed from whatever is in the buffer and
    // dropped at the group barrier below, which is also the abort vote
    const bool ok = mbar_wait_sleep(ring_bar(full, b, use), ring_parity(use), ctl);
    if (j == 0 && gtid == 0)  // group 0's first row is here: request the rest of the ring
      for (int i = first; i < depth && i < mine; ++i) issue(i, blockIdx.x + i * stride);
    // vectors past the row's end hold -inf: they add nothing to the max or the
    // sum and are not stored, so the row's work below needs no per-vector branch
    uint4 v[VPT];
    const uint4* sbuf = reinterpret_cast<const uint4*>(ring_smem + b * buf_stride);
    RowSpan sp = {0, 0, 0, 0, EPV};  // unaligned rows only
    if constexpr (UNAL) {
      sp = row_span<T>(row, row_bytes, tail_limit);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int vi = i * kGroupThreads + gtid;
        if (vi < sp.nld)
          v[i] = sbuf[vi];
        else if (vi < sp.nvr)  // the tensor's last partial 16 bytes
          v[i] = load_first_elems<T>(
              reinterpret_cast<const T*>(static_cast<const uint8_t*>(p.logits) + sp.a0 + 16ull * vi), sp.tail);
        else
          v[i] = neg_inf_vec<T>();
        if (vi == 0 || vi == sp.nvr - 1) mask_outside<T>(v[i], vi == 0 ? sp.lead : 0, vi == sp.nvr - 1 ? sp.tail : EPV);
      }
    } else if (full_rows) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) v[i] = sbuf[i * kGroupThreads + gtid];
    } else {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int vi = i * kGroupThreads + gtid;
        v[i] = vi < nvec ? sbuf[vi] : neg_inf_vec<T>();
      }
    }
    // where the target sits: its column here, and which thread / vector / lane holds it
    const int64_t tcl = t - p.v_offset;
    const bool valid = t != p.ignore_index && tcl >= 0 && tcl < p.V;
    const int tcol = valid ? static_cast<int>(tcl) : -1;
    const int tel = valid ? (UNAL ? sp.lead : 0) + tcol : -1;  // its element in the buffer
    const int tvec = valid ? tel / EPV : -1;
    const bool own_t = valid && (tvec % kGroupThreads) == gtid;
    // the target logit straight from the ring buffer (one shared load; the
    // buffer is not refilled before this group's barrier), or from global
    // memory in the tensor's last partial 16 bytes
    float zt;
    if constexpr (UNAL) {
      zt = 0.f;
      if (own_t) {
        if (tvec < sp.nld)
          zt = to_f<T>(reinterpret_cast<const T*>(ring_smem + b * buf_stride)[tel]);
        else
          zt = to_f<T>(static_cast<const T*>(p.logits)[static_cast<int64_t>(row) * p.V + tcol]);
      }
    } else {
      zt = own_t ? to_f<T>(reinterpret_cast<const T*>(ring_smem + b * buf_stride)[tcol]) : 0.f;
    }
    // warp max, then exp(z - warp max) in place and its warp sum
    const float mw = warp_max_redux(vec_max_all<T, VPT>(v, VPT, 1));
    const float nm = mw > -INFINITY ? -mw * kLog2e : 0.f;  // a warp past the row's end: all -inf, sum 0
    const float2 nmL = make_float2(nm, nm);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPT; ++i) vec_exp_acc<T>(v[i], nmL, acc);
    const float sw = warp_sum(acc.x + acc.y);
    if (lane == 0) s_part[grp][iter & 1][gwarp] = make_float2(mw, sw);
    // one group barrier per row: it publishes the partials, frees ring buffer
    // b and carries the abort vote
    if (group_sync_or(bar_id, kGroupThreads, !ok)) {
      s_abort = 1;
      if (gtid == 0) drain();  // bulk loads still in flight must land before leaving
      break;
    }
    if (gtid == 0 && j + depth < mine) issue(b, row + depth * stride);
    // every warp combines the group's warp partials itself
    const float2 q = lane < kGroupWarps ? s_part[grp][iter & 1][lane] : make_float2(-INFINITY, 0.f);
    const float M = warp_max_redux(q.x);
    const float S = warp_sum(q.x > -INFINITY ? q.y * ex2_approx((q.x - M) * kLog2e) : 0.f);
    const float lse = M + lg2_approx(S) * kLn2;  // S >= 1: the warp holding M adds exp(0)

    if (p.lse_out != nullptr) {  // partials of a vocabulary shard
      if (own_t) p.zt_out[row] = zt;
      if (gtid == 0) {
        p.lse_out[row] = lse;
        if (!valid) p.zt_out[row] = 0.f;
      }
      continue;
    }
    if (p.loss_out == nullptr) {  // reduction none: the row's loss
      if (own_t) p.loss_rows[row] = lse - zt;
      if (!valid && gtid == 0) p.loss_rows[row] = 0.f;
    }
    if (p.grad != nullptr) {
      const float scale = valid ? (p.reduction == FLCE_REDUCTION_NONE ? base_scale * go : base_scale) : 0.f;
      // softmax = exp(z - warp max) * exp(warp max - M) / S: one multiply per
      // element; the target element is formed again in fp32 from its logit
      const float factor = scale * ex2_approx((mw - M) * kLog2e) * rcp_approx(S);
#pragma unroll
      for (int i = 0; i < VPT; ++i) vec_scale<T>(v[i], factor);
      if constexpr (UNAL) {
        uint8_t* gb = static_cast<uint8_t*>(p.grad) + sp.a0;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int vi = i * kGroupThreads + gtid;
          if (vi >= sp.nvr) continue;
          const int lo = vi == 0 ? sp.lead : 0, hi = vi == sp.nvr - 1 ? sp.tail : EPV;
          if (lo > 0 || hi < EPV)  // a vector shared with a neighbouring row: this row's elements only
            store_elems<T>(reinterpret_cast<T*>(gb + 16ull * vi), v[i], lo, hi);
          else
            __stcs(reinterpret_cast<uint4*>(gb + 16ull * vi), v[i]);
        }
      } else {
        uint4* gvec = reinterpret_cast<uint4*>(static_cast<T*>(p.grad) + static_cast<int64_t>(row) * p.V) + gtid;
        if (full_rows) {
#pragma unroll
          for (int i = 0; i < VPT; ++i) __stcs(gvec + i * kGroupThreads, v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < VPT; ++i)
            if (i * kGroupThreads + gtid < nvec) __stcs(gvec + i * kGroupThreads, v[i]);
        }
      }
      // the target element, formed again in fp32 from its logit, replaces what
      // the vector store above wrote there (same thread, so it lands last)
      if (own_t)
        static_cast<T*>(p.grad)[static_cast<int64_t>(row) * p.V + tcol] = from_f<T>(scale * (__expf(zt - lse) - 1.f));
    }
    // sum / mean: the group adds its rows' losses in row order (ordered
    // across rows by the group barriers), after the row's stores are issued
    if (p.loss_out != nullptr && own_t) {
      const float y = (lse - zt) - s_gcomp[grp];
      const float t2 = s_gsum[grp] + y;
      s_gcomp[grp] = (t2 - s_gsum[grp]) - y;
      s_gsum[grp] = t2;
    }
  }
  // the other group gave up: copies it would have consumed must land first
  if (gtid == 0 && *static_cast<volatile int*>(&s_abort)) drain();

  // sum / mean: the CTA's partial (the per-row losses are not needed), then
  // one CTA adds the partials
  if (p.loss_out != nullptr) {
    __syncthreads();
    float part = 0.f;
    for (int q = 0; q < kRingGroups; ++q) part += s_gsum[q] - s_gcomp[q];
    ce_finish_loss(p, part, nv);
  }
}

template <typename T, int VPT, bool UNAL>
cudaError_t launch_ring_t(const CeParams& p, int depth, int grid, size_t smem, bool pdl, cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(ce_rows_ring_kernel<T, VPT, UNAL>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kRingSmemBudget + 1024));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  CeParams pc = p;
  return cudaLaunchKernelEx(&cfg, ce_rows_ring_kernel<T, VPT, UNAL>, pc, depth);
}

// Streaming form, for rows over 72 KB (16-bit V > 36864, fp32 V > 18432),
// too long for the row ring: persistent 512-thread CTAs, two per SM, take
// rows blockIdx.x, blockIdx.x + gridDim.x, ...; per row, pass 1 reads the row
// from DRAM in steps of 8 vectors per thread, keeping a per-thread online
// (max, sum of exp), and the CTA combines them into the LSE; pass 2 reads
// the row again (an L2 hit: the rows in flight on all SMs take well under
// L2's capacity) and writes the gradient.  DRAM moves each logit once each
// way; the exponentials are computed twice.  Rows that are not whole
// 16-byte vectors use their 16-byte-aligned covering range, masked as in the
// row ring.
constexpr int kStreamThreads = 512;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kStreamU = 8;  // vectors per thread per step

template <typename T, bool UNAL>
__device__ __forceinline__ void stream_load(uint4 (&v)[kStreamU], const uint8_t* logits, const RowSpan& sp, int base,
                                            bool last_use) {
  constexpr int EPV = 16 / sizeof(T);
  const uint4* src = reinterpret_cast<const uint4*>(logits + sp.a0);
#pragma unroll
  for (int i = 0; i < kStreamU; ++i) {
    const int vi = base + i * kStreamThreads + static_cast<int>(threadIdx.x);
    if (vi < sp.nld)
      v[i] = last_use ? __ldcs(src + vi) : src[vi];
    else if (UNAL && vi < sp.nvr)  // the tensor's last partial 16 bytes
      v[i] = load_first_elems<T>(reinterpret_cast<const T*>(logits + sp.a0 + 16ull * vi), sp.tail);
    else
      v[i] = neg_inf_vec<T>();
    if (UNAL && vi < sp.nvr && (vi == 0 || vi == sp.nvr - 1))
      mask_outside<T>(v[i], vi == 0 ? sp.lead : 0, vi == sp.nvr - 1 ? sp.tail : EPV);
  }
}

template <typename T, bool UNAL>
__global__ void __launch_bounds__(kStreamThreads, 2) ce_rows_stream_kernel(const CeParams p) {
  constexpr int EPV = 16 / sizeof(T);
  __shared__ float2 s_part[2][kStreamWarps];  // per warp (max, sum of exp), by row parity
  __shared__ float s_gsum, s_gcomp;           // compensated sum of the CTA's row losses
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t row_bytes = static_cast<uint64_t>(p.V) * sizeof(T);
  const uint64_t tail_limit = (static_cast<uint64_t>(p.N) * row_bytes) & ~15ull;
  const uint8_t* logits = static_cast<const uint8_t*>(p.logits);
  const int64_t t_first = p.self_count && threadIdx.x < p.N ? __ldg(p.target + threadIdx.x) : 0;
  if (threadIdx.x == 0) {
    s_gsum = s_gcomp = 0.f;
    if (blockIdx.x == 0 && p.done_flags != nullptr) tagged_install(p.done_flags, p.nonce);
    if (blockIdx.x == 0 && p.clear_status) *p.status = 0;  // before this CTA flags anything
  }
  int nv = 1;
  if (p.self_count) {
    nv = cta_count_valid(p, t_first);  // (its barriers also publish the zeroed sums)
  } else {
    grid_dependency_wait();  // n_valid and the zeroed ticket come from the count kernel
    if (p.reduction == FLCE_REDUCTION_MEAN) nv = *p.n_valid;
    __syncthreads();
  }

  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.N; row += gridDim.x, parity ^= 1) {
    RowSpan sp;
    if constexpr (UNAL) {
      sp = row_span<T>(row, row_bytes, tail_limit);
    } else {
      sp.a0 = static_cast<uint64_t>(row) * row_bytes;
      sp.nvr = sp.nld = static_cast<int>(row_bytes / 16);
      sp.lead = 0;
      sp.tail = EPV;
    }
    const int64_t t = __ldg(p.target + row);
    const float go = p.grad_out != nullptr ? __ldg(p.grad_out + row) : 1.f;
    const int64_t tcl = t - p.v_offset;
    const bool valid = t != p.ignore_index && tcl >= 0 && tcl < p.V;
    const int tcol = valid ? static_cast<int>(tcl) : -1;
    const int tvec = valid ? (sp.lead + tcol) / EPV : -1;
    const bool own_t = valid && (tvec % kStreamThreads) == static_cast<int>(threadIdx.x);
    // the target logit, read before anything of the row is overwritten
    const float zt = own_t ? to_f<T>(static_cast<const T*>(p.logits)[row * p.V + tcol]) : 0.f;

    // pass 1: online (max, sum of exp(z - max)) per thread
    float m = -INFINITY, sum = 0.f;
    for (int base = 0; base < sp.nvr; base += kStreamThreads * kStreamU) {
      uint4 v[kStreamU];
      stream_load<T, UNAL>(v, logits, sp, base, false);
      const float cm = vec_max_all<T, kStreamU>(v, kStreamU, 1);
      if (cm > m) {
        sum = m > -INFINITY ? sum * ex2_approx((m - cm) * kLog2e) : 0.f;
        m = cm;
      }
      if (m > -INFINITY) {
        const float nm = -m * kLog2e;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kStreamU; ++i) vec_exp_acc<T>(v[i], make_float2(nm, nm), acc);
        sum += acc.x + acc.y;
      }
    }
    // warp, then CTA combine of the (max, sum) pairs
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      const float mm = fmaxf(m, m2);
      if (mm > -INFINITY) {
        sum = (m > -INFINITY ? sum * ex2_approx((m - mm) * kLog2e) : 0.f) +
              (m2 > -INFINITY ? s2 * ex2_approx((m2 - mm) * kLog2e) : 0.f);
        m = mm;
      }
    }
    if (lane == 0) s_part[parity][warp] = make_float2(m, sum);
    __syncthreads();  // one barrier per row: the partials of row parity p are rewritten two rows later
    const float2 q = lane < kStreamWarps ? s_part[parity][lane] : make_float2(-INFINITY, 0.f);
    const float M = warp_max(q.x);
    const float S = warp_sum(q.x > -INFINITY ? q.y * ex2_approx((q.x - M) * kLog2e) : 0.f);
    const float lse = M + logf(S);

    if (p.lse_out != nullptr) {  // partials of a vocabulary shard
      if (own_t) p.zt_out[row] = zt;
      if (threadIdx.x == 0) {
        p.lse_out[row] = lse;
        if (!valid) p.zt_out[row] = 0.f;
      }
      continue;
    }
    if (p.loss_out != nullptr) {  // the CTA's rows' losses in row order (ordered by the barriers)
      if (own_t) {
        const float y = (lse - zt) - s_gcomp;
        const float t2 = s_gsum + y;
        s_gcomp = (t2 - s_gsum) - y;
        s_gsum = t2;
      }
    } else {
      if (own_t) p.loss_rows[row] = lse - zt;
      if (!valid && threadIdx.x == 0) p.loss_rows[row] = 0.f;
    }
    if (p.grad == nullptr) continue;
    float scale = 0.f;
    if (valid) {
      if (p.reduction == FLCE_REDUCTION_MEAN)
        scale = p.grad_scale / static_cast<float>(nv);
      else if (p.reduction == FLCE_REDUCTION_SUM)
        scale = p.grad_scale;
      else
        scale = p.grad_scale * go;
    }
    // pass 2: the gradient scale * exp(z - lse), from the row again
    uint8_t* gb = static_cast<uint8_t*>(p.grad) + sp.a0;
    const float nl = -lse * kLog2e;
    for (int base = 0; base < sp.nvr; base += kStreamThreads * kStreamU) {
      uint4 v[kStreamU];
      stream_load<T, UNAL>(v, logits, sp, base, true);
      float2 dummy = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kStreamU; ++i) {
        vec_exp_acc<T>(v[i], make_float2(nl, nl), dummy);
        vec_scale<T>(v[i], scale);
      }
#pragma unroll
      for (int i = 0; i < kStreamU; ++i) {
        const int vi = base + i * kStreamThreads + static_cast<int>(threadIdx.x);
        if (vi >= sp.nvr) continue;
        const int lo = UNAL && vi == 0 ? sp.lead : 0, hi = UNAL && vi == sp.nvr - 1 ? sp.tail : EPV;
        if (lo > 0 || hi < EPV)  // a vector shared with a neighbouring row: this row's elements only
          store_elems<T>(reinterpret_cast<T*>(gb + 16ull * vi), v[i], lo, hi);
        else
          __stcs(reinterpret_cast<uint4*>(gb + 16ull * vi), v[i]);
      }
    }
    // the target element replaces what the vector store wrote there (same thread)
    if (own_t) static_cast<T*>(p.grad)[row * p.V + tcol] = from_f<T>(scale * (__expf(zt - lse) - 1.f));
  }

  if (p.loss_out != nullptr) {
    __syncthreads();
    ce_finish_loss(p, s_gsum - s_gcomp, nv);
  }
}

template <typename T, bool UNAL>
cudaError_t launch_stream_t(const CeParams& p, int grid, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  CeParams pc = p;
  return cudaLaunchKernelEx(&cfg, ce_rows_stream_kernel<T, UNAL>, pc);
}


template <typename T, int EPV>
cudaError_t launch_ce_t(const CeParams& p, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.N * p.cluster));
  cfg.blockDim = dim3(kCeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  CeParams pc = p;
  return cudaLaunchKernelEx(&cfg, ce_rows_kernel<T, EPV>, pc);
}

// Vocabulary-shard partials of rows of at most kVpPartThreads * 8 16-byte
// vectors (32 KB): one CTA per row, every thread loading all of its vectors
// at once, so the rows of a call are all in flight together, as in a copy;
// then the row maximum and the sum of exp(z - max) (warp, then block), and
// the row's LSE and target logit (0 when the target is not in this shard).
// Rows must be whole 16-byte vectors and 16-byte aligned.
constexpr int kVpPartThreads = 256;
template <typename T, int VPT>
__global__ void __launch_bounds__(kVpPartThreads)
    ce_vp_partials_rows_kernel(const T* __restrict__ logits, const int64_t* __restrict__ target, int64_t N,
                               int64_t V, int64_t v_offset, int64_t ignore_index, float* __restrict__ lse_out,
                               float* __restrict__ zt_out) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int kWarps = kVpPartThreads / 32;
  __shared__ float s_max[kWarps], s_sum[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = V / EPV;
  for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
    const uint4* x = reinterpret_cast<const uint4*>(logits + row * V);
    uint4 u[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t vi = static_cast<int64_t>(i) * kVpPartThreads + threadIdx.x;
      u[i] = vi < nvec ? __ldcs(x + vi) : neg_inf_vec<T>();  // past the row's end: adds nothing
    }
    const float mt = warp_max_redux(vec_max_all<T, VPT>(u, VPT, 1));
    if (lane == 0) s_max[warp] = mt;
    __syncthreads();
    const float m = warp_max_redux(s_max[lane < kWarps ? lane : 0]);  // the row maximum, in every thread
    const float nm = m > -INFINITY ? -m * kLog2e : 0.f;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPT; ++i) vec_exp_acc<T>(u[i], make_float2(nm, nm), acc);
    const float st = warp_sum(acc.x + acc.y);
    if (lane == 0) s_sum[warp] = st;
    __syncthreads();
    if (warp == 0) {
      const float tot = warp_sum(lane < kWarps ? s_sum[lane] : 0.f);
      if (lane == 0) {
        lse_out[row] = m + lg2_approx(tot) * kLn2;
        const int64_t tg = target[row];
        const int64_t tl = tg - v_offset;
        zt_out[row] = (tg != ignore_index && tl >= 0 && tl < V) ? to_f<T>(logits[row * V + tl]) : 0.f;
      }
    }
    __syncthreads();  // s_max / s_sum are rewritten by the next row
  }
}

template <typename T>
cudaError_t launch_vp_partials_rows_t(const void* logits, const int64_t* target, int64_t N, int64_t V,
                                      int64_t v_offset, int64_t ignore_index, float* lse_out, float* zt_out,
                                      cudaStream_t s) {
  const int64_t nvec = V * static_cast<int64_t>(sizeof(T)) / 16;
  const unsigned grid = static_cast<unsigned>(N < (1 << 30) ? N : (1 << 30));
  const T* lg = static_cast<const T*>(logits);
  if (nvec <= 2 * kVpPartThreads)
    ce_vp_partials_rows_kernel<T, 2><<<grid, kVpPartThreads, 0, s>>>(lg, target, N, V, v_offset, ignore_index,
                                                                     lse_out, zt_out);
  else if (nvec <= 4 * kVpPartThreads)
    ce_vp_partials_rows_kernel<T, 4><<<grid, kVpPartThreads, 0, s>>>(lg, target, N, V, v_offset, ignore_index,
                                                                     lse_out, zt_out);
  else
    ce_vp_partials_rows_kernel<T, 8><<<grid, kVpPartThreads, 0, s>>>(lg, target, N, V, v_offset, ignore_index,
                                                                     lse_out, zt_out);
  return cudaGetLastError();
}

}  // namespace

// Vocabulary-shard partials (LSE and target logit per row) by one CTA per
// row, for rows of whole 16-byte vectors, 16-byte aligned, at most 32 KB
// (bf16 [1024, 16384] 14.3 -> 12.2 us against the row ring; on 64 KB rows
// the ring was faster: fp32 [1024, 16384] 18.4 against 20.5 us).
bool vp_partials_rows_fits(int dtype, int64_t V, bool vector_path) {
  const int64_t esz = dtype == FLCE_DTYPE_FP32 ? 4 : 2;
  return vector_path && V * esz <= 8 * kVpPartThreads * 16;
}

cudaError_t launch_vp_partials_rows(const void* logits, int dtype, const int64_t* target, int64_t N, int64_t V,
                                    int64_t v_offset, int64_t ignore_index, float* lse_out, float* zt_out,
                                    cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  prof_begin(s, FLCE_KERNEL_CE_ROWS);
  cudaError_t e;
  if (dtype == FLCE_DTYPE_BF16)
    e = launch_vp_partials_rows_t<uint16_t>(logits, target, N, V, v_offset, ignore_index, lse_out, zt_out, s);
  else if (dtype == FLCE_DTYPE_FP16)
    e = launch_vp_partials_rows_t<__half>(logits, target, N, V, v_offset, ignore_index, lse_out, zt_out, s);
  else
    e = launch_vp_partials_rows_t<float>(logits, target, N, V, v_offset, ignore_index, lse_out, zt_out, s);
  prof_end(s);
  return e;
}

// Elements per CTA held in registers (the segment length the host aims for).
int64_t ce_cta_capacity(int dtype, bool vector_path) {
  const int64_t epv = vector_path ? (dtype == FLCE_DTYPE_FP32 ? 4 : 8) : 1;
  return static_cast<int64_t>(kCeThreads) * kCeVecs * epv;
}

int64_t ce_vector_elems(int dtype, bool vector_path) {
  return vector_path ? (dtype == FLCE_DTYPE_FP32 ? 4 : 8) : 1;
}

// Rows that are not a whole number of 16-byte vectors go to the row-ring
// form too when both pointers are 16-byte aligned and a row has at least 32
// bytes (its covering range then always holds a whole vector TMA can load).
static bool ce_unaligned_ring_ok(int64_t V, int dtype, bool vector_path, bool aligned_ptrs) {
  const int64_t row_bytes = V * (dtype == FLCE_DTYPE_FP32 ? 4 : 2);
  return !vector_path && aligned_ptrs && row_bytes >= 32 && row_bytes <= 72 * 1024;
}

// Rows over 72 KB: the streaming form (16-byte-aligned pointers).
static bool ce_stream_rows_ok(int64_t V, int dtype, bool vector_path, bool aligned_ptrs) {
  const int64_t row_bytes = V * (dtype == FLCE_DTYPE_FP32 ? 4 : 2);
  return (vector_path || aligned_ptrs) && row_bytes > 72 * 1024 && row_bytes <= (int64_t(1) << 30);
}

bool ce_rows_single_launch_ok(int64_t V, int dtype, bool vector_path, bool aligned_ptrs) {
  const int64_t row_bytes = V * (dtype == FLCE_DTYPE_FP32 ? 4 : 2);
  return ((vector_path && row_bytes <= 72 * 1024) || ce_unaligned_ring_ok(V, dtype, vector_path, aligned_ptrs) ||
          ce_stream_rows_ok(V, dtype, vector_path, aligned_ptrs)) &&
         device_sm_count() <= kCeMaxFlags;
}

// Row-ring form when rows fit (see above); 0 when it does not apply.
int ce_ring_depth(int64_t V, int dtype, bool vector_path, bool unaligned) {
  if (!vector_path && !unaligned) return 0;
  const int64_t row_bytes = V * (dtype == FLCE_DTYPE_FP32 ? 4 : 2);
  if (row_bytes > 72 * 1024) return 0;
  int64_t depth = kRingSmemBudget / ring_buffer_stride(static_cast<uint32_t>(row_bytes), unaligned);
  if (depth > kRingMaxDepth) depth = kRingMaxDepth;
  return depth >= 2 ? static_cast<int>(depth) : 0;
}

template <bool UNAL>
static cudaError_t launch_ring(const CeParams& p, int dtype, int depth, int vpt, int grid, size_t smem, bool pdl,
                               cudaStream_t s) {
  if (dtype == FLCE_DTYPE_BF16)
    return vpt <= 2   ? launch_ring_t<uint16_t, 2, UNAL>(p, depth, grid, smem, pdl, s)
           : vpt <= 4 ? launch_ring_t<uint16_t, 4, UNAL>(p, depth, grid, smem, pdl, s)
           : vpt <= 8 ? launch_ring_t<uint16_t, 8, UNAL>(p, depth, grid, smem, pdl, s)
                      : launch_ring_t<uint16_t, 10, UNAL>(p, depth, grid, smem, pdl, s);
  if (dtype == FLCE_DTYPE_FP16)
    return vpt <= 2   ? launch_ring_t<__half, 2, UNAL>(p, depth, grid, smem, pdl, s)
           : vpt <= 4 ? launch_ring_t<__half, 4, UNAL>(p, depth, grid, smem, pdl, s)
           : vpt <= 8 ? launch_ring_t<__half, 8, UNAL>(p, depth, grid, smem, pdl, s)
                      : launch_ring_t<__half, 10, UNAL>(p, depth, grid, smem, pdl, s);
  return vpt <= 2   ? launch_ring_t<float, 2, UNAL>(p, depth, grid, smem, pdl, s)
         : vpt <= 4 ? launch_ring_t<float, 4, UNAL>(p, depth, grid, smem, pdl, s)
         : vpt <= 8 ? launch_ring_t<float, 8, UNAL>(p, depth, grid, smem, pdl, s)
                    : launch_ring_t<float, 10, UNAL>(p, depth, grid, smem, pdl, s);
}

cudaError_t launch_ce_rows(const CeParams& p, int dtype, bool vector_path, bool aligned_ptrs, bool pdl,
                           cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  prof_begin(s, FLCE_KERNEL_CE_ROWS);
  cudaError_t e;
  const bool unal = ce_unaligned_ring_ok(p.V, dtype, vector_path, aligned_ptrs);
  const int depth = ce_ring_depth(p.V, dtype, vector_path, unal);
  if (depth > 0) {
    const int64_t row_bytes = p.V * (dtype == FLCE_DTYPE_FP32 ? 4 : 2);
    // vectors a thread may hold: the row's, or those of its covering range
    const int64_t vecs = unal ? (row_bytes + 14 + 15) / 16 : row_bytes / 16;
    const int vpt = static_cast<int>((vecs + kGroupThreads - 1) / kGroupThreads);
    const size_t smem = static_cast<size_t>(depth) * ring_buffer_stride(static_cast<uint32_t>(row_bytes), unal);
    int grid = device_sm_count();
    if (grid > p.N) grid = static_cast<int>(p.N);
    e = unal ? launch_ring<true>(p, dtype, depth, vpt, grid, smem, pdl, s)
             : launch_ring<false>(p, dtype, depth, vpt, grid, smem, pdl, s);
    prof_end(s);
    return e;
  }
  const int64_t row_bytes = p.V * (dtype == FLCE_DTYPE_FP32 ? 4 : 2);
  // longer rows: the streaming form, two CTAs per SM while the rows they hold
  // in flight (one each) stay well inside L2, else one
  if (ce_stream_rows_ok(p.V, dtype, vector_path, aligned_ptrs)) {
    int grid = device_sm_count() * (row_bytes <= 256 * 1024 ? 2 : 1);
    if (grid > p.N) grid = static_cast<int>(p.N);
    if (dtype == FLCE_DTYPE_BF16)
      e = vector_path ? launch_stream_t<uint16_t, false>(p, grid, pdl, s) : launch_stream_t<uint16_t, true>(p, grid, pdl, s);
    else if (dtype == FLCE_DTYPE_FP16)
      e = vector_path ? launch_stream_t<__half, false>(p, grid, pdl, s) : launch_stream_t<__half, true>(p, grid, pdl, s);
    else
      e = vector_path ? launch_stream_t<float, false>(p, grid, pdl, s) : launch_stream_t<float, true>(p, grid, pdl, s);
    prof_end(s);
    return e;
  }
  if (dtype == FLCE_DTYPE_BF16)
    e = vector_path ? launch_ce_t<uint16_t, 8>(p, pdl, s) : launch_ce_t<uint16_t, 1>(p, pdl, s);
  else if (dtype == FLCE_DTYPE_FP16)
    e = vector_path ? launch_ce_t<__half, 8>(p, pdl, s) : launch_ce_t<__half, 1>(p, pdl, s);
  else
    e = vector_path ? launch_ce_t<float, 4>(p, pdl, s) : launch_ce_t<float, 1>(p, pdl, s);
  prof_end(s);
  return e;
}

}  // namespace flce
