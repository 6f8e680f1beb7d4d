// Cross entropy on materialised logits [N, V] (bf16 or fp32): loss and the
// logits gradient in one pass (liger-kernel 0.0.1 -> 0.1.1 PyPI diff, README
// "Kernels", CrossEntropy item: loss and gradient computed together, the
// gradient optionally replacing the input; DeepSpeed PR #8540 "Changes":
// FP32/FP16/BF16 logits).
//
// HBM-bound design: each row is split into `cluster` contiguous segments,
// one CTA per segment, the CTAs of a row forming a thread-block cluster.  A
// CTA holds its segment in registers (four 16-byte vectors per thread,
// coalesced across the CTA), reduces (max, sum of exp) with warp shuffles,
// and the cluster combines the segments' partials through distributed shared
// memory.  The gradient is then formed from the registers and written once,
// so every logit is read once and written once.  Segments longer than the
// register capacity fall back to a two-read streaming loop.
#include <cooperative_groups.h>
#include <math.h>

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

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ uint16_t from_f<uint16_t>(float v) {
  return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// A packet of EPV consecutive elements (EPV * sizeof(T) == 16 for the vector path).
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

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kCeWarps; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < kCeWarps; ++w) r += red[w];
  return r;
}

template <typename T, int EPV>
__global__ void __launch_bounds__(kCeThreads) ce_rows_kernel(const CeParams p) {
  __shared__ float red[kCeWarps];
  __shared__ float2 part;     // this CTA's (max, sum of exp), read by the cluster
  __shared__ float lse_bcast;

  cg::cluster_group cluster = cg::this_cluster();
  const int seg = static_cast<int>(cluster.block_rank());
  const int64_t row = blockIdx.x / p.cluster;
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
    const float m_cta = block_max(m_thr, red);
#pragma unroll
    for (int i = 0; i < kCeVecs; ++i) {
      const int64_t e = seg_start + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
#pragma unroll
      for (int k = 0; k < EPV; ++k)
        if (e + k < seg_end) s_thr += __expf(to_f<T>(buf[i].v[k]) - m_cta);
    }
    const float s_cta = block_sum(s_thr, red);
    if (threadIdx.x == 0) part = make_float2(m_cta, s_cta);
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
    const float m_cta = block_max(m_thr, red);
    const float s_cta = block_sum(m_thr > -INFINITY ? s_thr * __expf(m_thr - m_cta) : 0.f, red);
    if (threadIdx.x == 0) part = make_float2(m_cta, s_cta);
  }

  // combine the row's segments across the cluster
  cluster.sync();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int r = 0; r < p.cluster; ++r) M = fmaxf(M, cluster.map_shared_rank(&part, r)->x);
    float S = 0.f;
    for (int r = 0; r < p.cluster; ++r) {
      const float2 q = *cluster.map_shared_rank(&part, r);
      if (q.x > -INFINITY) S += q.y * __expf(q.x - M);
    }
    lse_bcast = M + logf(S);
  }
  cluster.sync();  // also keeps every CTA's `part` alive until all have read it
  const float lse = lse_bcast;

  const int64_t t = p.target[row];
  const bool valid = t != p.ignore_index && t >= 0 && t < p.V;
  grid_dependency_wait();  // n_valid comes from the preceding count kernel
  float scale = 0.f;
  if (valid) {
    if (p.reduction == FLCE_REDUCTION_MEAN)
      scale = p.grad_scale / static_cast<float>(*p.n_valid);
    else if (p.reduction == FLCE_REDUCTION_SUM)
      scale = p.grad_scale;
    else
      scale = p.grad_scale * (p.grad_out != nullptr ? p.grad_out[row] : 1.f);
  }
  if (!valid && seg == 0 && threadIdx.x == 0) p.loss_rows[row] = 0.f;

  auto emit = [&](Packet<T, EPV>& pk, int64_t e) {
#pragma unroll
    for (int k = 0; k < EPV; ++k) {
      const float z = to_f<T>(pk.v[k]);
      if (valid && e + k == t) p.loss_rows[row] = lse - z;
      const float d = valid ? scale * (__expf(z - lse) - (e + k == t ? 1.f : 0.f)) : 0.f;
      pk.v[k] = from_f<T>(d);
    }
  };

  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kCeVecs; ++i) {
      const int64_t e = seg_start + static_cast<int64_t>(i * kCeThreads + threadIdx.x) * EPV;
      if (e < seg_end) {
        if (g == nullptr) {
          if (valid && t >= e && t < e + EPV) p.loss_rows[row] = lse - to_f<T>(buf[i].v[t - e]);
        } else {
          emit(buf[i], e);
          if (e + EPV <= seg_end) {
            store_packet<T, EPV>(g + e, buf[i]);
          } else {
            for (int k = 0; k < EPV && e + k < seg_end; ++k) g[e + k] = buf[i].v[k];
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
            if (valid && t >= e && t < e + EPV && t < seg_end) p.loss_rows[row] = lse - to_f<T>(pk.v[t - e]);
          } else {
            emit(pk, e);
            if (e + EPV <= seg_end) {
              store_packet<T, EPV>(g + e, pk);
            } else {
              for (int k = 0; k < EPV && e + k < seg_end; ++k) g[e + k] = pk.v[k];
            }
          }
        }
      }
    }
  }
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

}  // namespace

// Elements per CTA held in registers (the segment length the host aims for).
int64_t ce_cta_capacity(int dtype, bool vector_path) {
  const int64_t epv = vector_path ? (dtype == FLCE_DTYPE_BF16 ? 8 : 4) : 1;
  return static_cast<int64_t>(kCeThreads) * kCeVecs * epv;
}

int64_t ce_vector_elems(int dtype, bool vector_path) {
  return vector_path ? (dtype == FLCE_DTYPE_BF16 ? 8 : 4) : 1;
}

cudaError_t launch_ce_rows(const CeParams& p, int dtype, bool vector_path, bool pdl, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  prof_begin(s, FLCE_KERNEL_CE_ROWS);
  cudaError_t e;
  if (dtype == FLCE_DTYPE_BF16)
    e = vector_path ? launch_ce_t<uint16_t, 8>(p, pdl, s) : launch_ce_t<uint16_t, 1>(p, pdl, s);
  else
    e = vector_path ? launch_ce_t<float, 4>(p, pdl, s) : launch_ce_t<float, 1>(p, pdl, s);
  prof_end(s);
  return e;
}

}  // namespace flce
