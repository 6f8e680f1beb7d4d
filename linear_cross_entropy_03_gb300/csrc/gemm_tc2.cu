// Tensor-core contractions of the fused linear cross entropy, CTA-pair form.
//
// The three products (torchtune post "Peak Performance, Minimized Memory
// ...", Figure 1 "Fused Linear Cross Entropy", steps 2 and 4): the chunk
// projection Z = H_c W^T with its cross-entropy epilogue, grad_H = dZ W and
// grad_W += dZ^T H_c, on 256 x 256 tiles computed by a pair of CTAs on two
// SMs with tcgen05.mma.cta_group::2: each CTA stages 128 rows of A and 128
// columns of B in its own shared memory, the pair's tensor cores read both
// halves, and each CTA's tensor memory receives its 128 rows of the
// accumulator.  Per SM this halves the operand bytes that TMA writes into
// shared memory and the MMA reads back out, which limits a one-CTA
// 128 x 256 form (measured at 71 % tensor-pipe busy against 83 % here).
//
// Roles (same in both CTAs unless noted):
//   warp 0    TMA producer for this CTA's halves; in the leader CTA (rank 0)
//             also the tile scheduler, which writes every tile id into both
//             CTAs' rings
//   warp 1    TMEM allocation for the pair; in the leader, the MMA issuer
//   warps 2.. epilogue of this CTA's 128 accumulator rows: 4 warps (one per
//             TMEM lane quarter), or 8 (two per quarter, each half of the
//             columns) in forward launches with a short k loop
// Operand bytes of both CTAs complete on the leader's stage barriers; the
// leader's tcgen05.commit arrives on the matching barriers of both CTAs.
#include <cuda_fp16.h>
#include <math.h>

#include "ptx.cuh"

namespace flce {
namespace {

constexpr int kHalf = 128;                       // rows of A / columns of B per CTA
// The operand ring (192 KB) holds 6 stages of 32 KB (A half + B half), or,
// while wide grad_H tiles run, 4 stages of 48 KB (A half + two B halves).
// Producer and MMA issuer switch layouts at the same tile; the producer first
// waits until the MMAs have released every stage.
constexpr int kWide = 2 * kBN;  // columns of a wide grad_H tile: 512
constexpr int kRingSlots = 6;
constexpr int kNarrowStageBytes = 2 * kHalf * kBK * 2;
constexpr int kWideStages = 4;
constexpr int kWideStageBytes = 3 * kHalf * kBK * 2;
static_assert(kWideStages * kWideStageBytes <= kRingSlots * kNarrowStageBytes, "wide layout exceeds the ring");
// Per CTA, 16 KB of staging for the epilogue's coalesced stores: 2 KB per
// warp with 8 epilogue warps, 4 KB with 4 (store_rows16 / store_rows32f).
constexpr int kEpiStageBytes = 16384;
static_assert(kEpiStageBytes / 4 >= 32 * 32 * 4, "backward launches (4 epilogue warps) stage 32 x 32 fp32 per warp");
static_assert(kEpiStageBytes / 8 >= 32 * 32 * 2, "8-warp forward launches stage 32 x 32 16-bit values per warp");
// ring, barrier area (1 KB), epilogue staging, 1 KB of alignment slack
constexpr int kGemm2SmemBytes = kRingSlots * kNarrowStageBytes + 1024 + kEpiStageBytes + 1024;
// tile-ring consumers: leader MMA issuer + epilogue warps, peer producer + epilogue warps
constexpr int ring_consumers(int epi_warps) { return 1 + epi_warps + 1 + epi_warps; }
constexpr int gemm_threads(int epi_warps) { return 64 + 32 * epi_warps; }
constexpr int kHGroup = 8;  // row tiles per group in the grad_H tile order
constexpr int kFGroup = 16;  // row tiles per group in the forward tile order
#ifndef FLCE_W_GROUP
#define FLCE_W_GROUP 8
#endif
constexpr int kWGroup = FLCE_W_GROUP;  // hidden-column tiles per group in the grad_W tile order

struct Tile2 {
  int kind;  // 0 forward, 1 grad_H, 2 grad_W
  int m0, n0, kblocks;
  int kb0, slice;  // first k block of the tile's K range (split grad_H tiles), and its slice
};

// Pair tiles: 256 rows of M, 256 columns of N.
__device__ __forceinline__ Tile2 decode_tile2(int mode, int t, const GemmParams& p) {
  Tile2 ti;
  ti.kb0 = 0;
  ti.slice = 0;
  if (mode == kModeForward) {
    // row tiles in groups of kFGroup (4096 tokens), vocabulary tiles varying
    // slowest within a group: the hidden rows in use stay resident in L2
    ti.kind = 0;
    const int num_n = p.num_tiles / p.f_num_m;
    const int per_group = kFGroup * num_n;
    const int grp = t / per_group, r = t % per_group;
    const int gm = min(kFGroup, p.f_num_m - grp * kFGroup);
    ti.m0 = (grp * kFGroup + r % gm) * 256;
    ti.n0 = (r / gm) * kBN;
    ti.kblocks = p.f_kblocks * (p.nseg > 1 ? p.nseg : 1);
  } else if (t < p.h_tiles) {
    // grad_H tiles (K = V, long) in groups of kHGroup row tiles, columns
    // varying within a group: the pairs running at once share fewer rows of
    // dZ and columns of W, so fewer of them are re-read from DRAM
    // (split along K: the slices of one output tile lie h_base tiles apart)
    ti.kind = 1;
    const int split = p.h_split > 1 ? p.h_split : 1;
    const int base = split > 1 ? p.h_base : p.h_tiles;
    const int b = t % base;
    ti.slice = t / base;
    const int per_group = kHGroup * (base / p.h_num_m);
    const int grp = b / per_group, r = b % per_group;
    const int gm = min(kHGroup, p.h_num_m - grp * kHGroup);
    ti.m0 = (grp * kHGroup + r % gm) * 256;
    ti.n0 = (r / gm) * kWide;
    const int kbs = split > 1 ? p.h_kbs : p.h_kblocks;
    ti.kb0 = ti.slice * kbs;
    ti.kblocks = (min(p.h_kblocks, ti.kb0 + kbs) - ti.kb0) * (p.nseg > 1 ? p.nseg : 1);
  } else {
    // grad_W tiles in groups of kWGroup hidden-column tiles, vocabulary rows
    // varying slowest within a group: the columns of H_c in use stay in L2
    // while dZ streams through once per group
    const int u = t - p.h_tiles;
    ti.kind = 2;
    const int per_group = kWGroup * (p.num_tiles - p.h_tiles) / p.w_num_n;
    const int grp = u / per_group, r = u % per_group;
    const int gn = min(kWGroup, p.w_num_n - grp * kWGroup);
    ti.n0 = (grp * kWGroup + r % gn) * kBN;
    ti.m0 = (r / gn) * 256;
    ti.kblocks = p.w_kblocks * (p.nseg > 1 ? p.nseg : 1);
  }
  return ti;
}

__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait_cluster(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// 16-bit operand values: bf16, or fp16 when F16.  A packed pair holds the
// element of the lower column in its low half.
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t w) {
  return F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))) : bf16_lo(w);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t w) {
  return F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))) : bf16_hi(w);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if (F16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  return pack_bf16x2(lo, hi);
}

constexpr float kLog2eF = 1.4426950408889634f;

template <bool F16>
__device__ __forceinline__ void add_bias32(float (&x)[32], const uint16_t* bias, int lim) {
  if (lim >= 32) {
    const uint4* b4 = reinterpret_cast<const uint4*>(bias);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 u = __ldg(b4 + g);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * g + 2 * i] += lo16<F16>(w[i]);
        x[8 * g + 2 * i + 1] += hi16<F16>(w[i]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < lim) x[j] += lo16<F16>(static_cast<uint32_t>(__ldg(bias + j)));
  }
}

// The epilogue holds one accumulator row per lane; stored as it is, every
// warp store would write 32 rows 16 bytes each.  These two store a warp's 32
// rows x 32 columns through its staging buffer instead: each lane writes its
// row's 16-byte pieces, then reads back pieces of other rows so that each
// store instruction covers whole 64- or 128-byte row segments.  The pieces'
// slots are XOR-swizzled so that both the row-wise writes and the
// column-wise reads touch eight different 16-byte bank groups per phase.
//
// 16-bit values (pk[i]: columns 2i, 2i + 1 of the lane's row); row r of the
// 32 goes to row0 + r * ld; rows >= nrows and columns >= lim are skipped.
__device__ __forceinline__ void store_rows16(uint4* stage, const uint32_t (&pk)[16], uint16_t* row0, int64_t ld,
                                             int nrows, int c, int lim, int lane) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    stage[lane * 4 + (k ^ ((lane >> 1) & 3))] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
  __syncwarp();
  const int k = lane & 3;  // this lane's 16-byte piece: columns 8k .. 8k + 7
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = (lane >> 2) + 8 * j;
    const uint4 val = stage[r * 4 + (k ^ ((r >> 1) & 3))];
    if (r < nrows && 8 * k < lim) __stcs(reinterpret_cast<uint4*>(row0 + r * ld + c + 8 * k), val);
  }
  __syncwarp();  // the buffer is rewritten by the next chunk
}

// fp32 values (a[k]: columns 4k .. 4k + 3 of the lane's row): streamed to
// memory (kStoreStream), added with vector reductions (kStoreAdd), or
// stored to stay in L2 for a kernel that reads them next (kStoreKeep).
constexpr int kStoreStream = 0, kStoreAdd = 1, kStoreKeep = 2;
__device__ __forceinline__ void store_rows32f(float4* stage, const float4 (&a)[8], float* row0, int64_t ld, int nrows,
                                              int c, int lim, int lane, int mode) {
#pragma unroll
  for (int k = 0; k < 8; ++k) stage[lane * 8 + (k ^ (lane & 7))] = a[k];
  __syncwarp();
  const int k = lane & 7;  // this lane's 16-byte piece: columns 4k .. 4k + 3
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = (lane >> 3) + 4 * j;
    const float4 val = stage[r * 8 + (k ^ (r & 7))];
    if (r < nrows && 4 * k < lim) {
      float4* dst = reinterpret_cast<float4*>(row0 + r * ld + c + 4 * k);
      if (mode == kStoreAdd)  // one fire-and-forget add per element and launch: the L2 does the read-add-write
        red_add_f32x4(dst, val);
      else if (mode == kStoreKeep)
        __stcg(dst, val);
      else
        __stcs(dst, val);
    }
  }
  __syncwarp();
}

// Epilogue of one tile for this warp's 32 accumulator rows (`rl` = row
// within the pair tile of this thread) and its PC columns from c_lo (with 8
// epilogue warps two share each TMEM lane quarter, one per half of the
// columns; with 4, PC is the whole tile).
// F16: fp16 operands (chunk logits and grad_hidden in fp16); SPLIT: fp32
// operands as bf16 hi + lo planes (chunk logits stored exactly, as the two
// halves of their fp32 bits; fp32 bias); out_scale multiplies the backward
// products.
template <bool F16, bool SPLIT, int PC>
__device__ __forceinline__ void epilogue_tile(const Tile2& ti, const GemmParams& p, uint32_t tbase, int rl,
                                              int c_lo, float out_scale, int64_t row_target, uint8_t* stage) {
  const int lane = threadIdx.x & 31;
  const int wrow = rl - lane;  // the warp's first row within the pair tile
  if (ti.kind == 0) {
    const int r = ti.m0 + rl;
    const bool row_ok = r < p.c_len;
    const int nrows = min(32, p.c_len - (ti.m0 + wrow));  // valid rows of the warp's 32
    uint16_t* zrow0 = p.zbuf + static_cast<int64_t>(ti.m0 + wrow) * p.ldz + ti.n0;
    const int ncols = min(kBN, p.V - ti.n0);
    int t_rel = -1;
    if (row_ok) {
      const int64_t tg = row_target - p.v_offset;
      if (tg >= ti.n0 && tg < ti.n0 + ncols) t_rel = static_cast<int>(tg - ti.n0);
    }
    float m_run = -INFINITY, s32 = 0.f, s16 = 0.f;
    for (int c = c_lo; c < c_lo + PC; c += 32) {
      if (c >= ncols) break;
      uint32_t v[32];
      tmem_load_32cols(tbase + c, v);
      tmem_load_wait();
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
      const int lim = ncols - c;
      if (SPLIT) {
        if (p.bias_f32 != nullptr) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < lim) x[j] += __ldg(p.bias_f32 + ti.n0 + c + j);
        }
      } else if (p.bias != nullptr) {
        add_bias32<F16>(x, p.bias + ti.n0 + c, lim);
      }
      // the 16-bit logits (SPLIT: the upper halves of the fp32 bits, the
      // lower halves going to the second plane)
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = SPLIT ? __byte_perm(__float_as_uint(x[2 * i]), __float_as_uint(x[2 * i + 1]), 0x7632)
                      : pack16<F16>(x[2 * i], x[2 * i + 1]);
      if (lim >= 32) {
        // a whole chunk: no per-column bounds, a three-input maximum tree,
        // exp(z - m) as ex2 of one fused multiply-add, packed fp32x2
        // arithmetic for two columns at a time, two independent sums
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(x[4 * i], x[4 * i + 1], fmax3(x[4 * i + 2], x[4 * i + 3], m_run));
        const float m_new = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        const float corr = ex2_approx((m_run - m_new) * kLog2eF);  // 0 on the first chunk (m_run = -inf)
        const float nmL = -m_new * kLog2eF;
        const float2 l2e = make_float2(kLog2eF, kLog2eF), nm2 = make_float2(nmL, nmL);
        float2 a32 = make_float2(0.f, 0.f), a16 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 t = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), l2e, nm2);
          a32 = __fadd2_rn(a32, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
          if (!SPLIT) {
            const float2 u = __ffma2_rn(make_float2(lo16<F16>(pk[i]), hi16<F16>(pk[i])), l2e, nm2);
            a16 = __fadd2_rn(a16, make_float2(ex2_approx(u.x), ex2_approx(u.y)));
          }
        }
        s32 = s32 * corr + (a32.x + a32.y);
        s16 = s16 * corr + (a16.x + a16.y);
        m_run = m_new;
      } else {
        float cmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < lim) cmax = fmaxf(cmax, x[j]);
        const float m_new = fmaxf(m_run, cmax);
        const float corr = __expf(m_run - m_new);
        s32 *= corr;
        s16 *= corr;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (2 * i < lim) {
            s32 += __expf(x[2 * i] - m_new);
            if (!SPLIT) s16 += __expf(lo16<F16>(pk[i]) - m_new);
          }
          if (2 * i + 1 < lim) {
            s32 += __expf(x[2 * i + 1] - m_new);
            if (!SPLIT) s16 += __expf(hi16<F16>(pk[i]) - m_new);
          }
        }
        m_run = m_new;
      }
      if (t_rel >= c && t_rel < c + 32) {
        float zt = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == t_rel - c) zt = x[j];
        p.tgt_logit[r] = zt;
      }
      store_rows16(reinterpret_cast<uint4*>(stage), pk, zrow0, p.ldz, nrows, c, lim, lane);
      if (SPLIT) {  // the lower halves of the fp32 bits, one plane further
        uint32_t lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          lo[i] = __byte_perm(__float_as_uint(x[2 * i]), __float_as_uint(x[2 * i + 1]), 0x5410);
        store_rows16(reinterpret_cast<uint4*>(stage), lo, zrow0 + p.z_plane, p.ldz, nrows, c, lim, lane);
      }
    }
    if (SPLIT) s16 = s32;  // the gradient is formed from the exact fp32 logits
    if (row_ok && ti.n0 + c_lo < p.V)
      p.partials[static_cast<int64_t>(r) * p.nvt + (ti.n0 + c_lo) / PC] = make_float4(m_run, s32, s16, 0.f);
  } else if (ti.kind == 1) {
    const int nrows = min(32, p.c_len - (ti.m0 + wrow));  // valid rows of the warp's 32
    const int ncols = min(kBN, p.H - ti.n0);
    const int64_t row0 = ti.m0 + wrow;
    const int64_t off = (p.row0 + row0) * static_cast<int64_t>(p.H) + ti.n0;
    // a K slice of a split tile: its fp32 partial sums, scaled like the output
    float* part0 = p.h_split > 1 ? p.gh_part + ti.slice * p.gh_part_ld + row0 * p.H + ti.n0 : nullptr;
    for (int c = c_lo; c < c_lo + PC; c += 32) {
      if (c >= ncols) break;
      uint32_t v[32];
      tmem_load_32cols(tbase + c, v);
      tmem_load_wait();
      if (part0 != nullptr || p.grad_hidden_f32 != nullptr) {
        // fp32: a K slice's partial sums, or the fp32 output (fp32 operands, a shard's partial)
        const float sc = part0 != nullptr ? out_scale : 1.f;
        float4 a[8];
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)
          a[g4] = make_float4(sc * __uint_as_float(v[4 * g4]), sc * __uint_as_float(v[4 * g4 + 1]),
                              sc * __uint_as_float(v[4 * g4 + 2]), sc * __uint_as_float(v[4 * g4 + 3]));
        store_rows32f(reinterpret_cast<float4*>(stage), a, part0 != nullptr ? part0 : p.grad_hidden_f32 + off, p.H,
                      nrows, c, ncols - c, lane, kStoreKeep);
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack16<F16>(out_scale * __uint_as_float(v[2 * i]), out_scale * __uint_as_float(v[2 * i + 1]));
        store_rows16(reinterpret_cast<uint4*>(stage), pk, p.grad_hidden + off, p.H, nrows, c, ncols - c, lane);
      }
    }
  } else {
    const int nrows = min(32, p.V - (ti.m0 + wrow));  // valid vocabulary rows of the warp's 32
    const int ncols = min(kBN, p.H - ti.n0);
    float* out0 = p.grad_weight + static_cast<int64_t>(ti.m0 + wrow) * p.H + ti.n0;
    for (int c = c_lo; c < c_lo + PC; c += 32) {
      if (c >= ncols) break;
      uint32_t v[32];
      tmem_load_32cols(tbase + c, v);
      tmem_load_wait();
      float4 a[8];
#pragma unroll
      for (int g = 0; g < 8; ++g)
        a[g] = make_float4(out_scale * __uint_as_float(v[4 * g]), out_scale * __uint_as_float(v[4 * g + 1]),
                           out_scale * __uint_as_float(v[4 * g + 2]), out_scale * __uint_as_float(v[4 * g + 3]));
      store_rows32f(reinterpret_cast<float4*>(stage), a, out0, p.H, nrows, c, ncols - c, lane,
                    p.gw_store ? kStoreStream : kStoreAdd);
    }
  }
}

template <int MODE, int EW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads(EW), 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_h2,
                 const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_z2,
                 const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bar_area = smem_raw + (base - raw) + kRingSlots * kNarrowStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_area);
  uint64_t* empty = full + kRingSlots;
  uint64_t* tfull = empty + kRingSlots;
  uint64_t* tempty = tfull + 2;
  uint64_t* ring_full = tempty + 2;
  uint64_t* ring_empty = ring_full + kTileRing;
  uint64_t* done = ring_empty + kTileRing;
  int* ring = reinterpret_cast<int*>(done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + kTileRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&tfull[a]), 1);
      mbar_init(smem_addr(&tempty[a]), 2 * EW);
    }
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(smem_addr(&ring_full[i]), 1);
      mbar_init(smem_addr(&ring_empty[i]), ring_consumers(EW));
    }
    mbar_init(smem_addr(done), 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_h);
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_z);
    if (p.nseg > 1) {
      tma_prefetch_desc(&tm_h2);
      tma_prefetch_desc(&tm_w2);
      tma_prefetch_desc(&tm_z2);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------ producer (+ scheduler in the leader)
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint64_t pol_stream = l2_policy_evict_first();
      int stage = 0, slot = 0;
      uint32_t rphase = 0;
      uint32_t fills = 0;  // bit s: parity of the number of fills of stage s
      bool wide = false;   // ring layout in use
      bool ok = true;
      while (ok) {
        int t;
        if (leader) {
          if (!mbar_wait_cluster(smem_addr(&ring_empty[slot]), rphase ^ 1u, ctl)) {
            ok = false;
            break;
          }
          t = static_cast<int>(atomicAdd(p.tile_counter, 1u));
          if (t >= p.num_tiles) t = -1;
          ring[slot] = t;
          st_shared_cluster_u32(map_to_cta(smem_addr(&ring[slot]), 1), static_cast<uint32_t>(t));
          mbar_arrive(smem_addr(&ring_full[slot]));
          mbar_arrive_cluster(map_to_cta(smem_addr(&ring_full[slot]), 1));
        } else {
          if (!mbar_wait_cluster(smem_addr(&ring_full[slot]), rphase, ctl)) {
            ok = false;
            break;
          }
          t = ring[slot];
          mbar_arrive_remote(map_to_cta(smem_addr(&ring_empty[slot]), 0));
        }
        if (++slot == kTileRing) {
          slot = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile2 ti = decode_tile2(MODE, t, p);
        const int mh = ti.m0 + kHalf * static_cast<int>(rank);  // this CTA's rows of A
        const int nh = ti.n0 + kHalf * static_cast<int>(rank);  // this CTA's columns of B
        if ((ti.kind == 1) != wide) {
          // the other layout's stages overlap these: wait until the MMAs have
          // released every stage (the latest fill of each)
          for (int s2 = 0; s2 < kRingSlots && ok; ++s2)
            ok = mbar_wait_cluster(smem_addr(&empty[s2]), ((fills >> s2) & 1u) ^ 1u, ctl);
          if (!ok) break;
          wide = ti.kind == 1;
          stage = 0;
        }
        const int nst = wide ? kWideStages : kRingSlots;
        const uint32_t sbytes = wide ? kWideStageBytes : kNarrowStageBytes;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!mbar_wait_cluster(smem_addr(&empty[stage]), ((fills >> stage) & 1u) ^ 1u, ctl)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * sbytes;
          const uint32_t sb = sa + kHalf * kBK * 2;
          const uint32_t fb = map_to_cta(smem_addr(&full[stage]), 0);
          // a wide grad_H tile whose second half lies wholly past H (H <= 256)
          // loads and multiplies its first half only
          const bool half1 = ti.kind == 1 && ti.n0 + kBN < p.H;
          if (leader)
            mbar_arrive_expect_tx(smem_addr(&full[stage]), (half1 ? 6 : 4) * kBoxBytes * 2);
          // k block kb: with split fp32 operands the three segments
          // (hi.hi, hi.lo, lo.hi) of each 64-wide k slice follow one another,
          // so the hi tile a segment re-reads is still in L2
          const int ns = p.nseg > 1 ? p.nseg : 1;
          const int seg = kb % ns;
          const int k0 = (ti.kb0 + kb / ns) * kBK;
          // segment 0 multiplies A hi by B hi, 1 A hi by B lo, 2 A lo by B hi;
          // H is A of the forward and B of grad_W, W is B, dZ is A
          const bool h_lo = ti.kind == 0 ? seg == 2 : seg == 1;
          const CUtensorMap* m_h = h_lo ? &tm_h2 : &tm_h;
          const CUtensorMap* m_w = seg == 1 ? &tm_w2 : &tm_w;
          const CUtensorMap* m_z = seg == 2 ? &tm_z2 : &tm_z;
          if (ti.kind == 0) {
            // the chunk's hidden rows are re-read by every vocabulary tile; the
            // weight is streamed once per chunk
            const int r = static_cast<int>(p.row0) + mh;
            tma_load_2d_pair_hint(sa, m_h, fb, k0, r, pol_keep);
            tma_load_2d_pair_hint(sa + kBoxBytes, m_h, fb, k0, r + 64, pol_keep);
            tma_load_2d_pair_hint(sb, m_w, fb, k0, nh, pol_stream);
            tma_load_2d_pair_hint(sb + kBoxBytes, m_w, fb, k0, nh + 64, pol_stream);
          } else if (ti.kind == 1) {
            // wide tile: this CTA's 128 columns of each 256-column half of B
            tma_load_2d_pair(sa, m_z, fb, k0, mh);
            tma_load_2d_pair(sa + kBoxBytes, m_z, fb, k0, mh + 64);
            tma_load_2d_pair(sb, m_w, fb, nh, k0);
            tma_load_2d_pair(sb + kBoxBytes, m_w, fb, nh + 64, k0);
            if (half1) {
              tma_load_2d_pair(sb + 2 * kBoxBytes, m_w, fb, nh + kBN, k0);
              tma_load_2d_pair(sb + 3 * kBoxBytes, m_w, fb, nh + kBN + 64, k0);
            }
          } else {
            // grad_W: every tile re-reads the chunk's hidden rows (kept in L2);
            // each dZ column panel serves only the tiles of one vocabulary row
            // running side by side (streamed)
            tma_load_2d_pair_hint(sa, m_z, fb, mh, k0, pol_stream);
            tma_load_2d_pair_hint(sa + kBoxBytes, m_z, fb, mh + 64, k0, pol_stream);
            const int r = static_cast<int>(p.row0) + k0;
            tma_load_2d_pair_hint(sb, m_h, fb, nh, r, pol_keep);
            tma_load_2d_pair_hint(sb + kBoxBytes, m_h, fb, nh + 64, r, pol_keep);
          }
          fills ^= 1u << stage;
          if (++stage == nst) stage = 0;
        }
      }
      if (!ok && leader) {
        // Drain: copies still in flight must land before the pair exits (the
        // latest fill of each stage; a stage never filled passes at once).
        for (int s2 = 0; s2 < kRingSlots; ++s2)
          mbar_wait_cluster_drain(smem_addr(&full[s2]), ((fills >> s2) & 1u) ^ 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && leader) {
      int stage = 0, slot = 0, acc = 0;
      uint32_t rphase = 0, aphase = 0;
      uint32_t uses = 0;  // bit s: parity of the number of times stage s was consumed
      bool wide = false;
      for (;;) {
        if (!mbar_wait(smem_addr(&ring_full[slot]), rphase, ctl)) break;
        const int t = ring[slot];
        mbar_arrive(smem_addr(&ring_empty[slot]));
        if (++slot == kTileRing) {
          slot = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile2 ti = decode_tile2(MODE, t, p);
        // a wide grad_H tile takes both accumulator buffers (all 512 columns),
        // one per 256-column half, in the order the epilogue frees them
        const int nbuf = ti.kind == 1 ? 2 : 1;
        int bufs[2] = {0, 0};
        bool got = true;
        for (int q = 0; q < nbuf; ++q) {
          if (!mbar_wait_cluster(smem_addr(&tempty[acc]), aphase ^ 1u, ctl)) {
            got = false;
            break;
          }
          bufs[q] = acc;
          if (++acc == 2) {
            acc = 0;
            aphase ^= 1u;
          }
        }
        if (!got) break;
        if ((ti.kind == 1) != wide) {  // same layout switch as the producer
          wide = ti.kind == 1;
          stage = 0;
        }
        const int nst = wide ? kWideStages : kRingSlots;
        const uint32_t sbytes = wide ? kWideStageBytes : kNarrowStageBytes;
        tc_fence_after_sync();
        const bool half1 = ti.kind == 1 && ti.n0 + kBN < p.H;  // as the producer decides
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(bufs[0] * kBN);
        const uint32_t d_tmem1 = tmem_base + static_cast<uint32_t>(bufs[1] * kBN);
        uint32_t idesc = ti.kind == 0   ? instr_desc_bf16(256, kBN, 0, 0)
                         : ti.kind == 1 ? instr_desc_bf16(256, kBN, 0, 1)
                                        : instr_desc_bf16(256, kBN, 1, 1);
        if (p.in_fp16) idesc &= ~((7u << 7) | (7u << 10));  // A and B format fields: fp16 (0)
        bool aborted = false;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!mbar_wait_cluster(smem_addr(&full[stage]), (uses >> stage) & 1u, ctl)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = base + stage * sbytes;
          const uint32_t sb = sa + kHalf * kBK * 2;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = ti.kind == 2 ? smem_desc(sa + k * 2048, 8192, 1024)
                                             : smem_desc(sa + k * 32, 16, 1024);
            const uint64_t bd = ti.kind == 0 ? smem_desc(sb + k * 32, 16, 1024)
                                             : smem_desc(sb + k * 2048, 8192, 1024);
            if (ti.kind == 1) {  // wide tile: the two 256-column halves share A
              mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
              if (half1)  // (a second half wholly past H is neither loaded nor multiplied)
                mma_bf16_pair(d_tmem1, ad, smem_desc(sb + 2 * kBoxBytes + k * 2048, 8192, 1024), idesc,
                              (kb | k) != 0 ? 1u : 0u);
            } else {
              mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          mma_commit_pair(smem_addr(&empty[stage]), 0x3);
          uses ^= 1u << stage;
          if (++stage == nst) stage = 0;
        }
        if (aborted) break;
        for (int q = 0; q < nbuf; ++q) mma_commit_pair(smem_addr(&tfull[bufs[q]]), 0x3);
      }
      // Every MMA must finish (it reads both CTAs' shared memory and writes
      // both CTAs' tensor memory) before either CTA frees anything.
      mma_commit_pair(smem_addr(done), 0x3);
      mbar_wait_cluster_drain(smem_addr(done), 0, p.timeout_ns);
    } else if (lane == 0) {
      mbar_wait_cluster_drain(smem_addr(done), 0, p.timeout_ns + 1000000000ull);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;                                // TMEM lane quarter (hardware rule: warp % 4)
    constexpr int PC = part_cols(EW);
    const int c_lo = ((warp - 2) / 4) * PC;               // this warp's columns of every tile
    uint8_t* stage = bar_area + 1024 + (warp - 2) * (kEpiStageBytes / EW);  // this warp's staging buffer
    // fp16: the chunk's dZ was stored divided by the rows' common scale
    const float out_scale = (MODE == kModeBackward && p.in_fp16)
                                ? uniform_scale(p.reduction, p.grad_scale, p.n_valid, p.gmax)
                                : 1.f;
    const uint32_t leader_tempty0 = map_to_cta(smem_addr(&tempty[0]), 0);
    const uint32_t leader_tempty1 = map_to_cta(smem_addr(&tempty[1]), 0);
    int slot = 0, acc = 0;
    uint32_t rphase = 0, aphase = 0;
    for (;;) {
      if (!warp_wait_cluster(smem_addr(&ring_full[slot]), rphase, ctl)) break;
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_to_cta(smem_addr(&ring_empty[slot]), 0));
      if (++slot == kTileRing) {
        slot = 0;
        rphase ^= 1u;
      }
      if (t < 0) break;
      Tile2 ti = decode_tile2(MODE, t, p);
      // a wide grad_H tile arrives as two 256-column halves, one per buffer
      const int nbuf = ti.kind == 1 ? 2 : 1;
      const int rl = kHalf * static_cast<int>(rank) + q * 32 + lane;
      // forward: the row's target, loaded while the accumulator is computed
      const int64_t row_target =
          (MODE == kModeForward && ti.m0 + rl < p.c_len) ? __ldg(p.target + p.row0 + ti.m0 + rl) : 0;
      bool ok = true;
      for (int half = 0; half < nbuf; ++half) {
        if (!warp_wait_cluster(smem_addr(&tfull[acc]), aphase, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tbase =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
        if (p.in_fp16)
          epilogue_tile<true, false, PC>(ti, p, tbase, rl, c_lo, out_scale, row_target, stage);
        else if (p.nseg > 1)
          epilogue_tile<false, true, PC>(ti, p, tbase, rl, c_lo, 1.f, row_target, stage);
        else
          epilogue_tile<false, false, PC>(ti, p, tbase, rl, c_lo, 1.f, row_target, stage);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acc == 0 ? leader_tempty0 : leader_tempty1);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
        ti.n0 += kBN;
      }
      if (!ok) break;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its pair may still touch its memory
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

int gemm2_max_smem_ok() {
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (configured[dev]) return 1;
  if (cudaFuncSetAttribute(gemm2_kernel<kModeForward, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemm2SmemBytes) != cudaSuccess)
    return 0;
  if (cudaFuncSetAttribute(gemm2_kernel<kModeForward, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemm2SmemBytes) != cudaSuccess)
    return 0;
  if (cudaFuncSetAttribute(gemm2_kernel<kModeBackward, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemm2SmemBytes) != cudaSuccess)
    return 0;
  configured[dev] = 1;
  return 1;
}

// grid: number of CTAs, even (two per tile pair).
cudaError_t launch_gemm2(int mode, const CUtensorMap& tm_h, const CUtensorMap& tm_w, const CUtensorMap& tm_z,
                         const GemmParams& p, int grid, cudaStream_t s, const CUtensorMap* tm_h2,
                         const CUtensorMap* tm_w2, const CUtensorMap* tm_z2) {
  if (!gemm2_max_smem_ok()) return cudaErrorInvalidConfiguration;
  prof_begin(s, mode == kModeForward ? FLCE_KERNEL_GEMM_FWD : FLCE_KERNEL_GEMM_BWD);
  const CUtensorMap& h2 = tm_h2 ? *tm_h2 : tm_h;
  const CUtensorMap& w2 = tm_w2 ? *tm_w2 : tm_w;
  const CUtensorMap& z2 = tm_z2 ? *tm_z2 : tm_z;
  if (mode == kModeForward && p.epi_warps == 8)
    gemm2_kernel<kModeForward, 8><<<grid, gemm_threads(8), kGemm2SmemBytes, s>>>(tm_h, tm_w, tm_z, h2, w2, z2, p);
  else if (mode == kModeForward)
    gemm2_kernel<kModeForward, 4><<<grid, gemm_threads(4), kGemm2SmemBytes, s>>>(tm_h, tm_w, tm_z, h2, w2, z2, p);
  else
    gemm2_kernel<kModeBackward, 4><<<grid, gemm_threads(4), kGemm2SmemBytes, s>>>(tm_h, tm_w, tm_z, h2, w2, z2, p);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

}  // namespace flce
