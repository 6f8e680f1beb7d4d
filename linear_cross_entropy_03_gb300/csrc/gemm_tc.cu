// Tensor-core contractions of the fused linear cross entropy on sm_103a.
//
// One persistent, warp-specialised kernel template serves the three products
// of a token chunk (torchtune post "Peak Performance, Minimized Memory ...",
// Figure 1 "Fused Linear Cross Entropy", steps 2 and 4):
//
//   forward  (kind 0)  Z_c[C, V]   = H_c[C, H] . W[V, H]^T      A, B K-major
//   grad_H   (kind 1)  dH_c[C, H]  = dZ_c[C, V] . W[V, H]        A K-major, B MN-major
//   grad_W   (kind 2)  dW[V, H]   += dZ_c[C, V]^T . H_c[C, H]    A, B MN-major
//
// Roles inside a CTA (one CTA per SM):
//   warp 0        TMA producer and tile scheduler (atomic tile counter)
//   warp 1        TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2..5    epilogue: tcgen05.ld of the 128 x 256 fp32 accumulator
// Operands arrive by TMA as 64 x 64 bf16 boxes with 128-byte swizzle into a
// 4-stage ring; the accumulator is double-buffered in tensor memory so the
// epilogue of tile i overlaps the mainloop of tile i+1.
//
// The forward epilogue keeps, per row and per 256-column vocabulary tile,
// the running max and sum of exp (an online log-sum-exp), gathers the
// target logit from the fp32 accumulator, and stores the bf16 logits of the
// chunk.  The backward launch puts the long grad_H tiles (K = V) first in its
// queue and the short grad_W tiles (K = C) after them, so the dynamic
// scheduler balances them across SMs; grad_W tiles overwrite (first chunk)
// or add to the fp32 gradient.
#include <math.h>

#include "ptx.cuh"

namespace flce {
namespace {

struct Tile {
  int kind;  // 0 forward, 1 grad_H, 2 grad_W
  int m0, n0, kblocks;
};

__device__ __forceinline__ Tile decode_tile(int mode, int t, const GemmParams& p) {
  Tile ti;
  if (mode == kModeForward) {
    // row tiles in groups of 32 (4096 tokens), vocabulary tiles varying
    // slowest within a group: the hidden rows in use stay resident in L2
    ti.kind = 0;
    const int num_n = p.num_tiles / p.f_num_m;
    const int per_group = 32 * num_n;
    const int grp = t / per_group, r = t % per_group;
    const int gm = min(32, p.f_num_m - grp * 32);
    ti.m0 = (grp * 32 + r % gm) * kBM;
    ti.n0 = (r / gm) * kBN;
    ti.kblocks = p.f_kblocks;
  } else if (t < p.h_tiles) {
    ti.kind = 1;
    ti.m0 = (t % p.h_num_m) * kBM;
    ti.n0 = (t / p.h_num_m) * kBN;
    ti.kblocks = p.h_kblocks;
  } else {
    const int u = t - p.h_tiles;
    ti.kind = 2;
    ti.n0 = (u % p.w_num_n) * kBN;
    ti.m0 = (u / p.w_num_n) * kBM;
    ti.kblocks = p.w_kblocks;
  }
  return ti;
}

// Every lane waits on the barrier; the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void add_bias_32(float (&x)[32], const uint16_t* bias, int lim) {
  if (lim >= 32) {
    const uint4* b4 = reinterpret_cast<const uint4*>(bias);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 u = __ldg(b4 + g);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * g + 2 * i] += bf16_lo(w[i]);
        x[8 * g + 2 * i + 1] += bf16_hi(w[i]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < lim) x[j] += __uint_as_float(static_cast<uint32_t>(__ldg(bias + j)) << 16);
  }
}

__device__ __forceinline__ void store_bf16_32(uint16_t* dst, const float (&x)[32], int lim) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (8 * g < lim) {
      uint4 u;
      u.x = pack_bf16x2(x[8 * g + 0], x[8 * g + 1]);
      u.y = pack_bf16x2(x[8 * g + 2], x[8 * g + 3]);
      u.z = pack_bf16x2(x[8 * g + 4], x[8 * g + 5]);
      u.w = pack_bf16x2(x[8 * g + 6], x[8 * g + 7]);
      *reinterpret_cast<uint4*>(dst + 8 * g) = u;
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_z, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bar_area = smem_raw + (base - raw) + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_area);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* ring_full = tempty + 2;
  uint64_t* ring_empty = ring_full + kTileRing;
  uint64_t* done = ring_empty + kTileRing;
  int* ring = reinterpret_cast<int*>(done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + kTileRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&tfull[a]), 1);
      mbar_init(smem_addr(&tempty[a]), kEpiWarps);
    }
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(smem_addr(&ring_full[i]), 1);
      mbar_init(smem_addr(&ring_empty[i]), 1 + kEpiWarps);
    }
    mbar_init(smem_addr(done), 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_h);
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_z);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------ producer / scheduler
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint64_t pol_stream = l2_policy_evict_first();
      int stage = 0, slot = 0;
      uint32_t phase = 0, rphase = 0;
      uint64_t issued = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait(smem_addr(&ring_empty[slot]), rphase ^ 1u, ctl)) {
          ok = false;
          break;
        }
        int t = static_cast<int>(atomicAdd(p.tile_counter, 1u));
        if (t >= p.num_tiles) t = -1;
        ring[slot] = t;
        mbar_arrive(smem_addr(&ring_full[slot]));
        if (++slot == kTileRing) {
          slot = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile ti = decode_tile(MODE, t, p);
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!mbar_wait(smem_addr(&empty[stage]), phase ^ 1u, ctl)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          const uint32_t sb = sa + kStageBytesA;
          const uint32_t fb = smem_addr(&full[stage]);
          mbar_arrive_expect_tx(fb, kStageBytes);
          const int k0 = kb * kBK;
          if (ti.kind == 0) {
            const int r = static_cast<int>(p.row0) + ti.m0;
            tma_load_2d_hint(sa, &tm_h, fb, k0, r, pol_keep);
            tma_load_2d_hint(sa + kBoxBytes, &tm_h, fb, k0, r + 64, pol_keep);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d_hint(sb + j * kBoxBytes, &tm_w, fb, k0, ti.n0 + 64 * j, pol_stream);
          } else if (ti.kind == 1) {
            tma_load_2d(sa, &tm_z, fb, k0, ti.m0);
            tma_load_2d(sa + kBoxBytes, &tm_z, fb, k0, ti.m0 + 64);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * kBoxBytes, &tm_w, fb, ti.n0 + 64 * j, k0);
          } else {
            tma_load_2d(sa, &tm_z, fb, ti.m0, k0);
            tma_load_2d(sa + kBoxBytes, &tm_z, fb, ti.m0 + 64, k0);
            const int r = static_cast<int>(p.row0) + k0;
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * kBoxBytes, &tm_h, fb, ti.n0 + 64 * j, r);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Drain: every copy still in flight must land before the CTA exits.
        for (int s = 0; s < kStages; ++s) {
          if (issued > static_cast<uint64_t>(s)) {
            const uint64_t uses = (issued - 1 - s) / kStages + 1;
            mbar_wait_drain(smem_addr(&full[s]), static_cast<uint32_t>((uses - 1) & 1u),
                            p.timeout_ns);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, slot = 0, acc = 0;
      uint32_t phase = 0, rphase = 0, aphase = 0;
      for (;;) {
        if (!mbar_wait(smem_addr(&ring_full[slot]), rphase, ctl)) break;
        const int t = ring[slot];
        mbar_arrive(smem_addr(&ring_empty[slot]));
        if (++slot == kTileRing) {
          slot = 0;
          rphase ^= 1u;
        }
        if (t < 0) break;
        const Tile ti = decode_tile(MODE, t, p);
        if (!mbar_wait(smem_addr(&tempty[acc]), aphase ^ 1u, ctl)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        const uint32_t idesc = ti.kind == 0   ? instr_desc_bf16(kBM, kBN, 0, 0)
                               : ti.kind == 1 ? instr_desc_bf16(kBM, kBN, 0, 1)
                                              : instr_desc_bf16(kBM, kBN, 1, 1);
        bool aborted = false;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!mbar_wait(smem_addr(&full[stage]), phase, ctl)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = base + stage * kStageBytes;
          const uint32_t sb = sa + kStageBytesA;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = ti.kind == 2 ? smem_desc(sa + k * 2048, 8192, 1024)
                                             : smem_desc(sa + k * 32, 16, 1024);
            const uint64_t bd = ti.kind == 0 ? smem_desc(sb + k * 32, 16, 1024)
                                             : smem_desc(sb + k * 2048, 8192, 1024);
            mma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(smem_addr(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        mma_commit(smem_addr(&tfull[acc]));
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      // Every MMA issued by this thread must finish before TMEM is freed.
      mma_commit(smem_addr(done));
      mbar_wait_drain(smem_addr(done), 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    int slot = 0, acc = 0;
    uint32_t rphase = 0, aphase = 0;
    for (;;) {
      if (!warp_wait(smem_addr(&ring_full[slot]), rphase, ctl)) break;
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&ring_empty[slot]));
      if (++slot == kTileRing) {
        slot = 0;
        rphase ^= 1u;
      }
      if (t < 0) break;
      const Tile ti = decode_tile(MODE, t, p);
      if (!warp_wait(smem_addr(&tfull[acc]), aphase, ctl)) break;
      tc_fence_after_sync();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      const int rl = q * 32 + lane;

      if (ti.kind == 0) {
        // forward: bias, online log-sum-exp (of the fp32 logits and of their
        // bf16 roundings), target gather, bf16 logits
        const int r = ti.m0 + rl;
        const bool row_ok = r < p.c_len;
        const int ncols = min(kBN, p.V - ti.n0);
        int t_rel = -1;
        if (row_ok) {
          const int64_t tg = p.target[p.row0 + r] - p.v_offset;
          if (tg >= ti.n0 && tg < ti.n0 + ncols) t_rel = static_cast<int>(tg - ti.n0);
        }
        uint16_t* zrow = p.zbuf + static_cast<int64_t>(row_ok ? r : 0) * p.ldz + ti.n0;
        float m_run = -INFINITY, s32 = 0.f, s16 = 0.f;
        for (int c = 0; c < kBN; c += 32) {
          if (c >= ncols) break;
          uint32_t v[32];
          tmem_load_32cols(tbase + c, v);
          tmem_load_wait();
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
          const int lim = ncols - c;
          if (p.bias != nullptr) add_bias_32(x, p.bias + ti.n0 + c, lim);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
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
              s16 += __expf(bf16_lo(pk[i]) - m_new);
            }
            if (2 * i + 1 < lim) {
              s32 += __expf(x[2 * i + 1] - m_new);
              s16 += __expf(bf16_hi(pk[i]) - m_new);
            }
          }
          m_run = m_new;
          if (t_rel >= c && t_rel < c + 32) {
            float zt = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j == t_rel - c) zt = x[j];
            p.tgt_logit[r] = zt;
          }
          if (row_ok) {
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4)
              if (8 * g4 < lim)
                __stcs(reinterpret_cast<uint4*>(zrow + c + 8 * g4),
                       make_uint4(pk[4 * g4], pk[4 * g4 + 1], pk[4 * g4 + 2], pk[4 * g4 + 3]));
          }
        }
        if (row_ok)
          p.partials[static_cast<int64_t>(r) * p.nvt + ti.n0 / kBN] = make_float4(m_run, s32, s16, 0.f);
      } else if (ti.kind == 1) {
        // grad_H rows of the chunk, written once: bf16, or fp32 for a shard's partial
        const int r = ti.m0 + rl;
        const bool row_ok = r < p.c_len;
        const int ncols = min(kBN, p.H - ti.n0);
        const int64_t off = (p.row0 + (row_ok ? r : 0)) * static_cast<int64_t>(p.H) + ti.n0;
        for (int c = 0; c < kBN; c += 32) {
          if (c >= ncols) break;
          uint32_t v[32];
          tmem_load_32cols(tbase + c, v);
          tmem_load_wait();
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
          if (!row_ok) continue;
          if (p.grad_hidden_f32 != nullptr) {
            float4* o4 = reinterpret_cast<float4*>(p.grad_hidden_f32 + off + c);
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4)
              if (c + 4 * g4 < ncols) o4[g4] = make_float4(x[4 * g4], x[4 * g4 + 1], x[4 * g4 + 2], x[4 * g4 + 3]);
          } else {
            store_bf16_32(p.grad_hidden + off + c, x, ncols - c);
          }
        }
      } else {
        // grad_W rows (vocabulary ids), fp32, overwrite or add
        const int vrow = ti.m0 + rl;
        const bool row_ok = vrow < p.V;
        const int ncols = min(kBN, p.H - ti.n0);
        float* out = p.grad_weight + static_cast<int64_t>(row_ok ? vrow : 0) * p.H + ti.n0;
        for (int c = 0; c < kBN; c += 32) {
          if (c >= ncols) break;
          uint32_t v[32];
          tmem_load_32cols(tbase + c, v);
          tmem_load_wait();
          if (row_ok) {
            float4* o4 = reinterpret_cast<float4*>(out + c);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              if (c + 4 * g < ncols) {
                float4 a = make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                       __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
                if (!p.gw_store) {
                  const float4 b = o4[g];
                  a.x += b.x;
                  a.y += b.y;
                  a.z += b.z;
                  a.w += b.w;
                }
                o4[g] = a;
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tempty[acc]));
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

int gemm_max_smem_ok() {
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (configured[dev]) return 1;
  if (cudaFuncSetAttribute(gemm_kernel<kModeForward>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemmSmemBytes) != cudaSuccess)
    return 0;
  if (cudaFuncSetAttribute(gemm_kernel<kModeBackward>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemmSmemBytes) != cudaSuccess)
    return 0;
  configured[dev] = 1;
  return 1;
}

cudaError_t launch_gemm(int mode, const CUtensorMap& tm_h, const CUtensorMap& tm_w,
                        const CUtensorMap& tm_z, const GemmParams& p, int grid, cudaStream_t s) {
  if (!gemm_max_smem_ok()) return cudaErrorInvalidConfiguration;
  prof_begin(s, mode == kModeForward ? FLCE_KERNEL_GEMM_FWD : FLCE_KERNEL_GEMM_BWD);
  if (mode == kModeForward)
    gemm_kernel<kModeForward><<<grid, kGemmThreads, kGemmSmemBytes, s>>>(tm_h, tm_w, tm_z, p);
  else
    gemm_kernel<kModeBackward><<<grid, kGemmThreads, kGemmSmemBytes, s>>>(tm_h, tm_w, tm_z, p);
  const cudaError_t e = cudaGetLastError();
  prof_end(s);
  return e;
}

}  // namespace flce
