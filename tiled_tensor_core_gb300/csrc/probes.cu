// probes.cu — diagnostic kernels behind tkg_debug.h: a TMA swizzled load whose
// raw shared-memory image is copied out, a one-tile tensor-core MMA with
// caller-chosen operands and (for the block-scaled kind) caller-chosen
// tensor-memory contents of the scale regions, and an MMA issue-rate timer.
// Each checks or measures one building block of the GEMM in isolation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "gemm_variants.h"
#include "tkg.h"
#include "tkg_debug.h"

namespace tkg {
tkg_status debug_encode_map(CUtensorMap* out, const void* ptr, uint64_t d0, uint64_t d1, uint64_t pitch, uint32_t b0,
                            uint32_t b1, int swz);
tkg_status debug_device_ready();
}  // namespace tkg

namespace {

using namespace tkg;

constexpr uint64_t kProbeTimeoutNs = 1000000000ull;

struct SwizzleProbeParams {
  CUtensorMap map;
  uint8_t* dst;
  int bytes;
  unsigned int* err;
};

__global__ void __launch_bounds__(32, 1) swizzle_probe_kernel(const __grid_constant__ SwizzleProbeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar;
  __shared__ int ok_flag;
  __shared__ int no_abort;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    no_abort = 0;
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(b, static_cast<uint32_t>(p.bytes));
    tma_load_2d<1>(smem_u32(smem), &p.map, b, 0, 0);
    ok_flag = mbar_wait(b, 0, kProbeTimeoutNs, &no_abort) ? 1 : 0;
    if (!ok_flag) {
      atomicOr(p.err, 1u);
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 50000ull) {
      }
    }
  }
  __syncthreads();
  if (ok_flag)
    for (int i = threadIdx.x; i < p.bytes; i += 32) p.dst[i] = smem[i];
}

struct MmaProbeParams {
  const uint8_t* a;
  const uint8_t* b;
  const uint32_t* sfa;
  const uint32_t* sfb;
  float* d;
  unsigned int* err;
  int kind;
  int n;
  int ksteps;
  int sf_cols[8];
};

constexpr uint32_t kSfaCol = 256;
constexpr uint32_t kSfbCol = 384;

__global__ void __launch_bounds__(128, 1) mma_probe_kernel(const MmaProbeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int ok_flag;
  __shared__ int no_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* sa = smem;               // 128 rows x 128 B
  uint8_t* sb = smem + 128 * 128;   // n rows x 128 B
  if (threadIdx.x == 0) {
    no_abort = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&tmem_slot), 512);
    tmem_relinquish<1>();
  }
  // operand tiles -> shared memory in the 128-byte swizzled K-major layout
  for (int i = threadIdx.x; i < 128 * 8; i += 128) {
    const int r = i >> 3, ch = i & 7;
    const uint4 v = reinterpret_cast<const uint4*>(p.a)[i];
    *reinterpret_cast<uint4*>(sa + swizzle_offset(r * 128 + ch * 16, 128)) = v;
  }
  for (int i = threadIdx.x; i < p.n * 8; i += 128) {
    const int r = i >> 3, ch = i & 7;
    const uint4 v = reinterpret_cast<const uint4*>(p.b)[i];
    *reinterpret_cast<uint4*>(sb + swizzle_offset(r * 128 + ch * 16, 128)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (p.kind == 2) {
    uint32_t wa[8], wb[8];
    const int row = warp * 32 + lane;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      wa[j] = p.sfa[row * 8 + j];
      wb[j] = p.sfb[row * 8 + j];
    }
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    tmem_st_32x32b_x8(tmem + lane_base + kSfaCol, wa);
    tmem_st_32x32b_x8(tmem + lane_base + kSfbCol, wb);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
    for (int ks = 0; ks < p.ksteps; ++ks) {
      const uint64_t ad = sdesc_sw128(a0 + 32u * ks);
      const uint64_t bd = sdesc_sw128(b0 + 32u * ks);
      const uint32_t acc = ks > 0 ? 1u : 0u;
      if (p.kind == 0) {
        mma_bf16<1>(tmem, ad, bd, idesc_dense(kFmtBF16, 128, p.n), acc);
      } else if (p.kind == 1) {
        mma_f8f6f4<1>(tmem, ad, bd, idesc_dense(kFmtE4M3, 128, p.n), acc);
      } else {
        mma_mxf4nvf4<1>(tmem, ad, bd, idesc_mxf4nvf4(128, p.n), tmem + kSfaCol + p.sf_cols[2 * ks],
                        tmem + kSfbCol + p.sf_cols[2 * ks + 1], acc);
      }
    }
    mma_commit_local(smem_u32(&bar));
    ok_flag = mbar_wait(smem_u32(&bar), 0, kProbeTimeoutNs, &no_abort) ? 1 : 0;
    if (!ok_flag) atomicOr(p.err, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (ok_flag) {
    const int row = warp * 32 + lane;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c = 0; c < p.n; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c, r);
      tmem_wait_ld();
      reg_fence(r);
#pragma unroll
      for (int j = 0; j < 32; ++j) p.d[row * p.n + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, 512);
  }
}

unsigned int* probe_err_word() {
  static unsigned int* w = nullptr;
  if (!w) {
    if (cudaMalloc(&w, sizeof(unsigned int)) != cudaSuccess) {
      cudaGetLastError();
      w = nullptr;
    }
  }
  return w;
}

// MMA issue rate: one thread issues `count` tcgen05.mma back to back (1-SM:
// one CTA; 2-SM: a cluster of two, the leader issuing cta_group::2) and the
// elapsed SM cycles until their commit lands are recorded.  Operands rotate
// over 2 stages x 4 K steps of 80 KB shared stages (A 16 KB, B0 and B1 up to
// 32 KB each) filled with 0x38 bytes; for the block-scaled kind both scale
// regions hold e4m3 1.0 (0x38) in every lane.  Patterns: 0 = every MMA
// accumulates into one TMEM accumulator (columns 0..n-1) from (A, B0);
// 1 = pairs (A, B0) -> D0 and (A, B1) -> D1 (columns n..2n-1), the 2x1 tile
// that shares one A between two accumulators; 2 = pattern 1 with the pair's
// first MMA filling the A collector buffer and the second reusing it
// (collector::a::fill / ::lastuse); 3 (block-scaled only) = one accumulator,
// the scale addresses moving like the GEMM's: MMA t of a 4-MMA stage reads A
// scales at slot + 4t and B scales at slot + 16 + 8t, the stage's 48-column
// slot cycling over five slots from column 256; 4..8 = one accumulator, and
// after every 4 MMAs the issuing thread does (part of) the GEMM's per-stage
// synchronisation work on barriers that never hold it up — 4: two mbarrier
// waits (acquire at cluster scope) that have already completed, each
// followed by tcgen05.fence::after_thread_sync, and two tcgen05.commit (to
// every CTA of a pair) to a barrier nobody waits on; 5: the two commits only;
// 6: the two waits only; 7: the two fences only; 8: the two waits with
// acquire at CTA scope only; 10..12 (bf16, one CTA only) = one accumulator
// with the operand forms of an attention P·V product — 10: B MN-major (16 K
// rows of 128 bytes per MMA, N in 64-element blocks 16 KB apart); 11: A read
// from tensor memory (8 columns per MMA from column 256); 12: both; 13 (n =
// 128): groups of 8 alternating between the form of 0 (D at column 0) and
// that of 12 (D at column 128), as the attention kernel issues S and P·V.  Scales
// otherwise at TMEM columns 256 (A) and 272 (B); columns 256..511 all hold
// e4m3 1.0 (bf16 pairs of 0x3838 for the A-from-TMEM patterns).
constexpr int kRateStages = 2;
constexpr int kRateStageBytes = 81920;
constexpr int kRateSmem = kRateStages * kRateStageBytes + 1024;

__device__ unsigned long long g_rate_cycles;

#define TKG_RATE_MMA(CGS, KIND, QUAL)                                                                      \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                                     \
               "tcgen05.mma.cta_group::" CGS ".kind::" KIND QUAL " [%0], %1, %2, %3, p;\n\t}" ::"r"(d),     \
               "l"(ad), "l"(bd), "r"(id), "r"(acc)                                                         \
               : "memory")
#define TKG_RATE_MMA_F4(CGS, QUAL)                                                                         \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"                                     \
               "tcgen05.mma.cta_group::" CGS ".kind::mxf4nvf4.block_scale.scale_vec::4X" QUAL                \
               " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),                                          \
               "l"(ad), "l"(bd), "r"(id), "r"(sfa), "r"(sfb), "r"(acc)                                     \
               : "memory")

// coll: 0 none, 1 collector::a::fill, 2 collector::a::lastuse.  Compile-time
// kind and collector use keep the issuing loop free of branches.
template <int CG, int kind, int coll>
__device__ __forceinline__ void rate_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  if constexpr (CG == 1) {
    if constexpr (kind == 0) {
      if constexpr (coll == 0) TKG_RATE_MMA("1", "f16", "");
      else if constexpr (coll == 1) TKG_RATE_MMA("1", "f16", ".collector::a::fill");
      else TKG_RATE_MMA("1", "f16", ".collector::a::lastuse");
    } else if constexpr (kind == 1) {
      if constexpr (coll == 0) TKG_RATE_MMA("1", "f8f6f4", "");
      else if constexpr (coll == 1) TKG_RATE_MMA("1", "f8f6f4", ".collector::a::fill");
      else TKG_RATE_MMA("1", "f8f6f4", ".collector::a::lastuse");
    } else {
      if constexpr (coll == 0) TKG_RATE_MMA_F4("1", "");
      else if constexpr (coll == 1) TKG_RATE_MMA_F4("1", ".collector::a::fill");
      else TKG_RATE_MMA_F4("1", ".collector::a::lastuse");
    }
  } else {
    if constexpr (kind == 0) {
      if constexpr (coll == 0) TKG_RATE_MMA("2", "f16", "");
      else if constexpr (coll == 1) TKG_RATE_MMA("2", "f16", ".collector::a::fill");
      else TKG_RATE_MMA("2", "f16", ".collector::a::lastuse");
    } else if constexpr (kind == 1) {
      if constexpr (coll == 0) TKG_RATE_MMA("2", "f8f6f4", "");
      else if constexpr (coll == 1) TKG_RATE_MMA("2", "f8f6f4", ".collector::a::fill");
      else TKG_RATE_MMA("2", "f8f6f4", ".collector::a::lastuse");
    } else {
      if constexpr (coll == 0) TKG_RATE_MMA_F4("2", "");
      else if constexpr (coll == 1) TKG_RATE_MMA_F4("2", ".collector::a::fill");
      else TKG_RATE_MMA_F4("2", ".collector::a::lastuse");
    }
  }
}

template <int CG, int kind, int pattern>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int n, int count, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar;
  __shared__ __align__(8) uint64_t sync_bars[2];  // pattern 4: [0] completed once, [1] collects commits
  __shared__ uint32_t slot;
  __shared__ int no_abort;
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  for (int i = threadIdx.x; i < kRateStages * kRateStageBytes / 4; i += 128) {
    uint32_t w = 0x38383838u;
    if constexpr (pattern == 9) {
      // varied operands of moderate magnitude: bf16 in +-[1, 2), e4m3 in +-[1, 2), any e2m1 code
      uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B9u + 0x7F4A7C15u;
      h ^= h >> 15;
      h *= 0x2C1B3C6Du;
      h ^= h >> 12;
      if constexpr (kind == 0) w = (h & 0x807F807Fu) | 0x3F803F80u;
      else if constexpr (kind == 1) w = (h & 0x87878787u) | 0x38383838u;
      else w = h;
    }
    reinterpret_cast<uint32_t*>(smem)[i] = w;
  }
  if (threadIdx.x == 0) {
    no_abort = 0;
    mbar_init(smem_u32(&bar), 1);
    mbar_init(smem_u32(&sync_bars[0]), 1);
    mbar_init(smem_u32(&sync_bars[1]), (1u << 20) - 1);
    fence_mbar_init();
    mbar_arrive_local(smem_u32(&sync_bars[0]));  // phase 0 of [0] complete
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc<CG>(smem_u32(&slot), 512);
    tmem_relinquish<CG>();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) {
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  const uint32_t tmem = slot;
  {
    uint32_t r[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) r[c] = 0x38383838u;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
    for (int c = 0; c < 16; ++c) tmem_st_32x32b_x16(lane_base + 256u + 16u * c, r);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) {
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  if (threadIdx.x == 0 && rank == 0) {
    const uint32_t s0 = smem_u32(smem);
    const uint32_t id = kind == 0   ? idesc_dense(kFmtBF16, 128 * CG, n)
                        : kind == 1 ? idesc_dense(kFmtE4M3, 128 * CG, n)
                                    : idesc_mxf4nvf4(128 * CG, n);
    const unsigned long long t0 = clock64();
    if constexpr (pattern >= 4) {
      constexpr bool kWait = pattern == 4 || pattern == 6, kFence = pattern == 4 || pattern == 7;
      constexpr bool kCommit = pattern == 4 || pattern == 5, kWaitCta = pattern == 8;
      const uint32_t done = smem_u32(&sync_bars[0]), sink = smem_u32(&sync_bars[1]);
      for (int i = 0; i < count; ++i) {
        const int t = i & 3;
        const uint32_t base = s0 + static_cast<uint32_t>(((i >> 2) % kRateStages) * kRateStageBytes) + 32u * t;
        if (t == 0) {
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            // the phase waited on completed before the loop: one try_wait returns true
            if constexpr (kWait) {
              uint32_t okw;
              asm volatile(
                  "{\n\t.reg .pred p;\n\t"
                  "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                  "selp.u32 %0, 1, 0, p;\n\t}"
                  : "=r"(okw)
                  : "r"(done), "r"(0u)
                  : "memory");
              if (!okw) atomicOr(err, 2u);
            }
            if constexpr (kWaitCta) {
              uint32_t okw;
              asm volatile(
                  "{\n\t.reg .pred p;\n\t"
                  "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                  "selp.u32 %0, 1, 0, p;\n\t}"
                  : "=r"(okw)
                  : "r"(done), "r"(0u)
                  : "memory");
              if (!okw) atomicOr(err, 2u);
            }
            if constexpr (kFence) tc_fence_after();
          }
        }
        rate_mma<CG, kind, 0>(tmem, sdesc_sw128(base), sdesc_sw128(base + 16384u), id, tmem + 256u, tmem + 272u,
                              i > 0 ? 1u : 0u);
        if (kCommit && t == 3) {
          if constexpr (CG == 2) {
            mma_commit_pair(sink, 0x3);
            mma_commit_pair(sink, 0x3);
          } else {
            mma_commit_local(sink);
            mma_commit_local(sink);
          }
        }
      }
    } else if constexpr (pattern == 13) {
      // groups of 8 alternate: S-like (A, B K-major in shared memory, D at column 0) and
      // P·V-like (A from tensor memory at column 256, B MN-major, D at column 128)
      static_assert(CG == 1 && kind == 0, "attention operand forms: bf16, one CTA");
      for (int i = 0; i < count; ++i) {
        const uint32_t stage = s0 + static_cast<uint32_t>(((i >> 3) % kRateStages) * kRateStageBytes);
        const uint32_t acc = i >= 16 ? 1u : 0u;
        if (((i >> 3) & 1) == 0) {
          rate_mma<CG, kind, 0>(tmem, sdesc_sw128(stage + 32u * (i & 3)), sdesc_sw128(stage + 16384u + 32u * (i & 3)),
                                id, 0u, 0u, acc);
        } else {
          mma_bf16_ts(tmem + 128u, tmem + 256u + 8u * static_cast<uint32_t>(i & 7),
                      sdesc_sw128_mn(stage + 16384u + 2048u * (i & 7), 16384u), id | (1u << 16), acc);
        }
      }
    } else if constexpr (pattern >= 10) {
      static_assert(CG == 1 && kind == 0, "attention operand forms: bf16, one CTA");
      const uint32_t id_mn = id | (pattern == 11 ? 0u : (1u << 16));
      for (int i = 0; i < count; ++i) {
        const uint32_t stage = s0 + static_cast<uint32_t>(((i >> 3) % kRateStages) * kRateStageBytes);
        const uint64_t bd = pattern == 11 ? sdesc_sw128(stage + 16384u + 32u * (i & 3))
                                          : sdesc_sw128_mn(stage + 16384u + 2048u * (i & 7), 16384u);
        if constexpr (pattern == 10) {
          rate_mma<CG, kind, 0>(tmem, sdesc_sw128(stage + 32u * (i & 3)), bd, id_mn, 0u, 0u, i > 0 ? 1u : 0u);
        } else {
          const uint32_t a_t = tmem + 256u + 8u * static_cast<uint32_t>(i & 7);
          const uint32_t acc = i > 0 ? 1u : 0u;
          mma_bf16_ts(tmem, a_t, bd, id_mn, acc);
        }
      }
    } else if constexpr (pattern == 3) {
      int slot = 0;
      for (int i = 0; i < count; ++i) {
        const int t = i & 3;
        const uint32_t base = s0 + static_cast<uint32_t>(((i >> 2) % kRateStages) * kRateStageBytes) + 32u * t;
        const uint32_t sf = tmem + 256u + 48u * static_cast<uint32_t>(slot);
        rate_mma<CG, kind, 0>(tmem, sdesc_sw128(base), sdesc_sw128(base + 16384u), id, sf + 4u * t, sf + 16u + 8u * t,
                              i > 0 ? 1u : 0u);
        if (t == 3 && ++slot == 5) slot = 0;
      }
    } else if constexpr (pattern == 0 || pattern == 9) {
      for (int i = 0; i < count; ++i) {
        const uint32_t base = s0 + static_cast<uint32_t>(((i >> 2) % kRateStages) * kRateStageBytes) + 32u * (i & 3);
        rate_mma<CG, kind, 0>(tmem, sdesc_sw128(base), sdesc_sw128(base + 16384u), id, tmem + 256u, tmem + 272u,
                              i > 0 ? 1u : 0u);
      }
    } else {
      // pairs sharing a K step (count rounded down to whole pairs)
      constexpr int c1 = pattern == 2 ? 1 : 0, c2 = pattern == 2 ? 2 : 0;
      for (int i = 0; i < count / 2; ++i) {
        const uint32_t base = s0 + static_cast<uint32_t>(((i >> 2) % kRateStages) * kRateStageBytes) + 32u * (i & 3);
        const uint64_t ad = sdesc_sw128(base);
        const uint32_t acc = i > 0 ? 1u : 0u;
        rate_mma<CG, kind, c1>(tmem, ad, sdesc_sw128(base + 16384u), id, tmem + 256u, tmem + 272u, acc);
        rate_mma<CG, kind, c2>(tmem + static_cast<uint32_t>(n), ad, sdesc_sw128(base + 49152u), id, tmem + 256u,
                               tmem + 272u, acc);
      }
    }
    if constexpr (CG == 2)
      mma_commit_pair(smem_u32(&bar), 0x1);
    else
      mma_commit_local(smem_u32(&bar));
    if (mbar_wait(smem_u32(&bar), 0, kProbeTimeoutNs, &no_abort))
      g_rate_cycles = clock64() - t0;
    else
      atomicOr(err, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) {
    cluster_arrive();
    cluster_wait();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, 512);
  }
}

}  // namespace

extern "C" {

tkg_status tkg_debug_tma_swizzle_probe(int s_bytes, const void* src, void* dst, void* stream) {
  if (!(s_bytes == 32 || s_bytes == 64 || s_bytes == 128) || !src || !dst) return TKG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return TKG_ERR_MISALIGNED;
  tkg_status st = debug_device_ready();
  if (st != TKG_OK) return st;
  SwizzleProbeParams p;
  std::memset(&p, 0, sizeof(p));
  st = debug_encode_map(&p.map, src, static_cast<uint64_t>(s_bytes), 64, static_cast<uint64_t>(s_bytes),
                        static_cast<uint32_t>(s_bytes), 64, s_bytes);
  if (st != TKG_OK) return st;
  p.dst = static_cast<uint8_t*>(dst);
  p.bytes = 64 * s_bytes;
  p.err = probe_err_word();
  if (!p.err) return TKG_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.err, 0, sizeof(unsigned int), s) != cudaSuccess) return TKG_ERR_CUDA;
  swizzle_probe_kernel<<<1, 32, 64 * 128 + 1024, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return TKG_ERR_CUDA;
  unsigned int err = 0;
  if (cudaMemcpyAsync(&err, p.err, sizeof(err), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return err ? TKG_ERR_TIMEOUT : TKG_OK;
}

tkg_status tkg_debug_mma_probe(int kind, int n, int ksteps, const void* a_tile, const void* b_tile,
                               const uint32_t* sfa_words, const uint32_t* sfb_words, const int32_t* sf_cols,
                               float* d_out, void* stream) {
  if (kind < 0 || kind > 2 || !(n == 64 || n == 128 || n == 256) || ksteps < 1 || ksteps > 4 || !a_tile ||
      !b_tile || !d_out)
    return TKG_ERR_INVALID_ARG;
  if (kind == 2 && (!sfa_words || !sfb_words || !sf_cols)) return TKG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a_tile) & 15u) || (reinterpret_cast<uintptr_t>(b_tile) & 15u))
    return TKG_ERR_MISALIGNED;
  MmaProbeParams p;
  std::memset(&p, 0, sizeof(p));
  if (kind == 2) {
    for (int i = 0; i < 2 * ksteps; ++i) {
      if (sf_cols[i] < 0 || sf_cols[i] > 7) return TKG_ERR_INVALID_ARG;
      p.sf_cols[i] = sf_cols[i];
    }
  }
  tkg_status st = debug_device_ready();
  if (st != TKG_OK) return st;
  p.a = static_cast<const uint8_t*>(a_tile);
  p.b = static_cast<const uint8_t*>(b_tile);
  p.sfa = sfa_words;
  p.sfb = sfb_words;
  p.d = d_out;
  p.kind = kind;
  p.n = n;
  p.ksteps = ksteps;
  p.err = probe_err_word();
  if (!p.err) return TKG_ERR_CUDA;
  const int smem = 128 * 128 + 256 * 128 + 1024;
  if (cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.err, 0, sizeof(unsigned int), s) != cudaSuccess) return TKG_ERR_CUDA;
  mma_probe_kernel<<<1, 128, smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return TKG_ERR_CUDA;
  unsigned int err = 0;
  if (cudaMemcpyAsync(&err, p.err, sizeof(err), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return err ? TKG_ERR_TIMEOUT : TKG_OK;
}

tkg_status tkg_debug_mma_rate(int kind, int cta_group, int n, int count, int pattern, unsigned long long* cycles,
                              void* stream) {
  if (kind < 0 || kind > 2 || (cta_group != 1 && cta_group != 2) || n < 64 || n > 256 || n % 32 != 0 || count < 1 ||
      count > 65536 || pattern < 0 || pattern > 13 || !cycles)
    return TKG_ERR_INVALID_ARG;
  if (pattern >= 10 && (kind != 0 || cta_group != 1)) return TKG_ERR_INVALID_ARG;
  if (pattern == 13 && n != 128) return TKG_ERR_INVALID_ARG;
  // two accumulators must fit beside the scale columns (256..287) for the block-scaled kind
  if ((pattern == 1 || pattern == 2) && kind == 2 && n != 128) return TKG_ERR_INVALID_ARG;
  if ((pattern == 1 || pattern == 2) && count < 2) return TKG_ERR_INVALID_ARG;  // at least one whole pair
  if (pattern == 3 && kind != 2) return TKG_ERR_INVALID_ARG;
  tkg_status st = debug_device_ready();
  if (st != TKG_OK) return st;
  unsigned int* err = probe_err_word();
  if (!err) return TKG_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(err, 0, sizeof(unsigned int), s) != cudaSuccess) return TKG_ERR_CUDA;
  static const void* const kFns[2][3][14] = {
      {{reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 0>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 1>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 2>), nullptr,
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 4>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 5>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 6>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 7>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 8>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 9>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 10>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 11>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 12>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 0, 13>)},
       {reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 0>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 1>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 2>), nullptr,
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 4>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 5>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 6>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 7>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 8>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 1, 9>), nullptr, nullptr, nullptr, nullptr},
       {reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 0>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 1>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 2>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 3>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 4>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 5>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 6>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 7>), reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 8>),
        reinterpret_cast<const void*>(&mma_rate_kernel<1, 2, 9>), nullptr, nullptr, nullptr, nullptr}},
      {{reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 0>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 1>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 2>), nullptr,
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 4>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 5>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 6>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 7>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 8>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 0, 9>), nullptr, nullptr, nullptr, nullptr},
       {reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 0>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 1>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 2>), nullptr,
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 4>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 5>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 6>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 7>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 8>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 1, 9>), nullptr, nullptr, nullptr, nullptr},
       {reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 0>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 1>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 2>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 3>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 4>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 5>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 6>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 7>), reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 8>),
        reinterpret_cast<const void*>(&mma_rate_kernel<2, 2, 9>), nullptr, nullptr, nullptr, nullptr}}};
  const void* fn = kFns[cta_group - 1][kind][pattern];
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(cta_group), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = kRateSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cta_group);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&n, &count, &err};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  unsigned int e = 0;
  unsigned long long c = 0;
  if (cudaMemcpyAsync(&e, err, sizeof(e), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&c, g_rate_cycles, sizeof(c), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  if (e) return TKG_ERR_TIMEOUT;
  *cycles = c;
  return TKG_OK;
}

}  // extern "C"
