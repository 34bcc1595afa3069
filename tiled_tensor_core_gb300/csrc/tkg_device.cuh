// tkg_device.cuh — sm_103a device primitives for the tiled GEMM, as inline PTX.
//
//   * shared-tile swizzle (the 32/64/128-byte XOR layouts of the ThunderKittens
//     shared tiles — paper summary "Shared Memory Tiles: Automated Swizzling")
//   * mbarrier ring primitives with bounded waits (the arrive / expect
//     synchronisation of the LCSF template — "Synchronization Primitives:
//     Arrive and Expect")
//   * TMA tile loads and stores ("Asynchronous I/O: Unified Interface over
//     cp.async and TMA"; tensor maps built on the host)
//   * tcgen05 tensor-memory allocation, MMA issue, commit and TMEM loads (the
//     Blackwell tensor-core path named on the Russian DSL page, "Compute и
//     memory movement", and the 2-SM MMA of "Swizzling и memory layout")
//   * the L2-aware tile order ("Block Launch Order and L2 Cache Reuse", Table 3)
#pragma once

#include <cstdint>
#include <cuda.h>

namespace tkg {

// ---------------------------------------------------------------- host+device

// XOR swizzle of a byte offset inside an S-byte-swizzled shared tile whose base
// is aligned to 8*S bytes: the 16-byte chunk index (bits 4..) is XOR-ed with
// the 128-byte row index (bits 7..) modulo S/16.  S = 0 means no swizzle.
__host__ __device__ constexpr uint32_t swizzle_offset(uint32_t off, uint32_t s_bytes) {
  return s_bytes == 0 ? off : off ^ (((off % (s_bytes * 8u)) >> 7) << 4);
}

// Widest swizzle (128, 64 or 32 bytes) that a row of `row_bytes` bytes is a
// multiple of; chosen at compile time for every shared tile.
__host__ __device__ constexpr uint32_t select_swizzle(uint32_t row_bytes) {
  return row_bytes % 128u == 0 ? 128u : row_bytes % 64u == 0 ? 64u : row_bytes % 32u == 0 ? 32u : 0u;
}

// L2-aware tile order.  Output tiles are visited in super-rows of `group_m`
// tile-rows: inside a super-row the M index runs fastest, then N, then the
// next super-row — the {G, N, M/G} order.  Linear id t in [0, tiles_m*tiles_n).
struct TileOrder {
  int tiles_m, tiles_n, group_m;
  __host__ __device__ __forceinline__ void coord(int t, int& tm, int& tn) const {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int rows_here = (tiles_m - first_m) < group_m ? (tiles_m - first_m) : group_m;
    const int r = t - g * per_group;
    tm = first_m + r % rows_here;
    tn = r / rows_here;
  }
};

#if defined(__CUDACC__)

// ---------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Acquire load at GPU scope (pairs with a fence + atomic on the writing side).
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory object in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive on a barrier given by a shared::cluster address (own or peer CTA),
// with the instruction's default semantics (release at CTA scope).  Every use
// signals "my tensor-memory accesses are done" and is preceded by the
// matching tcgen05.wait and tcgen05.fence::before_thread_sync, which order
// those accesses; a cluster-scope release would add nothing to that and on
// sm_103a it costs about a microsecond per arrival.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// Acquire at CTA scope (the instruction's default).  What the pipeline's
// waits order is tensor-core and TMA (async-proxy) work, which the tcgen05
// fences and the transaction counts already order; a cluster-scope acquire
// would add nothing and costs the MMA-issuing thread more per wait
// (tkg_debug_mma_rate patterns 6 and 8).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test, letting the hardware suspend the thread for up to 20 us while
// the phase is incomplete (it resumes when the phase completes): for waits
// that usually last long, so that the waiting warps stop competing with the
// MMA-issuing warp for issue slots and barrier accesses.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` to complete.  Every wait of
// the pipeline goes through here: after `timeout_ns` of waiting (or once some
// other role has raised the CTA's abort flag) it gives up and returns false.
// kSuspend: use the suspending test (long waits of non-critical roles).
template <bool kSuspend = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* abort_flag) {
  auto test = [&]() { return kSuspend ? mbar_try_wait_suspend(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (test()) return true;
    if ((n & (kSuspend ? 15u : 255u)) == 0) {
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > timeout_ns || *abort_flag) return false;
    }
  }
}

// Arrive on a barrier at a shared::cluster address (own or peer CTA) and add
// `bytes` to the transactions its current phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar), "r"(bytes)
               : "memory");
}

// ---------------------------------------------------------------- proxies / fences

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- launch overlap and tile scheduling

// Programmatic dependent launch.  `griddep_wait` returns once every grid this
// one was made dependent on has completed and its memory operations are
// visible (immediately when there is none); `griddep_launch_dependents` lets
// the grid launched after this one start its CTAs (and their prologue) on
// SMs this grid no longer occupies, once every CTA of this grid has said so.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Cluster launch control: ask the hardware to cancel the launch of a cluster
// of this grid that has not started yet.  The 16-byte answer is written to the
// shared-memory address `resp` of every CTA of the issuing cluster and
// completes 16 transaction bytes on the barrier at offset `bar` of each.
__device__ __forceinline__ void clc_try_cancel_multicast(uint32_t resp, uint32_t bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.multicast::cluster::all.b128 "
      "[%0], [%1];" ::"r"(resp),
      "r"(bar)
      : "memory");
}

// Decode an answer: the x index of the first CTA of the cancelled cluster, or
// -1 if the request cancelled nothing (every cluster has started).
__device__ __forceinline__ int clc_first_ctaid_x(uint4 r) {
  const uint64_t lo = static_cast<uint64_t>(r.x) | (static_cast<uint64_t>(r.y) << 32);
  const uint64_t hi = static_cast<uint64_t>(r.z) | (static_cast<uint64_t>(r.w) << 32);
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b128 q;\n\t"
      "mov.b128 q, {%2, %3};\n\t"
      "mov.u32 %1, 0;\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, q;\n\t}"
      : "=r"(ok), "=r"(x)
      : "l"(lo), "l"(hi)
      : "memory");
  return ok ? static_cast<int>(x) : -1;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// 2-D tiled load into this CTA's shared memory, completing `bar_cluster`
// (a shared::cluster barrier address; for CG == 2 it may be the peer's).
template <int CG>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar_cluster, int32_t x,
                                            int32_t y) {
  if constexpr (CG == 1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
  }
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}
// 3-D tiled load into this CTA's shared memory (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- tcgen05

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warpgroup register split: every thread of the warpgroup executes the same one of these; the
// warpgroups' new counts together may not exceed the registers the block was launched with.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Shared-memory matrix descriptor for a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (8-row, 1024-byte atoms):
//   start address >> 4 in bits 0-13, leading byte offset (unused for swizzled
//   K-major, 16 B) in 16-29, stride byte offset 1024 B (next 8-row group) in
//   32-45, descriptor version 1 in 46-48, base offset 0, swizzle mode
//   "128-byte" (2) in bits 61-63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Shared-memory descriptor for 32 (or more) rows of 16 bytes stored one after
// another with no swizzle: 8-row groups of 128 bytes at a 128-byte stride (the
// source of a tcgen05.cp of 32 rows x 128 bits).
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Shared-memory descriptor for an MN-major operand tile with the 128-byte
// swizzle: each row of 128 bytes holds 64 consecutive M (or N) elements of one
// K index, 8 rows (8 K indices) form a 1024-byte atom.  `mn_stride` = bytes
// from one 64-element M/N block to the next (leading byte offset), 1024 B from
// one 8-row K group to the next (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, dense kinds (kind::f16, kind::f8f6f4): D fp32
// (bits 4-5 = 1), A/B format in bits 7-9 / 10-12, both K-major, N>>3 in bits
// 17-22, M>>4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_dense(uint32_t ab_format, int M, int N) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// Instruction descriptor, block-scaled kind::mxf4nvf4: A/B = E2M1 (1), scale
// type UE4M3 (bit 23 = 0), K-major, N>>3 in bits 17-22, M>>7 in bits 27-28,
// scale-factor ids 0.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 7) << 27);
}

constexpr uint32_t kFmtBF16 = 1;  // kind::f16 operand format
constexpr uint32_t kFmtE4M3 = 0;  // kind::f8f6f4 operand format

// Use of the tensor core's A collector buffer by a dense MMA
// (tcgen05.mma ... .collector::a::*): kCollFill reads A from shared memory and
// keeps it in the buffer, kCollLastUse takes A from the buffer (no shared-memory
// read) and then releases it.  Two consecutive MMAs with the same A descriptor
// issued fill / lastuse read A once.
constexpr int kCollNone = 0, kCollFill = 1, kCollLastUse = 2;

#define TKG_MMA_DENSE_ASM(HEAD)                                                                        \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t" HEAD " [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem), \
               "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)                                    \
               : "memory")

// D[tmem] (+)= A · Bᵀ, bf16 operands (kind::f16), fp32 accumulator; `accumulate` = 0 overwrites D.
template <int CG, int COLL = kCollNone>
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  static_assert(CG == 2 || COLL == kCollNone, "collector use is built for the CTA-pair form");
  if constexpr (CG == 1)
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::1.kind::f16");
  else if constexpr (COLL == kCollFill)
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::2.kind::f16.collector::a::fill");
  else if constexpr (COLL == kCollLastUse)
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::2.kind::f16.collector::a::lastuse");
  else
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::2.kind::f16");
}

// The same with e4m3 operands (kind::f8f6f4; the formats are in the instruction descriptor).
template <int CG, int COLL = kCollNone>
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  static_assert(CG == 2 || COLL == kCollNone, "collector use is built for the CTA-pair form");
  if constexpr (CG == 1)
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::1.kind::f8f6f4");
  else if constexpr (COLL == kCollFill)
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::2.kind::f8f6f4.collector::a::fill");
  else if constexpr (COLL == kCollLastUse)
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::2.kind::f8f6f4.collector::a::lastuse");
  else
    TKG_MMA_DENSE_ASM("tcgen05.mma.cta_group::2.kind::f8f6f4");
}
#undef TKG_MMA_DENSE_ASM

template <int CG>
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// bf16 MMA with A read from tensor memory (M rows at lanes 0..M-1, two K
// elements per 32-bit column, the even one in the low half) and B from shared
// memory; one CTA.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Make `bar` (own CTA) track completion of all prior tcgen05 async ops of this thread.
__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Same, arriving on the barrier at the same offset in every CTA of `mask` (CTA pair).
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Shared -> tensor memory copy of 32 rows x 128 bits into lanes taddr.lane + r
// of every 32-lane quarter (row r of the source to lane r of each quarter),
// four consecutive columns from taddr.col; with cta_group::2, issued by the
// leader, each CTA of the pair copies from its own shared memory into its own
// tensor memory.  Runs on the tensor pipe in issue order with this thread's
// MMAs.
template <int CG>
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
  else
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp receives lane
// (taddr.lane + i), columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties registers written by an asynchronous tcgen05.ld to a point after
// tcgen05.wait::ld: the compiler may not move their first use above this.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]),
                 "+r"(r[i + 6]), "+r"(r[i + 7]));
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 2^x by the special-function unit (one instruction; flushes subnormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// 32 lanes x 8 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
      "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- conversions / stores

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

#endif  // __CUDACC__

}  // namespace tkg
