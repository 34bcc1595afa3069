// gemm_kernel.cuh — persistent load / compute / store-finish GEMM kernel for
// sm_103a:  C[M,N] (bf16) = A[M,K] · B[N,K]ᵀ with fp32 accumulation in TMEM.
//
// Structure (the LCSF template of "ThunderKittens: Simple, Fast, and Adorable
// AI Kernels", "The Four Functions: Load, Compute, Store, Finish", re-cast for
// tcgen05):
//   producer, one lane LOAD     TMA 2-D tile loads of A and B (and the NVFP4
//                               block scales) into a STAGES-deep shared ring,
//                               guarded by full/empty mbarriers
//                               ("Multi-Stage Buffer", Table 1).
//   MMA warp, one lane COMPUTE  tcgen05.mma into fp32 accumulators in tensor
//                               memory (two for 256-wide bf16 / FP8 tiles, one
//                               when a 512-wide tile or the NVFP4 scales fill
//                               the rest); each stage is released by
//                               tcgen05.commit on its empty barrier.
//   epilogue warps     STORE /  TMEM -> registers (tcgen05.ld), per-tensor
//                      FINISH   scales, round to bf16, 128-byte-swizzled
//                               staging tile, TMA store.  The accumulator is
//                               handed back early so the next tile's MMAs
//                               overlap this tile's store ("overlapping one
//                               chunk's load with the previous chunk's finish").
//   scale warps        (NVFP4)  copy the stage's block scales into tensor
//                               memory (tcgen05.cp), one lane of each.
// Warps: producer 0, MMA 1, epilogue 2.., scale warps after them; or, with the
// NVFP4 kernel's register split, four warpgroups: scale warps 0-3, epilogue
// 4-11, producer 12, MMA 13 (14-15 idle).
// Grid: persistent, one CTA (or CTA pair for the 2-SM MMA) per SM, walking the
// output tiles in the L2-aware grouped order ("Persistent Grid Launch",
// "Block Launch Order and L2 Cache Reuse").
//
// Every wait is bounded (TKG_OPT_TIMEOUT_NS).  A role that gives up records
// TKG timeout bits in the status word, raises the CTA abort flag so the others
// stop too, lets its in-flight copies land, and the CTA still frees its TMEM.
#pragma once

#include <cuda_runtime.h>

#include "tkg_device.cuh"

namespace tkg {

enum class Kind : int { BF16 = 0, FP8 = 1, NVFP4 = 2 };

// Status word bits written by the device.
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusRoleShift = 8;  // bit (8 + role) names the role that timed out
constexpr int kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2;

struct GemmParams {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b;
  CUtensorMap tmap_c;
  CUtensorMap tmap_sfa;
  CUtensorMap tmap_sfb;
  void* c_ptr;
  const float* a_scale;
  const float* b_scale;
  unsigned int* status;
  unsigned long long timeout_ns;
  int M, N, K;
  int tiles_m, tiles_n, num_kb;
  int group_m;
  int c_via_tma;
  int fault_mode;  // 0 = none; 1 = the producer skips the loads of its first stage (timeout test)
  int sf_blocks_a;  // NVFP4: 128-row scale blocks per K stage in the staged A scales
  int sf_blocks_b;  // same for B
  int sched;            // tile schedule (kSchedStatic / kSchedDynamic / kSchedSingle)
  unsigned int* visits;  // debug: if set, one increment per tile each time a CTA (pair) stores it
  // split-K head of the static schedule (split_tiles = 0: off): the first split_tiles tiles of
  // the tile order are cut into split_s K-ranges, run as the first work items
  int split_tiles;
  int split_s;
  float* split_ws;            // fp32 partial accumulators, one block per (piece, CTA, epilogue warp)
  unsigned int* split_cnt;    // per (split tile, CTA, epilogue warp): {pieces written, pieces done}
  int k_serpentine;           // 1: a CTA's odd-numbered work items walk their K blocks from the last one down
};

// Tile schedules ("Persistent Grid Launch"; Cluster Launch Control for the
// dynamic form):
//   kSchedStatic:  persistent grid, one CTA (pair) per SM; cluster c takes
//                  tiles c, c + clusters, c + 2 clusters, ...
//   kSchedDynamic: one cluster per tile is launched; a running cluster takes
//                  its own tile, then asks the hardware to cancel the launch
//                  of a cluster that has not started and takes that one's tile
//                  instead, until nothing is left to cancel.  One lane of the
//                  leader CTA asks one tile ahead; the answers reach every
//                  role of both CTAs through a ring of SCHED_SLOTS slots.
//   kSchedSingle:  one cluster per tile, each does its own tile only (the
//                  non-persistent launch).
constexpr int kSchedStatic = 0, kSchedDynamic = 1, kSchedSingle = 2;

// Split-K head ("Persistent Grid Launch": the persistent grid walks T output
// tiles in rounds of P clusters; when the last round would be at most half
// full, its tail tiles are cut into S pieces along K instead and run first).
// Work item w < split_tiles * S is piece s = w % S of tile w / S, covering the
// K blocks [s * num_kb / S, (s + 1) * num_kb / S); item w >= split_tiles * S is
// the whole tile w - split_tiles * (S - 1).  The pieces of a tile share the
// reduction: each epilogue warp's column chunks are dealt out, chunk j to
// piece j % S.  A piece writes the fp32 partials of the chunks it does not own
// to a workspace, counts itself in, waits (bounded) until all S pieces have,
// then adds, for each chunk it owns, the S partials in the order s = 0, 1, ...
// (its own read again from tensor memory at its place), and stores the chunk:
// the sum does not depend on timing.  The pieces of a tile are the first work
// items of S clusters of the persistent grid, which is never larger than the
// clusters that fit on the GPU at once, so the wait only waits for CTAs that
// are running or about to run; the last piece past the wait resets the counts.
struct WorkItem {
  int tile;
  int kb0, kb1;
  int piece;  // -1: whole tile
};
__host__ __device__ inline WorkItem work_item(int w, int split_tiles, int split_s, int num_kb) {
  const int split_items = split_tiles * split_s;
  if (w < split_items) {
    const int s = w % split_s;
    return WorkItem{w / split_s, s * num_kb / split_s, (s + 1) * num_kb / split_s, w};
  }
  return WorkItem{w - split_items + split_tiles, 0, num_kb, -1};
}

// NVFP4 block scales.  The caller's row-major [rows][K/16] e4m3 scales are
// first rewritten on the device into 2 KB runs, one per (256-deep K stage,
// 128-row block), each run four 512-byte atoms, one per MMA of the stage
// (gemm_nvfp4.cu).  The producers' TMA brings each stage's runs (A: the CTA's
// own 128 rows; B: all BN rows of the tile, since every CTA of a pair
// multiplies by all of B, and each TMEM lane quarter reads all of B's scales
// from its own lanes) into shared memory beside the operands, both CTAs' on
// the leader's sf_full barrier.  One lane of each of four scale warps of the
// leader then copies them into the stage's TMEM scale slot in both CTAs with
// tcgen05.cp (three 32x128b.warpx4 copies per MMA: one atom of A, BN / 128 of
// B) and commits to the stage's full barrier, so the MMA thread waits once per
// stage.  A thread issues a copy about every 60-80 cycles, so copies from one
// thread cannot keep up with the MMAs; from four warps, each taking one MMA
// of every stage, they run beside them.
template <Kind KIND_, int CG_, int BN_, int STAGES_, int EPI_WARPS_, int NUM_ACC_ = 2, bool COLL_A_ = false,
          int EPI_BUFS_ = 2, bool REG_SPLIT_ = false>
struct GemmCfg {
  static constexpr Kind KIND = KIND_;
  static constexpr int CG = CG_;                // CTAs per MMA (1, or 2 for the CTA pair) = CTAs per cluster
  static constexpr int BN = BN_;                // output-tile columns (whole pair)
  static constexpr int BM = 128;                // output-tile rows per CTA = TMEM lanes
  static constexpr int TILE_M = BM * CG;        // output-tile rows (whole pair)
  static constexpr int STAGES = STAGES_;
  static constexpr int EPI_WARPS = EPI_WARPS_;  // 4 or 8
  static constexpr int NUM_ACC = NUM_ACC_;      // fp32 accumulators in TMEM (2 = epilogue overlaps next tile)
  static constexpr bool SCALED = (KIND == Kind::NVFP4);
  static constexpr int ROW_BYTES = 128;         // K bytes per operand row per stage
  static constexpr uint32_t SWZ = select_swizzle(ROW_BYTES);
  static_assert(SWZ == 128, "operand rows must take the 128-byte swizzle");
  // K per stage in tensor-map x units (bf16 elements, or bytes for e4m3 / packed e2m1)
  static constexpr int K_TMAP = (KIND == Kind::BF16) ? 64 : 128;
  static constexpr int KSTEPS = 4;              // MMAs per stage: 32 bytes of K each
  static constexpr int B_ROWS = BN / CG;        // B rows staged by each CTA
  // tiles wider than one MMA (BN = 512): NSUB MMAs of N = 256 per K step, into adjacent
  // accumulator column ranges; each CTA stages B_ROWS / NSUB rows of B for each of them
  static constexpr int NSUB = BN > 256 ? BN / 256 : 1;
  static constexpr int MMA_N = BN / NSUB;
  static constexpr int B_SUB_ROWS = B_ROWS / NSUB;
  // 512-wide tiles: the K step's two MMAs share A; with COLL_A the first keeps A in the tensor
  // core's collector buffer and the second takes it from there instead of shared memory
  static constexpr bool COLL_A = COLL_A_;
  static constexpr int A_STAGE = BM * ROW_BYTES;
  static constexpr int B_BOX = B_ROWS * ROW_BYTES;             // bytes of one B tile load
  static constexpr int B_STAGE = (B_BOX + 1023) / 1024 * 1024;  // keeps every stage 1024-byte aligned
  // NVFP4 block scales per stage in shared memory: 16 bytes (the 16 scales of 256 K elements) per row,
  // this CTA's 128 rows of A and all BN rows of B, as per-MMA atoms
  static constexpr int SF_ROW_BYTES = 16;
  static constexpr int SFA_STAGE = SCALED ? BM * SF_ROW_BYTES : 0;
  static constexpr int SFB_STAGE = SCALED ? BN * SF_ROW_BYTES : 0;
  // four scale warps: lane 0 of scale warp q of the leader copies the scales of MMA q of every stage
  static constexpr int SF_WARPS = SCALED ? 4 : 0;
  static constexpr int SF_TX = SFA_STAGE + SFB_STAGE;
  // operand bytes landing per CTA per stage on the leader's full barrier (the scales land on its
  // sf_full barrier)
  static constexpr int STAGE_TX = A_STAGE + B_BOX;
  // one 512-byte shared-memory atom per MMA and 128 rows: the 4 scales of rows r, r + 32, r + 64,
  // r + 96 at byte 16 r (r < 32), which tcgen05.cp.32x128b.warpx4 puts at lane r of every TMEM lane
  // quarter, columns c .. c + 3 -- row m's scales at lane m, column c + m / 32
  static constexpr int SF_ATOM = 512;
  static constexpr int ACC_STRIDE = BN <= 128 ? 128 : BN <= 256 ? 256 : BN;  // accumulators start on aligned columns
  static constexpr int ACC_COLS = NUM_ACC * ACC_STRIDE;
  // TMEM columns of one stage's scales: A: 4 per MMA (row m at column m/32);
  // B: BN/32 per MMA (row n at column n/32).
  static constexpr int SF_COLS_A = 4 * KSTEPS;
  static constexpr int SF_COLS_B = (BN / 32) * KSTEPS;
  static constexpr int SF_COLS_STAGE = SCALED ? SF_COLS_A + SF_COLS_B : 0;
  // one TMEM scale slot per ring stage
  static constexpr int TMEM_USED = ACC_COLS + STAGES * SF_COLS_STAGE;
  static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                 : TMEM_USED <= 256 ? 256 : 512;
  // output columns per epilogue chunk: 64 (rows of 128 B of bf16) when BN allows, else 32 (64 B)
  static constexpr int EPI_COLS = (BN % 64 == 0) ? 64 : 32;
  static constexpr int EPI_ROW_BYTES = EPI_COLS * 2;
  static constexpr uint32_t EPI_SWZ = select_swizzle(EPI_ROW_BYTES);
  static constexpr int EPI_BUF = 32 * EPI_ROW_BYTES;  // one warp's 32-row staging tile
  // staging tiles per epilogue warp: 2 lets a chunk's shared-memory writes overlap the previous
  // chunk's TMA store; 1 halves the staging memory (eight epilogue warps then fit beside the ring)
  static constexpr int EPI_BUFS = EPI_BUFS_;
  // Register split: 16 warps in four warpgroups -- the copy issuers (warps 0-3; idle without block
  // scales), the epilogue (4-11), the producer, the MMA issuer and two idle warps (12-15) -- launched
  // at 128 registers each; the epilogue warpgroups take 192 (setmaxnreg), enough to read their whole
  // share of the accumulator before storing any of it, the other two give theirs down to 64.
  static constexpr bool REG_SPLIT = REG_SPLIT_;
  static constexpr int THREADS = REG_SPLIT ? 512 : 64 + 32 * (EPI_WARPS + SF_WARPS);
  static constexpr int PRODUCER_WARP = REG_SPLIT ? 12 : 0;
  static constexpr int MMA_WARP = REG_SPLIT ? 13 : 1;
  static constexpr int EPI_WARP0 = REG_SPLIT ? 4 : 2;
  static constexpr int SF_WARP0 = REG_SPLIT ? 0 : 2 + EPI_WARPS;
  static constexpr int EPI_REGS = 192, OTHER_REGS = 64;
  static constexpr uint32_t IDESC = (KIND == Kind::BF16)   ? idesc_dense(kFmtBF16, BM * CG, MMA_N)
                                    : (KIND == Kind::FP8) ? idesc_dense(kFmtE4M3, BM * CG, MMA_N)
                                                          : idesc_mxf4nvf4(BM * CG, MMA_N);

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
  static constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_STAGE;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF;
  // full / empty per stage, tensor-memory full / empty per accumulator, drain, and (NVFP4) the
  // per-stage sf_full barriers
  // (+1 for tiles of two MMAs per K step: the accumulator's upper half is handed back on its own
  // barrier, so the next tile's first MMAs into the lower half need not wait for the whole drain)
  static constexpr int NUM_BARS =
      2 * STAGES + 2 * NUM_ACC + 1 + (SCALED ? STAGES : 0) + (SCALED ? 1 : 0) + (NSUB > 1 ? 1 : 0);
  // dynamic schedule: ring of cancellation answers (16 bytes each) with a full
  // barrier per slot in every CTA and an empty barrier per slot in the leader,
  // after the barriers above
  static constexpr int SCHED_SLOTS = 8;
  static constexpr int SCHED_BAR0 = NUM_BARS;
  static constexpr int OFF_MISC = OFF_BAR + 8 * (NUM_BARS + 2 * SCHED_SLOTS);
  static constexpr int OFF_SCHED = (OFF_MISC + 16 + 15) / 16 * 16;
  // readers of every answer: each CTA's producer lane, epilogue warps and scale
  // warps, and the leader's MMA lane
  static constexpr int SCHED_READERS = CG * (1 + EPI_WARPS + SF_WARPS) + 1;
  static constexpr int SMEM_BYTES = OFF_SCHED + 16 * SCHED_SLOTS + 1024;  // + slack to align the base to 1024

  static_assert(B_STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "stages must keep 1024-byte swizzle atoms aligned");
  static_assert((OFF_SFA % 1024) == 0 && (OFF_EPI % 1024) == 0, "region alignment");
  static_assert(BN % 32 == 0 && BN >= 64 && (BN <= 256 || BN == 512), "BN: a multiple of 32 in [64,256], or 512");
  static_assert(NSUB == 1 || (NSUB == 2 && !SCALED && NUM_ACC == 1 && CG == 2), "512-wide tiles: bf16 / FP8 pairs");
  static_assert(!COLL_A || NSUB == 2, "the A collector is shared by the two MMAs of a 512-wide K step");
  static_assert(B_ROWS % 8 == 0, "B rows per CTA must fill whole 8-row swizzle atoms");
  static_assert(EPI_BUF % (8 * EPI_SWZ) == 0, "staging tiles must keep swizzle atoms aligned");
  static_assert(EPI_BUFS == 1 || EPI_BUFS == 2, "one or two staging tiles per epilogue warp");
  static_assert(!SCALED || BN % 128 == 0, "block-scaled tiles cover whole 128-row scale blocks of B");
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "epilogue is one or two warpgroups");
  static_assert(NUM_ACC == 1 || NUM_ACC == 2, "one or two accumulators");
  static_assert(TMEM_USED <= 512, "tensor memory has 512 columns");
  static_assert(!SCALED || (ACC_COLS % 16 == 0 && SF_COLS_STAGE % 16 == 0 && SF_COLS_A == 16),
                "scale columns are written 16 at a time at 16-column-aligned addresses");
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB shared-memory limit");
  static_assert(!REG_SPLIT || (EPI_WARPS == 8 && (SF_WARPS == 4 || !SCALED) && CG == 2 && (BN / EPI_COLS) % 2 == 0),
                "register split: eight epilogue warps, four copy issuers (NVFP4), CTA pairs");
  // the warpgroups' shares may not exceed what the block was launched with (512 threads x 128)
  static_assert(!REG_SPLIT || 2 * 128 * EPI_REGS + 2 * 128 * OTHER_REGS <= 512 * 128, "register split over budget");
};

__device__ __forceinline__ void record_timeout(unsigned int* status, int role, volatile int* abort_flag) {
  atomicOr(status, kStatusTimeout | (1u << (kStatusRoleShift + role)));
  *abort_flag = 1;
}

// Spin (bounded) so that copies already issued by this CTA can land before it
// gives up its shared memory.
__device__ __forceinline__ void settle_inflight_copies() {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < 50000ull) {
  }
}

template <int CG>
__device__ __forceinline__ void mma_commit(uint32_t bar, uint16_t mask) {
  if constexpr (CG == 1) {
    (void)mask;
    mma_commit_local(bar);
  } else {
    mma_commit_pair(bar, mask);
  }
}

// 32 lanes x 16 consecutive fp32 columns of tensor memory (the split-K reduction's own partial,
// a quarter chunk at a time), and the matching register tie after tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
  asm volatile("" : "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
               "+r"(r[15]));
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) tkg_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase + C::OFF_A;
  const uint32_t sB = sbase + C::OFF_B;
  const uint32_t sEpi = sbase + C::OFF_EPI;
  const uint32_t sSFA = sbase + C::OFF_SFA;
  const uint32_t sSFB = sbase + C::OFF_SFB;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + C::NUM_ACC + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 2 * C::NUM_ACC);
  // two MMAs per K step (one accumulator): the epilogue has read the accumulator's upper half
  const uint32_t tempty_hi_bar = bar0 + 8u * (C::NUM_BARS - 1);
  // NVFP4: stage s's block scales landed in this CTA's shared memory
  auto sf_full_bar = [&](int st) { return bar0 + 8u * (2 * C::STAGES + 2 * C::NUM_ACC + 1 + st); };
  // NVFP4, copied scales: the four copy issuers' last copies are done
  const uint32_t cp_drain_bar = bar0 + 8u * (3 * C::STAGES + 2 * C::NUM_ACC + 1);
  auto sched_full_bar = [&](int j) { return bar0 + 8u * (C::SCHED_BAR0 + j); };
  auto sched_empty_bar = [&](int j) { return bar0 + 8u * (C::SCHED_BAR0 + C::SCHED_SLOTS + j); };
  const uint32_t sResp = sbase + C::OFF_SCHED;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // a cluster is one CTA, or the CTA pair of the 2-SM MMA whose rank-0 CTA (the leader) issues it
  const uint32_t prank = (C::CG > 1) ? cluster_ctarank() : 0u;  // rank in the CTA pair
  constexpr uint32_t leader = 0;
  const int cluster_id = blockIdx.x / C::CG;
  const int num_clusters = gridDim.x / C::CG;
  const int num_units = p.tiles_m * p.tiles_n;
  // work items: tiles, each of the split_tiles first ones replaced by split_s pieces
  const int num_tiles = num_units + p.split_tiles * (p.split_s - 1);
  const TileOrder order{p.tiles_m, p.tiles_n, p.group_m};
  auto work_of = [&](int w) { return work_item(w, p.split_tiles, p.split_s, p.num_kb); };
  auto tile_coord = [&](int t, int& tm, int& tn) { order.coord(t, tm, tn); };
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // + one arrival per copy issuer of the leader (NVFP4; its tcgen05.commit, once its copies are done)
      mbar_init(full_bar(s), C::SCALED ? 1 + 4 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < C::NUM_ACC; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), C::CG * C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    if constexpr (C::NSUB > 1) mbar_init(tempty_hi_bar, C::CG * C::EPI_WARPS);
    if constexpr (C::SCALED) {
      for (int st = 0; st < C::STAGES; ++st) mbar_init(sf_full_bar(st), 1);
    }
    if constexpr (C::SCALED) mbar_init(cp_drain_bar, 4);
    for (int j = 0; j < C::SCHED_SLOTS; ++j) {
      mbar_init(sched_full_bar(j), 1);  // the leader's expect_tx arrival + the 16-byte answer
      mbar_init(sched_empty_bar(j), C::SCHED_READERS);
    }
    *abort_flag = 0;
    *never_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmap_a);
    tma_prefetch_desc(&p.tmap_b);
    if constexpr (C::SCALED) {
      tma_prefetch_desc(&p.tmap_sfa);
      tma_prefetch_desc(&p.tmap_sfb);
    }
    if (p.c_via_tma) tma_prefetch_desc(&p.tmap_c);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc<C::CG>(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish<C::CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (C::CG > 1) {
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Up to here the CTA touched only its own shared and tensor memory.  From
  // here on it reads A, B and the scales and writes C, which the grid before
  // it on the stream may still be producing or reading: wait for that grid
  // (no-op without a programmatic dependency), then let the next grid's CTAs
  // start their own set-up wherever an SM becomes free.
  griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------------- tile sequence
  const int first_tile = cluster_id < num_tiles ? cluster_id : -1;
  const uint32_t sched_empty_leader0 = (C::CG > 1) ? mapa_shared(sched_empty_bar(0), 0) : sched_empty_bar(0);
  // The tile after tile t, the k-th (k = 0, 1, ...) of this CTA's sequence, or
  // -1 when there is none.  Called by one thread of each role, in order k.
  auto next_tile = [&](int t, int k, bool& ok) -> int {
    if (!ok) return -1;
    if (p.sched == kSchedStatic) {
      const int n = t + num_clusters;
      return n < num_tiles ? n : -1;
    }
    if (p.sched == kSchedSingle) return -1;
    const int j = k % C::SCHED_SLOTS;
    const uint32_t ph = static_cast<uint32_t>(k / C::SCHED_SLOTS) & 1u;
    if (!mbar_wait(sched_full_bar(j), ph, tmo, abort_flag)) {
      ok = false;
      return -1;
    }
    // decoded into a register before the slot is handed back for the next answer
    const int x = clc_first_ctaid_x(ld_shared_v4(sResp + 16u * static_cast<uint32_t>(j)));
    mbar_arrive_cluster(sched_empty_leader0 + 8u * static_cast<uint32_t>(j));
    return x < 0 ? -1 : x / C::CG;
  };
  // Dynamic schedule, the leader's producer lane at the start of its k-th tile:
  // ask for the tile after it, answered into slot k % SCHED_SLOTS of every CTA
  // once all readers of that slot's previous answer are done with it.
  auto request_tile = [&](int k) -> bool {
    const int j = k % C::SCHED_SLOTS;
    const uint32_t ph = static_cast<uint32_t>(k / C::SCHED_SLOTS) & 1u;
    if (!mbar_wait(sched_empty_bar(j), ph ^ 1u, tmo, abort_flag)) return false;
#pragma unroll
    for (int r = 0; r < C::CG; ++r)
      mbar_arrive_expect_tx_cluster(C::CG > 1 ? mapa_shared(sched_full_bar(j), static_cast<uint32_t>(r))
                                              : sched_full_bar(j),
                                    16u);
    clc_try_cancel_multicast(sResp + 16u * static_cast<uint32_t>(j), sched_full_bar(j));
    return true;
  };
  // The same for a whole warp: lane 0 reads the ring, the others follow.
  auto next_tile_warp = [&](int t, int k, bool& ok) -> int {
    bool okl = ok;
    int n = -1;
    if (lane == 0) n = next_tile(t, k, okl);
    n = __shfl_sync(0xffffffffu, n, 0);
    ok = __shfl_sync(0xffffffffu, okl ? 1 : 0, 0) != 0;
    return n;
  };

  if (warp >= C::EPI_WARP0 && warp < C::EPI_WARP0 + C::EPI_WARPS) {
    if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::EPI_REGS>();
    // ------------------------------------------------------------ STORE / FINISH
    constexpr int SUBS = C::EPI_WARPS / 4;
    const int ew = warp - C::EPI_WARP0;
    const int quad = warp & 3;  // the TMEM lane quarter this warp may read
    const int sub = ew / 4;
    const uint32_t stage0 = sEpi + static_cast<uint32_t>(ew * C::EPI_BUFS * C::EPI_BUF);
    float sa = 1.0f, sb = 1.0f;
    if constexpr (C::KIND != Kind::BF16) {
      sa = *p.a_scale;
      sb = *p.b_scale;
    }
    const uint32_t tempty_leader0 = (C::CG == 2) ? mapa_shared(tempty_bar(0), leader) : tempty_bar(0);
    const uint32_t tempty_hi_leader = (C::CG == 2) ? mapa_shared(tempty_hi_bar, leader) : tempty_hi_bar;
    int it = 0;
    int chunk_ctr = 0;
    bool seq_ok = true;
    constexpr int NCH = C::BN / C::EPI_COLS;  // chunks of the accumulator
    constexpr int NLD = C::EPI_COLS / 32;  // 32-column TMEM loads per chunk
    constexpr int NPK = C::EPI_COLS / 2;   // packed bf16 pairs per row
    constexpr int RB = C::EPI_ROW_BYTES;
    constexpr int NQ = C::EPI_COLS / 4;    // 16-byte groups of fp32 per row per chunk
    static_assert(NQ % 4 == 0, "the split-K reduction takes 16 columns at a time");
    // split-K: this warp's block of a piece's partial accumulator: its 32 rows x its chunks,
    // laid out [chunk][16-byte column group][lane] so that each store / load of a warp is 512
    // contiguous bytes
    constexpr int WS_WARP = 32 * (C::BN / SUBS);  // floats
    // tiles of one MMA per K step may be split along K; the 256x512 tile never is
    constexpr bool CAN_SPLIT = C::NSUB == 1;
    auto ws_block = [&](int piece) {
      return reinterpret_cast<float4*>(p.split_ws) +
             ((static_cast<size_t>(piece) * C::CG + prank) * C::EPI_WARPS + ew) * (WS_WARP / 4);
    };
    for (int t = first_tile; t >= 0; t = next_tile_warp(t, it, seq_ok), ++it) {
      const WorkItem wk = work_of(t);
      int tm, tn;
      tile_coord(wk.tile, tm, tn);
      const int acc = it % C::NUM_ACC;
      const uint32_t acc_phase = (it / C::NUM_ACC) & 1;
      const bool got = __all_sync(0xffffffffu, mbar_wait<true>(tfull_bar(acc), acc_phase, tmo, abort_flag));
      if (!got) {
        if (lane == 0) record_timeout(p.status, kRoleEpilogue, abort_flag);
        break;
      }
      tc_fence_after();
      const int row0 = tm * C::TILE_M + static_cast<int>(prank) * C::BM + quad * 32;
      const int col0 = tn * C::BN;

      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * C::ACC_STRIDE);
      // after this warp's last read of chunk c: hand back what it no longer needs
      auto release_after = [&](int c, bool may_release) {
        if constexpr (C::NSUB > 1) {
          // the two MMAs' halves of the accumulator are handed back one after the other
          if (may_release && c < NCH / 2 && c + SUBS >= NCH / 2) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8u * acc);
          }
          if (may_release && c + SUBS >= NCH) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_hi_leader);
          }
        } else if (may_release && c + SUBS >= NCH) {
          // last TMEM read of this accumulator by this warp: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8u * acc);
        }
      };
      auto load_chunk = [&](int c, uint32_t (&r)[NLD][32], bool may_release) {
        __syncwarp();
#pragma unroll
        for (int l = 0; l < NLD; ++l) tmem_ld_32x32b_x32(t_row + c * C::EPI_COLS + 32 * l, r[l]);
        tmem_wait_ld();
#pragma unroll
        for (int l = 0; l < NLD; ++l) reg_fence(r[l]);
        release_after(c, may_release);
      };
      // two fp32 values, scaled (FP8 / NVFP4: by scale_a, then scale_b) and rounded to a bf16 pair
      auto scale_pack = [&](float x0, float x1) -> uint32_t {
        if constexpr (C::KIND != Kind::BF16) {
          x0 = x0 * sa;
          x0 = x0 * sb;
          x1 = x1 * sa;
          x1 = x1 * sb;
        }
        return pack_bf16x2(x0, x1);
      };
      // store chunk c of this warp's rows, given as packed bf16 pairs: through a staging tile and
      // a TMA store, or (an output whose row pitch TMA cannot take) with generic stores
      auto store_chunk_tma = [&](int c, const uint32_t (&pk)[NPK]) {
        {
          uint32_t buf = stage0 + static_cast<uint32_t>(chunk_ctr % C::EPI_BUFS) * C::EPI_BUF;
          // one staging tile: its row addresses are loop-invariant, and the 128-register kernels
          // cannot keep them live across the tile loop; make the base opaque so they are
          // recomputed per chunk
          if constexpr (C::EPI_BUFS == 1) asm volatile("mov.b32 %0, %0;" : "+r"(buf));
          if (lane == 0) bulk_wait_group_read<C::EPI_BUFS - 1>();  // the store that last used `buf` has read it
          __syncwarp();
          const uint32_t row_off = static_cast<uint32_t>(lane) * RB;
#pragma unroll
          for (int ch = 0; ch < RB / 16; ++ch) {
            const uint32_t off = swizzle_offset(row_off + ch * 16u, C::EPI_SWZ);
            st_shared_v4(buf + off, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmap_c, buf, col0 + c * C::EPI_COLS, row0);
            bulk_commit_group();
          }
        }
        ++chunk_ctr;
      };
      auto store_chunk_generic = [&](int c, const uint32_t (&pk)[NPK]) {
        {
          const int row = row0 + lane;
          if (row < p.M) {
            uint16_t* out = static_cast<uint16_t*>(p.c_ptr) + static_cast<size_t>(row) * p.N;
#pragma unroll
            for (int j = 0; j < NPK; ++j) {
              const int col = col0 + c * C::EPI_COLS + 2 * j;
              const uint32_t v = pk[j];
              if (col < p.N) out[col] = static_cast<uint16_t>(v & 0xFFFFu);
              if (col + 1 < p.N) out[col + 1] = static_cast<uint16_t>(v >> 16);
            }
          }
        }
        ++chunk_ctr;
      };
      auto store_chunk = [&](int c, const uint32_t (&pk)[NPK]) {
        if (p.c_via_tma)
          store_chunk_tma(c, pk);
        else
          store_chunk_generic(c, pk);
      };
      auto count_visit = [&]() {
        if (p.visits != nullptr && ew == 0 && lane == 0 && prank == 0)
          atomicAdd(p.visits + tm * p.tiles_n + tn, 1u);
      };
      if (!CAN_SPLIT || wk.piece < 0) {
        count_visit();
        constexpr int NL = NCH / SUBS;
        if constexpr (C::REG_SPLIT && NL * NLD * 32 > 128) {
          // the warp's whole share of the accumulator first, each chunk scaled and packed to bf16 as it
          // is read (its fp32 values do not fit the registers at once; each half is handed back after
          // its last read), then stored chunk by chunk while the next tile's MMAs run
          if (!p.c_via_tma) {
            // generic stores (an output row pitch TMA cannot take): 32 columns at a time, straight
            // from the registers they were read into; this rare path need not hand back early
            const int row = row0 + lane;
            for (int c = sub; c < NCH; c += SUBS) {
              for (int l = 0; l < NLD; ++l) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + c * C::EPI_COLS + 32 * l, r);
                tmem_wait_ld();
                reg_fence(r);
                if (row < p.M) {
                  uint16_t* out = static_cast<uint16_t*>(p.c_ptr) + static_cast<size_t>(row) * p.N;
#pragma unroll
                  for (int i = 0; i < 16; ++i) {
                    const uint32_t v = scale_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    const int col = col0 + c * C::EPI_COLS + 32 * l + 2 * i;
                    if (col < p.N) out[col] = static_cast<uint16_t>(v & 0xFFFFu);
                    if (col + 1 < p.N) out[col + 1] = static_cast<uint16_t>(v >> 16);
                  }
                }
              }
              release_after(c, true);
            }
          } else {
            uint32_t pk[NL][NPK];
#pragma unroll
            for (int j = 0; j < NL; ++j) {
              const int c = sub + SUBS * j;
#pragma unroll
              for (int l = 0; l < NLD; ++l) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld_32x32b_x32(t_row + c * C::EPI_COLS + 32 * l, r);
                tmem_wait_ld();
                reg_fence(r);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  pk[j][16 * l + i] = scale_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
              }
              release_after(c, true);
            }
#pragma unroll
            for (int j = 0; j < NL; ++j) store_chunk_tma(sub + SUBS * j, pk[j]);
          }
        } else if constexpr (C::REG_SPLIT) {
          // the warp's whole share of the accumulator first (handed back after the last read), then
          // scaled, packed and stored chunk by chunk while the next tile's MMAs run
          uint32_t r[NL][NLD][32];
#pragma unroll
          for (int j = 0; j < NL; ++j) load_chunk(sub + SUBS * j, r[j], true);
#pragma unroll
          for (int j = 0; j < NL; ++j) {
            uint32_t pk[NPK];
#pragma unroll
            for (int l = 0; l < NLD; ++l)
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[16 * l + i] = scale_pack(__uint_as_float(r[j][l][2 * i]), __uint_as_float(r[j][l][2 * i + 1]));
            store_chunk(sub + SUBS * j, pk);
          }
        } else {
          for (int c = sub; c < NCH; c += SUBS) {
            uint32_t r[NLD][32];
            load_chunk(c, r, true);
            uint32_t pk[NPK];
#pragma unroll
            for (int l = 0; l < NLD; ++l)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                pk[16 * l + j] = scale_pack(__uint_as_float(r[l][2 * j]), __uint_as_float(r[l][2 * j + 1]));
            store_chunk(c, pk);
          }
        }
      } else {
        const int S = p.split_s;
        const int my_s = wk.piece % S;
        constexpr int NLOC = (NCH + SUBS - 1) / SUBS;  // this warp's chunks: c = sub + SUBS * j
        constexpr size_t PIECE_STRIDE = static_cast<size_t>(C::CG) * C::EPI_WARPS * (WS_WARP / 4);
        // 1. partials of the chunks other pieces own -> this piece's workspace block
        float4* mine = ws_block(wk.piece);
        for (int j = 0; j < NLOC; ++j) {
          const int c = sub + SUBS * j;
          if (c >= NCH || j % S == my_s) continue;
          float4* dst = mine + j * (NQ * 32) + lane;
          __syncwarp();
#pragma unroll
          for (int q0 = 0; q0 < NQ; q0 += 4) {
            uint32_t o[16];
            tmem_ld_32x32b_x16(t_row + static_cast<uint32_t>(c * C::EPI_COLS + 4 * q0), o);
            tmem_wait_ld();
            reg_fence16(o);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              __stcg(dst + (q0 + q) * 32, make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                                      __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3])));
          }
        }
        // 2. count in (fence + atomic), wait until all S pieces have (acquire), bounded
        unsigned int* cnt = p.split_cnt + 2 * ((static_cast<size_t>(wk.tile) * C::CG + prank) * C::EPI_WARPS + ew);
        __threadfence();
        __syncwarp();
        int arrived = 1;
        if (lane == 0) {
          atomicAdd(cnt, 1u);
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu(cnt) < static_cast<unsigned int>(S)) {
            if (*abort_flag || globaltimer_ns() - t0 > tmo) {
              arrived = 0;
              break;
            }
            __nanosleep(64);
          }
        }
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        __threadfence();
        if (arrived) {
          // 3. the chunks this piece owns: the S partials added in piece order, stored as bf16
          const float4* first = ws_block(wk.tile * S) + lane;
          for (int j = my_s; j < NLOC; j += S) {
            const int c = sub + SUBS * j;
            if (c >= NCH) break;
            if (j == 0) count_visit();
            // a quarter chunk (16 columns) at a time: the S partials added in piece order, this
            // piece's own read from tensor memory at its place, then scaled and packed, so that
            // no fp32 chunk stays in registers (the 128-register kernels hold no more)
            uint32_t pk[NPK];
#pragma unroll
            for (int q0 = 0; q0 < NQ; q0 += 4) {
              float4 sum[4];
              for (int s2 = 0; s2 < S; ++s2) {
                float4 part[4];
                if (s2 == my_s) {
                  uint32_t o[16];
                  tmem_ld_32x32b_x16(t_row + static_cast<uint32_t>(c * C::EPI_COLS + 4 * q0), o);
                  tmem_wait_ld();
                  reg_fence16(o);
#pragma unroll
                  for (int q = 0; q < 4; ++q)
                    part[q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                          __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
                } else {
                  const float4* src = first + s2 * PIECE_STRIDE + j * (NQ * 32) + q0 * 32;
#pragma unroll
                  for (int q = 0; q < 4; ++q) part[q] = __ldcg(src + q * 32);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  if (s2 == 0) {
                    sum[q] = part[q];
                  } else {
                    sum[q].x += part[q].x;
                    sum[q].y += part[q].y;
                    sum[q].z += part[q].z;
                    sum[q].w += part[q].w;
                  }
                }
              }
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                pk[2 * (q0 + q)] = scale_pack(sum[q].x, sum[q].y);
                pk[2 * (q0 + q) + 1] = scale_pack(sum[q].z, sum[q].w);
              }
            }
            store_chunk(c, pk);
          }
        } else if (lane == 0) {
          record_timeout(p.status, kRoleEpilogue, abort_flag);
        }
        // the accumulator has been read for the last time: hand it back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8u * acc);
        // 4. the last piece past the wait resets both counts for the next launch
        if (arrived && lane == 0 && atomicAdd(cnt + 1, 1u) == static_cast<unsigned int>(S - 1)) {
          cnt[0] = 0u;
          cnt[1] = 0u;
        }
      }
    }
    if (!seq_ok && lane == 0) record_timeout(p.status, kRoleEpilogue, abort_flag);
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  } else {
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::OTHER_REGS>();
    if (warp == C::PRODUCER_WARP) {
      // ------------------------------------------------------------ LOAD
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        bool first = true;
        int k = 0;
        for (int t = first_tile; t >= 0 && ok; t = next_tile(t, k, ok), ++k) {
          if (p.sched == kSchedDynamic && prank == 0 && !request_tile(k)) {
            ok = false;
            break;
          }
          const WorkItem wk = work_of(t);
          int tm, tn;
          tile_coord(wk.tile, tm, tn);
          const int a_row = tm * C::TILE_M + static_cast<int>(prank) * C::BM;
          // this CTA's rows of B for each MMA of the K step (one MMA unless the tile is 512 wide)
          const int b_row = tn * C::BN + static_cast<int>(prank) * C::B_SUB_ROWS;
          // serpentine K: odd items start where the previous item's K walk ended, on the
          // operand panels' tails that are still in L2
          const bool rev = p.k_serpentine && (k & 1);
          for (int i = 0; i < wk.kb1 - wk.kb0; ++i) {
            const int kb = rev ? wk.kb1 - 1 - i : wk.kb0 + i;
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, tmo, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t fb = (C::CG == 2) ? mapa_shared(full_bar(stage), leader) : full_bar(stage);
            if (prank == 0) mbar_arrive_expect_tx(full_bar(stage), C::STAGE_TX * C::CG);
            if (!(first && p.fault_mode == 1)) {
              if constexpr (C::SCALED) {
                // staged scales: 2 KB (16 rows of 128 B) per (K stage, 128-row block), the blocks of
                // one K stage contiguous; both CTAs' land on the leader's sf_full barrier, since the
                // leader's copies read them from both CTAs' shared memory.  Requested before the
                // operands, so that the copies into tensor memory run while the operands arrive.
                const int ya = (kb * p.sf_blocks_a + a_row / 128) * 16;
                const int yb = (kb * p.sf_blocks_b + (tn * C::BN) / 128) * 16;
                const uint32_t sfb_bar = (C::CG == 2) ? mapa_shared(sf_full_bar(stage), leader) : sf_full_bar(stage);
                if (prank == 0) mbar_arrive_expect_tx(sf_full_bar(stage), C::SF_TX * C::CG);
                tma_load_2d<C::CG>(sSFA + stage * C::SFA_STAGE, &p.tmap_sfa, sfb_bar, 0, ya);
                tma_load_2d<C::CG>(sSFB + stage * C::SFB_STAGE, &p.tmap_sfb, sfb_bar, 0, yb);
              }
              tma_load_2d<C::CG>(sA + stage * C::A_STAGE, &p.tmap_a, fb, kb * C::K_TMAP, a_row);
  #pragma unroll
              for (int sub = 0; sub < C::NSUB; ++sub)
                tma_load_2d<C::CG>(sB + stage * C::B_STAGE + sub * C::B_SUB_ROWS * C::ROW_BYTES, &p.tmap_b, fb,
                                   kb * C::K_TMAP, b_row + sub * C::MMA_N);
            }
            first = false;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) {
          record_timeout(p.status, kRoleProducer, abort_flag);
          settle_inflight_copies();
        }
      }
      __syncwarp();
    } else if (warp == C::MMA_WARP) {
      // ------------------------------------------------------------ COMPUTE
      if (lane == 0 && prank == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int it = 0;
        for (int t = first_tile; t >= 0 && ok; t = next_tile(t, it, ok), ++it) {
          const int acc = it % C::NUM_ACC;
          const uint32_t acc_phase = (it / C::NUM_ACC) & 1;
          if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, tmo, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::ACC_STRIDE);
          const WorkItem wk = work_of(t);
          // K blocks in the producer's order (see the LOAD role); only the first MMA of the item
          // overwrites the accumulator
          for (int i = 0; i < wk.kb1 - wk.kb0; ++i) {
            if (!mbar_wait(full_bar(stage), phase, tmo, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = sA + stage * C::A_STAGE;
            const uint32_t b0 = sB + stage * C::B_STAGE;
            // this stage's TMEM scale slot (NVFP4): the stage's full barrier also counts the copy
            // issuers that filled it
            const uint32_t sf_tmem = tmem_base + static_cast<uint32_t>(C::ACC_COLS + stage * C::SF_COLS_STAGE);
  #pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
              const uint64_t ad = sdesc_sw128(a0 + 32u * kk);
              const uint64_t bd = sdesc_sw128(b0 + 32u * kk);
              const uint32_t accum = (i != 0 || kk != 0) ? 1u : 0u;
              if constexpr (C::NSUB > 1) {
                // the two N = 256 halves of the tile, into adjacent accumulator column ranges
                constexpr int C0 = C::COLL_A ? kCollFill : kCollNone;
                constexpr int C1 = C::COLL_A ? kCollLastUse : kCollNone;
                const uint64_t bd1 = sdesc_sw128(b0 + static_cast<uint32_t>(C::B_SUB_ROWS * C::ROW_BYTES) + 32u * kk);
                const uint32_t d1 = d_tmem + static_cast<uint32_t>(C::MMA_N);
                if constexpr (C::KIND == Kind::BF16)
                  mma_bf16<C::CG, C0>(d_tmem, ad, bd, C::IDESC, accum);
                else
                  mma_f8f6f4<C::CG, C0>(d_tmem, ad, bd, C::IDESC, accum);
                if (kk == 0 && i == 0) {
                  // the tile's first MMA into the upper half: the epilogue has read it
                  if (!mbar_wait(tempty_hi_bar, acc_phase ^ 1u, tmo, abort_flag)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                }
                if constexpr (C::KIND == Kind::BF16)
                  mma_bf16<C::CG, C1>(d1, ad, bd1, C::IDESC, accum);
                else
                  mma_f8f6f4<C::CG, C1>(d1, ad, bd1, C::IDESC, accum);
              } else if constexpr (C::KIND == Kind::BF16)
                mma_bf16<C::CG>(d_tmem, ad, bd, C::IDESC, accum);
              else if constexpr (C::KIND == Kind::FP8)
                mma_f8f6f4<C::CG>(d_tmem, ad, bd, C::IDESC, accum);
              else
                mma_mxf4nvf4<C::CG>(d_tmem, ad, bd, C::IDESC, sf_tmem + 4u * kk,
                                    sf_tmem + C::SF_COLS_A + (C::BN / 32) * kk, accum);
            }
            if (!ok) break;  // (the wait for the accumulator's upper half ran out)
            // the stage (operands and, NVFP4, scale slot) is free for both CTAs of the pair
            mma_commit<C::CG>(empty_bar(stage), (1u << C::CG) - 1u);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit<C::CG>(tfull_bar(acc), static_cast<uint16_t>((1u << C::CG) - 1u));
        }
        // No MMA may still be writing TMEM when it is released.
        mma_commit<C::CG>(drain_bar, 0x1u);
        mbar_wait(drain_bar, 0, tmo, never_abort);
        if (!ok) record_timeout(p.status, kRoleMma, abort_flag);
      }
      __syncwarp();
    } else if (warp >= C::SF_WARP0 && warp < C::SF_WARP0 + C::SF_WARPS) {
      // ------------------------------------------------------------ SCALES (NVFP4)
      // Lane 0 of scale warp q of the leader CTA copies, for every K stage of the CTA pair's tile
      // sequence, the scales of MMA q of the stage (one 512-byte atom of A's rows, BN / 128 of B's)
      // from both CTAs' shared memory into the stage's TMEM scale slot of both CTAs, once the scales
      // have landed (the leader's sf_full barrier counts both CTAs' copies), and then commits to the
      // stage's full barrier: its arrival comes when the copies are done.  The slot is free by then:
      // the producer refilled the stage only after the MMAs that last read it had completed.  The
      // other warps, and the peer CTA's, only follow the tile sequence.
      if constexpr (C::SCALED) {
        const int q = warp & 3;
        const bool issuer = prank == 0 && lane == 0;
        bool ok = true;
        int k = 0;
        int step = 0;
        for (int t = first_tile; t >= 0 && ok; t = next_tile_warp(t, k, ok), ++k) {
          const WorkItem wk = work_of(t);
          if (issuer) {
            for (int kb = wk.kb0; kb < wk.kb1 && ok; ++kb, ++step) {
              const int j = step % C::STAGES;
              const uint32_t ph = static_cast<uint32_t>(step / C::STAGES) & 1u;
              if (!mbar_wait(sf_full_bar(j), ph, tmo, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t slot = tmem_base + static_cast<uint32_t>(C::ACC_COLS + j * C::SF_COLS_STAGE);
              const uint32_t sfa_s = sSFA + j * C::SFA_STAGE + q * C::SF_ATOM;
              const uint32_t sfb_s = sSFB + j * C::SFB_STAGE + q * C::SF_ATOM;
              tmem_cp_32x128b_warpx4<C::CG>(slot + 4u * q, sdesc_rows16(sfa_s));
  #pragma unroll
              for (int g = 0; g < C::BN / 128; ++g)
                tmem_cp_32x128b_warpx4<C::CG>(slot + C::SF_COLS_A + (C::BN / 32) * q + 4u * g,
                                              sdesc_rows16(sfb_s + g * C::KSTEPS * C::SF_ATOM));
              mma_commit<C::CG>(full_bar(j), 0x1u);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        if (issuer) {
          // no copy may still be writing tensor memory when it is released (a stage whose MMAs never
          // ran, after a timeout elsewhere)
          mma_commit<C::CG>(cp_drain_bar, 0x1u);
          mbar_wait(cp_drain_bar, 0, tmo, never_abort);
        }
        if (!ok && lane == 0) record_timeout(p.status, kRoleProducer, abort_flag);
        __syncwarp();
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if constexpr (C::CG > 1) {
    cluster_arrive();
    cluster_wait();
  }
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc<C::CG>(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

struct KernelVariant {
  int kind;
  int cg;
  int bn;
  int tile_m;    // output-tile rows (whole CTA pair)
  int epi_cols;  // columns of one epilogue TMA store box (64: 128-byte swizzle, 32: 64-byte swizzle)
  int stages;
  int epi_warps;
  int threads;
  int smem_bytes;
  int launch_regs;  // registers a thread the kernel must be launched with (register split), else 0
  const char* name;
  const void* func;
};

template <class C>
KernelVariant make_variant(const char* name) {
  return KernelVariant{static_cast<int>(C::KIND), C::CG,        C::BN,      C::TILE_M,    C::EPI_COLS,
                       C::STAGES,                 C::EPI_WARPS, C::THREADS, C::SMEM_BYTES, C::REG_SPLIT ? 128 : 0, name,
                       reinterpret_cast<const void*>(&tkg_gemm_kernel<C>)};
}

}  // namespace tkg
