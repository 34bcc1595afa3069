// attention.cu — non-causal attention forward on sm_103a:
//   O[b,h] = softmax(Q[b,h] · K[b,h]ᵀ / √D) · V[b,h],  bf16 in and out, fp32
//   scores, softmax statistics and accumulation, plus the log-sum-exp of every
//   score row.
//
// The attention example of "ThunderKittens: Simple, Fast, and Adorable AI
// Kernels" ("The Four Functions: Load, Compute, Store, Finish"; Figure 5) and
// the attention prefill of the ThunderKittens DSL page ("Реальный пример:
// attention prefill") use the same template as the GEMM: one warp loads K and
// V tiles through a shared-memory ring while compute workers run Q·Kᵀ, an
// online softmax (subtract the running row maximum, exponentiate, keep the
// running row sum), a conversion of the probabilities to bf16 and P·V; the
// finish step divides by the row sum and stores O.  Q stays in shared memory
// for the whole task.  Re-cast for tcgen05, two 128-row query tiles (A, B)
// per CTA sharing the K and V tiles:
//   warp 0, one lane   LOAD     TMA (3-D maps over [B·H][N][D]) of both Q tiles
//                               once and of K_j, V_j into two rings
//   warp 1, one lane   COMPUTE  per query tile t: S_t(j) = Q_t·K_jᵀ into the
//                               tile's TMEM score buffer
//   warp 2, one lane   COMPUTE  O_t += P_t(j)·V_j into the tile's TMEM
//                               accumulator (P read from tensor memory, V as an
//                               MN-major shared operand)
//   warps 3-6 (A),     SOFTMAX  one thread per query row (its TMEM lane): scores
//   warps 7-10 (B)     / FINISH from TMEM, running max and sum, P_t(j) (bf16)
//                               written over the first half of the tile's
//                               score buffer, rescale of the row's O when its
//                               maximum grew; at the end O / l to bf16, a TMA
//                               store, the log-sum-exp
// The tensor core runs P_A(j)·V_j, S_A(j+1), P_B(j)·V_j, S_B(j+1), ...: while
// one tile's softmax runs, the tensor core has the other tile's P·V and next
// scores to compute, and with two issuing threads one of them waits on its
// barriers while the other's MMAs keep the tensor core fed (the tensor core
// queues only one or two MMAs ahead).  At D = 64 tensor memory has room for P
// columns of each tile's own, so the next scores wait only until the softmax
// has read the previous ones.  P never touches shared memory.  Every wait is bounded
// (TKG_OPT_TIMEOUT_NS) and reported through the status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "gemm_variants.h"
#include "tkg.h"

namespace tkg {
namespace {

struct AttnParams {
  CUtensorMap tmap_q;  // [B·H][Nq][D] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap tmap_k;  // [B·H][Nkv][D]
  CUtensorMap tmap_v;
  CUtensorMap tmap_o;  // [B·H][Nq][D], box 64 x 32 x 1
  float* lse;          // [B·H][Nq] fp32 or null
  unsigned int* status;
  unsigned long long timeout_ns;
  int Nq, Nkv;
  int fault_mode;  // 2: the producer skips the K copies of the first key tile (timeout test)
  float scale_log2;  // log2(e) / sqrt(D): scores enter exp2 pre-multiplied by it
  float scale;       // 1 / sqrt(D)
};

template <int D>
struct AttnCfg {
  static constexpr int BQ = 128;             // query rows per tile (TMEM lanes)
  static constexpr int NT = 2;               // query tiles per CTA
  static constexpr int BKV = 128;            // keys per tile
  static constexpr int DC = D / 64;          // 128-byte column chunks of a Q/K/V row
  static constexpr int CHUNK = 128 * 128;    // [128 rows][128 B] swizzled tile
  static constexpr int KST = D == 128 ? 2 : 3;  // K ring depth
  static constexpr int VST = D == 128 ? 2 : 3;  // V ring depth
  static constexpr int KV_STAGE = DC * CHUNK;
  static constexpr int Q_TILE = DC * CHUNK;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KST * KV_STAGE;
  static constexpr int OFF_Q = OFF_V + VST * KV_STAGE;  // tile t at OFF_Q + t * Q_TILE; the output staging at the end
  static constexpr int OFF_BAR = OFF_Q + NT * Q_TILE;
  static constexpr int NUM_BARS = 1 + 2 * KST + 2 * VST + 6 * NT + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 96 + 32 * 4 * NT;  // producer, two MMA issuers, a softmax warpgroup per query tile
  // TMEM columns: tile t's score buffer at 128 t (its P, bf16 pairs, over the
  // first 64 of them once the scores are read), its output accumulator at 256 + D t
  // D = 64: room for P columns of its own per tile (S 128, P 64, O 64 per tile), so the
  // next scores wait only until the softmax has read the previous ones
  static constexpr bool SEP_P = (D == 64);
  static constexpr uint32_t T_S = 0, T_O = (SEP_P ? 192 : 128) * NT;
  static constexpr uint32_t S_STRIDE = SEP_P ? 192 : 128;  // tile t's scores at T_S + S_STRIDE t
  static constexpr uint32_t P_OFF = SEP_P ? 128 : 0;       // its P at T_S + S_STRIDE t + P_OFF
  static constexpr uint32_t TMEM_COLS = 512;
  // S = Q·Kᵀ: M = 128, N = BKV, both K-major;  O += P·V: M = 128, N = D, P from
  // tensor memory, V an MN-major shared operand (bit 16)
  static constexpr uint32_t IDESC_S = idesc_dense(kFmtBF16, BQ, BKV);
  static constexpr uint32_t IDESC_PV = idesc_dense(kFmtBF16, BQ, D) | (1u << 16);
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  static_assert(T_O + NT * D <= TMEM_COLS, "tensor memory has 512 columns");
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB shared-memory limit");
  // more than half of the SM's shared memory: one CTA per SM, so the 512-column
  // TMEM allocation never waits for another CTA of this kernel
  static_assert(SMEM_BYTES > 116 * 1024, "one CTA per SM");
};

constexpr int kRoleLoad = 0, kRoleMma = 1, kRoleSoftmax = 2;

// Paired fp32 arithmetic (two lanes of a 64-bit register, each rounded as the
// scalar instruction would be) and the three-input maximum: the same results
// as the scalar forms in fewer issued instructions.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void attn_timeout(unsigned int* status, int role, volatile int* abort_flag) {
  atomicOr(status, 1u | (1u << (8 + role)));
  *abort_flag = 1;
}

template <int D>
__global__ void __launch_bounds__(AttnCfg<D>::THREADS, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using C = AttnCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sQ = sbase + C::OFF_Q;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t q_full = bar0;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + C::KST + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * C::KST + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * C::KST + C::VST + s); };
  constexpr int B1 = 1 + 2 * C::KST + 2 * C::VST;
  // query tile t: S_t(j) is in its score buffer / P_t(j) was written (and O_t rescaled) /
  // P_t(j)·V_j has finished (the score buffer is free, O_t holds key tiles 0..j)
  auto s_full = [&](int t) { return bar0 + 8u * (B1 + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (B1 + C::NT + t); };
  auto pv_done = [&](int t) { return bar0 + 8u * (B1 + 2 * C::NT + t); };
  // S_t(j) has been issued (the P·V thread keeps the tensor core's order P_A·V, S_A, P_B·V, S_B)
  auto s_issued = [&](int t) { return bar0 + 8u * (B1 + 3 * C::NT + t); };
  // separate P columns (D = 64): S_t(j) has been read into the softmax warps' registers
  auto s_loaded = [&](int t) { return bar0 + 8u * (B1 + 4 * C::NT + t); };
  // tile t's last P·V has finished (its finish need not wait for the other tile's)
  auto o_final = [&](int t) { return bar0 + 8u * (B1 + 5 * C::NT + t); };
  const uint32_t drain = bar0 + 8u * (B1 + 6 * C::NT);  // both issuers' MMAs finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = static_cast<int>(blockIdx.x) * C::BQ * C::NT;
  const int bh = static_cast<int>(blockIdx.y);
  const int nkv = (p.Nkv + C::BKV - 1) / C::BKV;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < C::NT; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 4);  // one arrival per warp of the tile's softmax warpgroup
      mbar_init(pv_done(t), 1);
      mbar_init(s_issued(t), 1);
      mbar_init(s_loaded(t), 4);  // one arrival per warp of the tile's softmax warpgroup
    }
    for (int t = 0; t < C::NT; ++t) mbar_init(o_final(t), 1);
    mbar_init(drain, 2);
    *abort_flag = 0;
    *never_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmap_q);
    tma_prefetch_desc(&p.tmap_k);
    tma_prefetch_desc(&p.tmap_v);
    tma_prefetch_desc(&p.tmap_o);
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the previous kernel on the stream may still be writing Q, K, V or reading O
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ LOAD
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(q_full, C::NT * C::Q_TILE);
#pragma unroll
      for (int t = 0; t < C::NT; ++t)
#pragma unroll
        for (int c = 0; c < C::DC; ++c)
          tma_load_3d(sQ + t * C::Q_TILE + c * C::CHUNK, &p.tmap_q, q_full, 64 * c, q0 + t * C::BQ, bh);
      for (int j = 0; j < nkv && ok; ++j) {
        const int ks = j % C::KST, vs = j % C::VST;
        if (!mbar_wait(k_empty(ks), (static_cast<uint32_t>(j / C::KST) & 1u) ^ 1u, tmo, abort_flag)) {
          ok = false;
          break;
        }
        if (!(j == 0 && p.fault_mode == 2)) {
          mbar_arrive_expect_tx(k_full(ks), C::KV_STAGE);
#pragma unroll
          for (int c = 0; c < C::DC; ++c)
            tma_load_3d(sK + ks * C::KV_STAGE + c * C::CHUNK, &p.tmap_k, k_full(ks), 64 * c, j * C::BKV, bh);
        }
        if (!mbar_wait(v_empty(vs), (static_cast<uint32_t>(j / C::VST) & 1u) ^ 1u, tmo, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(v_full(vs), C::KV_STAGE);
#pragma unroll
        for (int c = 0; c < C::DC; ++c)
          tma_load_3d(sV + vs * C::KV_STAGE + c * C::CHUNK, &p.tmap_v, v_full(vs), 64 * c, j * C::BKV, bh);
      }
      if (!ok) {
        attn_timeout(p.status, kRoleLoad, abort_flag);
        const uint64_t t0 = globaltimer_ns();  // let issued copies land before the CTA leaves
        while (globaltimer_ns() - t0 < 50000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ COMPUTE
    // Two issuing threads: warp 1 issues the score products S_t(j), warp 2
    // the products P_t(j)·V_j, so that one waits on its barriers while the
    // other's MMAs keep the tensor core busy.  The tensor core is kept to the
    // order P_A(j)·V_j, S_A(j+1), P_B(j)·V_j, S_B(j+1): each tile's softmax
    // runs between its S_t(j+1) and its P_t(j+1)·V_{j+1}, while the other
    // tile's products are computed.  S_t(j+1) overwrites the score buffer
    // P_t(j) was read from, and MMAs on different accumulators are not ordered
    // by the hardware, so it waits until P_t(j)·V_j has finished; a P·V waits
    // until the score product before it in that order has been issued.  Each
    // thread's commits track its own MMAs.  Each barrier's phases are waited
    // on in order.
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, tmo, abort_flag);
      tc_fence_after();
      if (warp == 1) {
        for (int j = 0; j < nkv && ok; ++j) {
          for (int t = 0; t < C::NT && ok; ++t) {
            // the wait that usually has completed first, the ordering one last: once it is seen,
            // the MMAs go out at once
            if (t == 0 && !mbar_wait(k_full(j % C::KST), static_cast<uint32_t>(j / C::KST) & 1u, tmo, abort_flag)) {
              ok = false;
              break;
            }
            // the score buffer is free once S_t(j-1) has been read (P elsewhere) or, with P over
            // the scores, once P_t(j-1)·V_{j-1} has finished
            if (j > 0 && !mbar_wait(C::SEP_P ? s_loaded(t) : pv_done(t), static_cast<uint32_t>(j - 1) & 1u, tmo,
                                    abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t k0 = sK + (j % C::KST) * C::KV_STAGE;
            const uint32_t q_t = sQ + t * C::Q_TILE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(q_t + (kk / 4) * C::CHUNK + 32u * (kk % 4));
              const uint64_t bd = sdesc_sw128(k0 + (kk / 4) * C::CHUNK + 32u * (kk % 4));
              mma_bf16<1>(tmem_base + C::T_S + C::S_STRIDE * t, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
            }
            if constexpr (!C::SEP_P) mbar_arrive_local(s_issued(t));
            mma_commit_local(s_full(t));
            if (t == C::NT - 1) mma_commit_local(k_empty(j % C::KST));  // the last reader of K_j
          }
        }
      } else {
        for (int j = 0; j < nkv && ok; ++j) {
          for (int t = 0; t < C::NT && ok; ++t) {
            // P and V (usually ready) first; last the score product that goes before this P·V
            // in the tensor core's order: S_B(j) for tile A, S_A(j+1) for tile B
            if (!mbar_wait(p_full(t), static_cast<uint32_t>(j) & 1u, tmo, abort_flag)) {
              ok = false;
              break;
            }
            if (t == 0 && !mbar_wait(v_full(j % C::VST), static_cast<uint32_t>(j / C::VST) & 1u, tmo, abort_flag)) {
              ok = false;
              break;
            }
            // (not with P in columns of its own: the score thread then runs up to two products
            // ahead, past what a parity wait on this barrier can tell apart, and the order is free)
            const int tp = (t + C::NT - 1) % C::NT;
            const int jp = t == 0 ? j : j + 1;
            if (!C::SEP_P && jp < nkv &&
                !mbar_wait(s_issued(tp), static_cast<uint32_t>(jp) & 1u, tmo, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t v0 = sV + (j % C::VST) * C::KV_STAGE;
            const uint32_t a0 = tmem_base + C::T_S + C::S_STRIDE * t + C::P_OFF;  // P_t(j), bf16 pairs
#pragma unroll
            for (int kk = 0; kk < C::BKV / 16; ++kk) {
              // A: 16 keys of P_t = 8 of its columns; B: 16 rows of V (keys), D columns
              const uint64_t bd = sdesc_sw128_mn(v0 + 2048u * kk, C::CHUNK);
              mma_bf16_ts(tmem_base + C::T_O + static_cast<uint32_t>(D * t), a0 + 8u * kk, bd, C::IDESC_PV,
                          (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_local(pv_done(t));
            if (t == C::NT - 1) mma_commit_local(v_empty(j % C::VST));  // the last reader of V_j
            if (j == nkv - 1) mma_commit_local(o_final(t));
          }
        }
      }
      // no MMA of either thread may still be writing TMEM when it is released
      mma_commit_local(drain);
      mbar_wait(drain, 0, tmo, never_abort);
      if (!ok) attn_timeout(p.status, kRoleMma, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ SOFTMAX / FINISH
    // Warpgroup t (warps 3+4t .. 6+4t) owns query tile t, one thread per row
    // (its TMEM lane).
    const int t = (warp - 3) / 4;
    const int quad = warp & 3;  // TMEM lane quarter this warp may access (rows 32 quad ..)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_s = tmem_base + lane_off + C::T_S + C::S_STRIDE * static_cast<uint32_t>(t);
    const uint32_t t_p = t_s + C::P_OFF;  // P: its own columns, or over the scores once they are read
    const uint32_t t_o = tmem_base + lane_off + C::T_O + static_cast<uint32_t>(D * t);
    const float c2 = p.scale_log2;
    float m = -INFINITY;  // reference maximum of the raw scores of this row (lazily raised)
    float l = 0.0f;       // running sum of exp2((s - m) * c2)
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait<true>(s_full(t), static_cast<uint32_t>(j) & 1u, tmo, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x32(t_s + 32u * q, s[q]);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) reg_fence(s[q]);
      if constexpr (C::SEP_P) {
        // the scores are in registers: the buffer may take the next ones
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_local(s_loaded(t));
      }
      // keys of this tile past the end of the sequence score -inf (only the last tile has any)
      const int valid = p.Nkv - j * C::BKV;
      if (valid < C::BKV) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * q + i >= valid) s[q][i] = __float_as_uint(-INFINITY);
      }
      // tile row maximum: eight independent chains of three-input maxima, then a tree
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(s[0][e]);
#pragma unroll
      for (int e = 8; e < 128; e += 16)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          mx[c] = fmax3(mx[c], __uint_as_float(s[(e + c) / 32][(e + c) % 32]),
                        __uint_as_float(s[(e + 8 + c) / 32][(e + 8 + c) % 32]));
#pragma unroll
      for (int w = 4; w >= 1; w /= 2)
#pragma unroll
        for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
      const float mt = mx[0];
      // Lazy reference maximum: the row keeps m (and so its O and l) until a
      // tile's maximum exceeds it by more than 8 in exp2 units, so that every
      // probability stays <= 2^8; only then is m raised and O, l rescaled.  The
      // result is the same softmax: m cancels between O and l.  The first tile
      // always sets m (m = -inf, alpha = 0).
      float alpha = 1.0f;
      if ((mt - m) * c2 > 8.0f) {
        alpha = ex2_approx((m - mt) * c2);
        m = mt;
      }
      const float neg = -m * c2;
      // scores scaled in pairs (s * c2 - m * c2), exponentiated, summed in pairs: sum k
      // (k = 0..3) collects the pairs i = k, k + 4, ...; lane 0 the even, lane 1 the odd keys
      const uint64_t c2x2 = f32x2_pack(c2, c2), negx2 = f32x2_pack(neg, neg);
      uint64_t lsx2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[64];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t y = f32x2_fma(f32x2_pack(__uint_as_float(s[q][2 * i]), __uint_as_float(s[q][2 * i + 1])),
                                       c2x2, negx2);
          float y0, y1;
          f32x2_unpack(y, y0, y1);
          const float x0 = ex2_approx(y0);
          const float x1 = ex2_approx(y1);
          lsx2[i % 4] = f32x2_add(lsx2[i % 4], f32x2_pack(x0, x1));
          pk[16 * q + i] = pack_bf16x2(x0, x1);
        }
      float ls[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) f32x2_unpack(lsx2[k], ls[2 * k], ls[2 * k + 1]);
#pragma unroll
      for (int w = 4; w >= 1; w /= 2)
#pragma unroll
        for (int e = 0; e < w; ++e) ls[e] += ls[e + w];
      l = l * alpha + ls[0];
      // P_t(j) may be written and O_t rescaled once P_t(j-1)·V_{j-1} has finished: with P over
      // the scores that was so before S_t(j) was issued; with P in its own columns, wait for it
      if constexpr (C::SEP_P) {
        if (j >= 1 && !__all_sync(0xffffffffu, mbar_wait<true>(pv_done(t), static_cast<uint32_t>(j - 1) & 1u, tmo,
                                                                abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // O_t holds key tiles 0..j-1
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + 32u * q, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32x32b_x32(t_o + 32u * q, o);
        }
      }
      // P row (bf16 pairs)
      tmem_st_32x32b_x32(t_p, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st_32x32b_x32(t_p + 32u, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_local(p_full(t));
    }
    if (ok && !__all_sync(0xffffffffu, mbar_wait<true>(o_final(t), 0, tmo, abort_flag))) ok = false;
    if (ok) {
      // FINISH: O / l to bf16, staged per warp ([32 rows][128 B] per 64 columns) in the tile's Q buffer
      tc_fence_after();
      const float inv = 1.0f / l;
      const uint32_t stg = sQ + static_cast<uint32_t>(t * C::Q_TILE + quad * C::DC * 4096);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(t_o + 32u * q, o);
        tmem_wait_ld();
        uint32_t ob[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          ob[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        const uint32_t chunk = stg + static_cast<uint32_t>(q / 2) * 4096u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t off = swizzle_offset(static_cast<uint32_t>(lane) * 128u + 16u * (4 * (q % 2) + u), 128u);
          st_shared_v4(chunk + off, ob[4 * u], ob[4 * u + 1], ob[4 * u + 2], ob[4 * u + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int row0 = q0 + t * C::BQ + quad * 32;
      if (lane == 0) {
#pragma unroll
        for (int c = 0; c < C::DC; ++c) tma_store_3d(&p.tmap_o, stg + c * 4096u, 64 * c, row0, bh);
        bulk_commit_group();
        bulk_wait_group<0>();
      }
      if (p.lse != nullptr && row0 + lane < p.Nq)
        p.lse[static_cast<size_t>(bh) * p.Nq + row0 + lane] = m * p.scale + logf(l);
    } else if (lane == 0) {
      attn_timeout(p.status, kRoleSoftmax, abort_flag);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, C::TMEM_COLS);
  }
}

template <int D>
tkg_status attn_launch(int64_t BH, int64_t Nq, int64_t Nkv, const void* Q, const void* K, const void* V, void* O,
                       float* lse, cudaStream_t stream, unsigned long long timeout_ns, bool overlap) {
  using C = AttnCfg<D>;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  const uint64_t row_bytes = static_cast<uint64_t>(D) * 2;
  const uint64_t dq[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nq), static_cast<uint64_t>(BH)};
  const uint64_t dk[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nkv), static_cast<uint64_t>(BH)};
  const uint64_t sq[2] = {row_bytes, row_bytes * static_cast<uint64_t>(Nq)};
  const uint64_t sk[2] = {row_bytes, row_bytes * static_cast<uint64_t>(Nkv)};
  const uint32_t box_in[3] = {64, 128, 1};
  const uint32_t box_out[3] = {64, 32, 1};
  tkg_status st = encode_tiled_map(&p.tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, Q, dq, sq, box_in, 128);
  if (st == TKG_OK) st = encode_tiled_map(&p.tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, K, dk, sk, box_in, 128);
  if (st == TKG_OK) st = encode_tiled_map(&p.tmap_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, V, dk, sk, box_in, 128);
  if (st == TKG_OK) st = encode_tiled_map(&p.tmap_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, O, dq, sq, box_out, 128);
  if (st != TKG_OK) return st;
  st = device_status_word(&p.status);
  if (st != TKG_OK) return st;
  p.lse = lse;
  p.fault_mode = take_fault_mode(2);
  p.timeout_ns = timeout_ns;
  p.Nq = static_cast<int>(Nq);
  p.Nkv = static_cast<int>(Nkv);
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));

  // the shared-memory opt-in is per device: set it once on each
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  if (!(attr_set.load() & (1ull << dev))) {
    if (cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
        cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    attr_set.fetch_or(1ull << dev);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((Nq + C::BQ * C::NT - 1) / (C::BQ * C::NT)), static_cast<unsigned>(BH), 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D>, p) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}

}  // namespace
}  // namespace tkg

extern "C" tkg_status tkg_attention_fwd(int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D, const void* Q,
                                        const void* K, const void* V, void* O, float* lse, void* stream) {
  using namespace tkg;
  const int64_t kMax = 0x7FFFFFFF;
  if (B < 1 || H < 1 || Nq < 1 || Nkv < 1 || Nq > kMax || Nkv > kMax) return TKG_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TKG_ERR_INVALID_ARG;
  if (B * H > 65535 || (Nq + 127) / 128 > kMax) return TKG_ERR_INVALID_ARG;  // grid y limit
  if (!Q || !K || !V || !O) return TKG_ERR_INVALID_ARG;
  auto a16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  if (!a16(Q) || !a16(K) || !a16(V) || !a16(O) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return TKG_ERR_MISALIGNED;
  const unsigned long long tmo = static_cast<unsigned long long>(tkg_get_option(TKG_OPT_TIMEOUT_NS));
  const bool overlap = tkg_get_option(TKG_OPT_LAUNCH_OVERLAP) == TKG_OVERLAP_ON;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return D == 128 ? attn_launch<128>(B * H, Nq, Nkv, Q, K, V, O, lse, s, tmo, overlap)
                  : attn_launch<64>(B * H, Nq, Nkv, Q, K, V, O, lse, s, tmo, overlap);
}
