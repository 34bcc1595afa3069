// probes.cu — diagnostic kernels behind tkg_debug.h: a TMA swizzled load whose
// raw shared-memory image is copied out, a one-tile tensor-core MMA with
// caller-chosen operands and (for the block-scaled kind) caller-chosen
// tensor-memory contents of the scale regions.  Each checks one building block
// of the GEMM in isolation.
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
  if (kind < 0 || kind > 2 || !(n == 64 || n == 128 || n == 192 || n == 256) || ksteps < 1 || ksteps > 4 || !a_tile ||
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

}  // extern "C"
