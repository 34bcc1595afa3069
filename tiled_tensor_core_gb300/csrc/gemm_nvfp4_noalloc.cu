// gemm_nvfp4_noalloc.cu — an NVFP4 GEMM entry point that allocates nothing.
//
// The regular NVFP4 entry point takes the scratch for its on-device re-layout
// of the block scales from a stream-ordered memory pool, and may make a
// per-stream split-K workspace.  Some callers cannot allocate device memory at
// call time: code that runs while a CUDA graph is being captured into a region
// whose allocations are forbidden, runtimes that hand the library a fixed
// memory budget, or hosts where a cudaMalloc / cudaFree would synchronise or
// fragment memory that another framework manages.  For them this file provides
// tkg_gemm_nvfp4_noalloc: the same two kernels (scale re-layout + block-scaled
// GEMM), planned, parameterised and launched by the same code as
// tkg_gemm_nvfp4 (api.cu), with the scratch placed in a file-scope device array
// of fixed size and without the split-K head.  Tensor maps are encoded on the
// stack (no host-side cache entry either).
//
// Host code never dereferences the array: its name in host code stands for a
// host-side shadow, so the device address is looked up with
// cudaGetSymbolAddress once per device (on that device's first call, with the
// device current) and that address is what the kernels receive.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gemm_variants.h"
#include "tkg.h"

// Scratch shared by every call of tkg_gemm_nvfp4_noalloc on a device.
static __device__ __align__(256) uint8_t g_nvfp4_noalloc_scratch[TKG_NVFP4_NOALLOC_SCRATCH_BYTES];

namespace {

using namespace tkg;

constexpr int kMaxDev = 64;
uint8_t* g_scratch_addr[kMaxDev] = {};  // device address of the array, per device (set once)
std::mutex g_na_mu;

// The current device's address of the scratch array (looked up on the
// device's first call).  No memory is allocated.
tkg_status scratch_address(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_nvfp4_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return TKG_OK;
}

}  // namespace

extern "C" tkg_status tkg_gemm_nvfp4_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                                             const tkg_scales* scales, void* stream) {
  tkg_status st = check_gemm_args(2, M, N, K, A, B, C, scales);
  if (st != TKG_OK) return st;
  // The NVFP4 kernel does not depend on the SM count: plan on the host first, so that a problem
  // whose staged scales would not fit the fixed scratch is rejected before any GPU work.
  GemmPlan g;
  st = plan_gemm(2, M, N, K, 0, &g);
  if (st != TKG_OK) return st;
  if (g.sf_bytes > static_cast<size_t>(TKG_NVFP4_NOALLOC_SCRATCH_BYTES)) return TKG_ERR_INVALID_ARG;
  uint8_t* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != TKG_OK) return st;
  // Every byte of the region this call uses is rewritten by the re-layout
  // kernel (zeros for padding), so no clearing is needed between calls.
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (nvfp4_interleave_scales(scales->a_block_scale, scales->b_block_scale, static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), g.sf_blocks_a, g.sf_blocks_b, g.num_kb, scratch, g.sf_b_off, cs,
                              launch_overlap()) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  GemmParams p;
  st = gemm_params(&p, g, 2, M, N, K, A, B, C, scales, scratch, false);
  if (st != TKG_OK) return st;
  return gemm_enqueue(2, g, p, stream, false);
}
