// gemm_nvfp4_noalloc.cu — an NVFP4 GEMM entry point that allocates nothing.
//
// The regular NVFP4 entry point takes its scale-interleave scratch from a
// stream-ordered memory pool.  Some callers cannot allocate device memory at
// call time: code running while a CUDA graph is being captured into a region
// whose allocations are forbidden, runtimes that hand the library a fixed
// memory budget, or hosts where any cudaMalloc/cudaFree would synchronise or
// fragment memory another framework manages.  For them this file provides
// tkg_gemm_nvfp4_noalloc: the same two kernels (scale interleave + block-scaled
// GEMM), with the scratch placed in a file-scope device array of fixed size.
//
// Host code never dereferences the array: its name in host code stands for a
// host-side shadow, so the device address is looked up with
// cudaGetSymbolAddress once per device (on that device's first call) and that
// address is what the kernels receive.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gemm_variants.h"
#include "tkg.h"
#include "tkg_debug.h"

namespace tkg {
tkg_status status_word_address(unsigned int** out);
}

// Scratch shared by every call of tkg_gemm_nvfp4_noalloc on a device.
static __device__ __align__(256) uint8_t g_nvfp4_noalloc_scratch[TKG_NVFP4_NOALLOC_SCRATCH_BYTES];

namespace {

using namespace tkg;

constexpr int kMaxDev = 64;

struct NoAllocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;   // device address of g_nvfp4_noalloc_scratch
  unsigned int* status = nullptr;
  int sm_count = 0;
};
NoAllocDevice g_na[kMaxDev];
std::mutex g_na_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// First call on a device: check the device, look up the scratch and status
// addresses.  No memory is allocated.
tkg_status noalloc_setup(int dev, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  NoAllocDevice& d = g_na[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    if (!(major == 10 && minor == 3)) return TKG_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_nvfp4_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    d.scratch = static_cast<uint8_t*>(p);
    if (status_word_address(&d.status) != TKG_OK) return TKG_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return TKG_OK;
}

tkg_status encode(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t pitch,
                  uint32_t b0, uint32_t b1, bool swizzle128) {
  const cuuint64_t dims[2] = {d0, d1};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {b0, b1};
  const cuuint32_t estr[2] = {1, 1};
  std::memset(m, 0, sizeof(*m));
  CUresult r = g_na_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TKG_OK : TKG_ERR_INVALID_ARG;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" tkg_status tkg_gemm_nvfp4_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                                             const tkg_scales* scales, void* stream) {
  const int64_t kMax = 0x7FFFFFFF;
  if (M < 1 || N < 1 || K < 1 || M > kMax || N > kMax || K > kMax || K % 32 != 0) return TKG_ERR_INVALID_ARG;
  if (!A || !B || !C || !scales || !scales->a_scale || !scales->b_scale || !scales->a_block_scale ||
      !scales->b_block_scale)
    return TKG_ERR_INVALID_ARG;
  if (!al16(A) || !al16(B) || !al16(C) || !al16(scales->a_block_scale) || !al16(scales->b_block_scale) ||
      (reinterpret_cast<uintptr_t>(scales->a_scale) & 3u) || (reinterpret_cast<uintptr_t>(scales->b_scale) & 3u))
    return TKG_ERR_MISALIGNED;

  const int id = tkg_debug_pick_variant(2, M, N, K);
  const KernelVariant* v = nvfp4_variant(id);
  if (!v) return TKG_ERR_INTERNAL;
  const int64_t tiles_m = (M + 128LL * v->cg - 1) / (128LL * v->cg);
  const int64_t tiles_n = (N + v->bn - 1) / v->bn;
  const int64_t num_kb = (K / 2 + 127) / 128;
  const int64_t blocks_a = tiles_m * v->cg;
  const int64_t blocks_b = tiles_n * (v->bn / 128);
  const int64_t need = (blocks_a + blocks_b) * num_kb * 2048;
  // The fixed scratch bounds the problem size: reject before touching the GPU.
  if (tiles_m * tiles_n > kMax || need > static_cast<int64_t>(TKG_NVFP4_NOALLOC_SCRATCH_BYTES))
    return TKG_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  NoAllocDevice* d = nullptr;
  tkg_status st = noalloc_setup(dev, &d);
  if (st != TKG_OK) return st;

  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.num_kb = static_cast<int>(num_kb);
  p.sf_blocks_a = static_cast<int>(blocks_a);
  p.sf_blocks_b = static_cast<int>(blocks_b);
  const size_t b_off = static_cast<size_t>(blocks_a) * num_kb * 2048;
  uint8_t* scratch = d->scratch;
  st = encode(&p.tmap_a, A, CU_TENSOR_MAP_DATA_TYPE_UINT8, K / 2, M, K / 2, 128, 128, true);
  if (st == TKG_OK)
    st = encode(&p.tmap_b, B, CU_TENSOR_MAP_DATA_TYPE_UINT8, K / 2, N, K / 2, 128,
                static_cast<uint32_t>(v->bn / v->cg), true);
  if (st == TKG_OK)
    st = encode(&p.tmap_sfa, scratch, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128, static_cast<uint64_t>(blocks_a) * num_kb * 16,
                128, 128, 16, false);
  if (st == TKG_OK)
    st = encode(&p.tmap_sfb, scratch + b_off, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128,
                static_cast<uint64_t>(blocks_b) * num_kb * 16, 128, 128, static_cast<uint32_t>(16 * (v->bn / 128)),
                false);
  p.c_via_tma = (N % 8 == 0) ? 1 : 0;
  if (st == TKG_OK && p.c_via_tma)
    st = encode(&p.tmap_c, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, N * 2, static_cast<uint32_t>(v->epi_cols), 32,
                v->epi_cols == 64);
  if (st != TKG_OK) return st;
  p.c_ptr = C;
  p.a_scale = scales->a_scale;
  p.b_scale = scales->b_scale;
  p.status = d->status;
  p.timeout_ns = static_cast<unsigned long long>(tkg_get_option(TKG_OPT_TIMEOUT_NS));
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.tiles_m = static_cast<int>(tiles_m);
  p.tiles_n = static_cast<int>(tiles_n);
  p.group_m = static_cast<int>(tkg_get_option(TKG_OPT_GROUP_M));
  p.fault_mode = 0;

  // Every byte of the region this call uses is rewritten by the interleave
  // kernel (zeros for padding), so no clearing is needed between calls.
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (nvfp4_interleave_scales(scales->a_block_scale, scales->b_block_scale, static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), p.sf_blocks_a, p.sf_blocks_b, p.num_kb, v->sf_mode, scratch,
                              b_off, cs, false) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  p.sf_a = scratch;
  p.sf_b = scratch + b_off;

  if (cudaFuncSetAttribute(v->func, cudaFuncAttributeMaxDynamicSharedMemorySize, v->smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(v->cg);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(static_cast<unsigned>(v->threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(v->smem_bytes);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(v->cg * d->sm_count), 1, 1);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, v->func, &cfg) != cudaSuccess || clusters <= 0) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  int64_t grid_clusters = clusters;
  const int64_t cap = tkg_get_option(TKG_OPT_MAX_CTAS);
  if (cap > 0 && cap / v->cg < grid_clusters) grid_clusters = cap / v->cg > 0 ? cap / v->cg : 1;
  if (tiles_m * tiles_n < grid_clusters) grid_clusters = tiles_m * tiles_n;
  cfg.gridDim = dim3(static_cast<unsigned>(grid_clusters * v->cg), 1, 1);
  cfg.stream = cs;
  void* args[] = {&p};
  if (cudaLaunchKernelExC(&cfg, v->func, args) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}
