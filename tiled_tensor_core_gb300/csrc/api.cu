// api.cu — the tkg C ABI: argument validation, TMA tensor-map construction and
// caching, per-device launch data, variant choice and the persistent launch.
//
// Tensor maps are the host-side half of the TMA path: they carry the global
// shape, pitch, tile box and swizzle of each operand so that the copy engine
// computes every address ("Asynchronous I/O: Unified Interface over cp.async
// and TMA" — TK builds them from its global layout descriptors).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "gemm_variants.h"
#include "tkg.h"
#include "tkg_debug.h"

// Device status word (one per device, lives as long as the module).
static __device__ unsigned int g_tkg_status;

namespace {

using namespace tkg;

constexpr int64_t kDefaultTimeoutNs = 2000000000LL;
// Super-group height of the tile order: 16 tile rows measured best on GB300's 76 CTA pairs with
// 256-row pair tiles (NVFP4 16384^3 DRAM reads 1.13 GB at 16 against 1.47 / 2.79 / 2.82 GB at
// 8 / 4 / 32; bf16 8192^3 846 MB against 889 / 1271 / 1133 MB), where the pages' H100 GEMM takes 8
constexpr int64_t kDefaultGroupM = 16;
constexpr int kMaxSplit = 4;     // split-K head: at most 4 pieces per tile
constexpr int kMinSplitKb = 16;  // of at least 16 K blocks each
constexpr int kMinSplitKbOneRound = 48;  // and, when all tiles fit in one round, 48 K blocks a tile
constexpr int kMaxDevices = 64;
constexpr int kNumKinds = 3;

std::atomic<int64_t> g_opt_timeout{0};
std::atomic<int64_t> g_opt_group{0};
std::atomic<int64_t> g_opt_variant{0};
std::atomic<int64_t> g_opt_max_ctas{0};
std::atomic<int64_t> g_opt_overlap{0};
std::atomic<int64_t> g_opt_schedule{0};
std::atomic<int64_t> g_opt_split{0};
std::atomic<int64_t> g_opt_k_order{0};
std::atomic<int> g_fault{0};
std::atomic<unsigned int*> g_visits{nullptr};

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct DevState {
  bool ready = false;
  int dev = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned int* status = nullptr;
  int max_clusters[kNumKinds][kNumVariants] = {};
  cudaMemPool_t pool = nullptr;  // stream-ordered scratch for the NVFP4 scale interleave
  // split-K head: a workspace and zeroed piece counters per stream (launches on one stream are
  // ordered, and the kernel leaves the counters at zero), created on first use outside capture
  struct SplitWs {
    float* ws = nullptr;
    unsigned int* cnt = nullptr;
  };
  std::unordered_map<cudaStream_t, SplitWs> split;
};
DevState g_dev[kMaxDevices];

struct MapKey {
  const void* ptr;
  int dtype;
  uint64_t d0, d1, pitch;
  uint32_t b0, b1;
  int swz;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dtype == o.dtype && d0 == o.d0 && d1 == o.d1 && pitch == o.pitch && b0 == o.b0 &&
           b1 == o.b1 && swz == o.swz;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = reinterpret_cast<uint64_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
    auto mix = [&](uint64_t v) { h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2); };
    mix(static_cast<uint64_t>(k.dtype));
    mix(k.d0);
    mix(k.d1);
    mix(k.pitch);
    mix((static_cast<uint64_t>(k.b0) << 32) | k.b1);
    mix(static_cast<uint64_t>(k.swz));
    return static_cast<size_t>(h);
  }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxMaps = 4096;

int64_t opt_or(const std::atomic<int64_t>& v, int64_t dflt) {
  const int64_t x = v.load(std::memory_order_relaxed);
  return x == 0 ? dflt : x;
}

// Caller holds g_mu.
tkg_status ensure_encode_locked() {
  if (g_encode) return TKG_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return TKG_OK;
}

// Per-device initialisation (device must be current).  Caller holds g_mu.
tkg_status device_state_locked(int dev, DevState** out) {
  if (dev < 0 || dev >= kMaxDevices) return TKG_ERR_UNSUPPORTED_DEVICE;
  DevState& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return TKG_ERR_UNSUPPORTED_DEVICE;
    void* sp = nullptr;
    if (cudaGetSymbolAddress(&sp, g_tkg_status) != cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    d.status = static_cast<unsigned int*>(sp);
    d.dev = dev;
    for (auto& row : d.max_clusters)
      for (int& v : row) v = 0;
    d.ready = true;
  }
  *out = &d;
  return TKG_OK;
}

// The device's stream-ordered memory pool for the NVFP4 scale scratch, made on
// the first regular NVFP4 call (the allocation-free entry point never makes it).
tkg_status device_pool(DevState& d, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!d.pool) {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = d.dev;
    if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
      cudaGetLastError();
      d.pool = nullptr;
      return TKG_ERR_CUDA;
    }
    uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse by the next call
    cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
  }
  *out = d.pool;
  return TKG_OK;
}

tkg_status current_device(DevState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  tkg_status st = ensure_encode_locked();
  if (st != TKG_OK) return st;
  return device_state_locked(dev, out);
}

// 2-D row-major tensor map: d0 = elements per row (innermost), d1 = rows,
// pitch in bytes, box b0 x b1 elements, swizzle in bytes (0/32/64/128).
// Encoded on the caller's stack, no cache.  Caller holds g_mu.
tkg_status encode_map_2d_locked(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, uint64_t d0,
                                uint64_t d1, uint64_t pitch, uint32_t b0, uint32_t b1, int swz) {
  tkg_status st = ensure_encode_locked();
  if (st != TKG_OK) return st;
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swz == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  if (swz == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swz == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const cuuint64_t dims[2] = {d0, d1};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {b0, b1};
  const cuuint32_t estr[2] = {1, 1};
  std::memset(out, 0, sizeof(*out));
  CUresult r = g_encode(out, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TKG_OK : TKG_ERR_INVALID_ARG;
}

// The same map, through the host-side cache (a miss adds an entry) unless
// `cached` is false.
tkg_status get_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1,
                   uint64_t pitch, uint32_t b0, uint32_t b1, int swz, bool cached = true) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!cached) return encode_map_2d_locked(out, ptr, dtype, d0, d1, pitch, b0, b1, swz);
  const MapKey key{ptr, static_cast<int>(dtype), d0, d1, pitch, b0, b1, swz};
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *out = it->second;
    return TKG_OK;
  }
  CUtensorMap m;
  const tkg_status st = encode_map_2d_locked(&m, ptr, dtype, d0, d1, pitch, b0, b1, swz);
  if (st != TKG_OK) return st;
  if (g_maps.size() >= kMaxMaps) g_maps.clear();
  g_maps.emplace(key, m);
  *out = m;
  return TKG_OK;
}

const KernelVariant* variant_of(int kind, int id) {
  switch (kind) {
    case 0: return bf16_variant(id);
    case 1: return fp8_variant(id);
    case 2: return nvfp4_variant(id);
    default: return nullptr;
  }
}

// Tile choice: the 2-SM 256 x 256 tile.  An MMA of N columns costs about
// max(77, N / 2) cycles on sm_103a, so narrower tiles (N = 224, 192) keep the
// tensor pipe's rate per column, but each SM then receives more operand bytes
// per flop (A is re-read for every tile column) and the measured throughput
// falls with that ratio; sharing A between two CTA pairs by TMA multicast saved
// L2 reads and power but not throughput.  NVFP4 takes the scale-warp form of
// the 256 x 256 tile with the scales riding the ring: copying the block scales
// with tcgen05.cp costs the tensor pipe about 60 cycles per copy, twelve copies
// per 256-deep K stage, and reading the scales from shared memory, where the
// ring's TMA put them stages ahead, keeps global-load latency off the scale
// warps' critical path.
//
// bf16 / FP8 with K of 2048 or more and many tiles take the 256 x 512 pair tile
// instead: it moves a third fewer operand bytes per flop, which draws less power,
// and under the power cap that buys clock (8192^3 bf16: 1779 against 1710
// TFLOP/s, at 1601 against 1507 MHz); it keeps a single accumulator, which its
// eight register-split epilogue warps read whole and hand back before storing
// (16384 x 8192 x 2048: 1787 / 1778 against 1758 / 1747 for the 256 x 256 tile),
// and coarser rounds of tiles, so it loses with few tiles (4096^3: 1609 against
// 1639, where the split-K head of the 256 x 256 tile helps more).  "Many" is
// four rounds of 256 x 512 tiles over the device's CTA pairs (SMs / 2).
constexpr int64_t kWideMinK = 2048;
constexpr int64_t kWideMinRounds = 4;
int pick_variant(int kind, int64_t M, int64_t N, int64_t K, int sm_count) {
  const int forced = static_cast<int>(g_opt_variant.load(std::memory_order_relaxed));
  if (forced > 0 && variant_of(kind, forced)) return forced;
  if (kind == 2) return kVariant2Sm256x256SfCopy;
  const int64_t wide_tiles = ((M + 255) / 256) * ((N + 511) / 512);
  if (K >= kWideMinK && wide_tiles >= kWideMinRounds * (sm_count / 2)) return kVariant2Sm256x512;
  return kVariant2Sm256x256;
}

// Occupancy-limited number of co-resident clusters for a variant (cached).
tkg_status max_clusters(DevState& d, int kind, int id, const KernelVariant& v, int* out) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (d.max_clusters[kind][id] > 0) {
      *out = d.max_clusters[kind][id];
      return TKG_OK;
    }
  }
  if (cudaFuncSetAttribute(v.func, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  // a register split hands registers between warpgroups out of what the block was launched with;
  // launched with fewer than it was written for, its setmaxnreg.inc would wait forever
  if (v.launch_regs > 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, v.func) != cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    if (fa.numRegs != v.launch_regs) return TKG_ERR_UNSUPPORTED_DEVICE;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(v.cg * d.sm_count), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(v.threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(v.smem_bytes);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(v.cg);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, v.func, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  d.max_clusters[kind][id] = n;
  *out = n;
  return TKG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Split-K head plan for `tiles` output tiles on a persistent grid of `clusters`
// clusters walking `num_kb` K blocks per tile.  The grid takes R = ceil(tiles /
// clusters) rounds, the last holding `tail` tiles; if that round would be at
// most half full, the tail tiles are cut into S = min(clusters / tail, 4,
// num_kb / 16) pieces that run first, next to whole tiles, so the grid
// finishes after R - 1 + 1/S rounds of work instead of R.  A piece's share of
// the reduction is a chain of dependent global-memory round trips (~6 us on
// GB300); pieces of at least 16 K blocks (bf16: 1024 K elements) keep it below
// what the split saves when it overlaps the next tile, and a single round (no
// next tile) needs tiles of at least 48 K blocks (measured over M = N = 1024
// and 4096, K 512 to 16384).
void split_plan(int64_t tiles, int64_t clusters, int num_kb, int* split_tiles, int* split_s) {
  *split_tiles = 0;
  *split_s = 1;
  if (tiles < 1 || clusters < 2) return;
  const int64_t rounds = (tiles + clusters - 1) / clusters;
  const int64_t tail = tiles - (rounds - 1) * clusters;
  if (2 * tail > clusters) return;
  if (rounds == 1 && num_kb < kMinSplitKbOneRound) return;
  int64_t s = clusters / tail;
  if (s > kMaxSplit) s = kMaxSplit;
  if (s > num_kb / kMinSplitKb) s = num_kb / kMinSplitKb;
  if (s < 2) return;
  *split_tiles = static_cast<int>(tail);
  *split_s = static_cast<int>(s);
}

// The stream's split workspace (created on first use; not while the stream is
// being captured, where the caller runs without the split instead).  Capacity:
// one 128 x 256 fp32 block per SM (pieces <= clusters, CTAs <= SMs) and eight
// counters per SM (tail tiles <= clusters / 2, x CTAs x epilogue warps x 2).
bool split_workspace(DevState& d, cudaStream_t stream, DevState::SplitWs* out) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = d.split.find(stream);
    if (it != d.split.end()) {
      *out = it->second;
      return true;
    }
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return false;
  }
  DevState::SplitWs w;
  const size_t ws_bytes = static_cast<size_t>(d.sm_count) * 128 * 256 * sizeof(float);
  const size_t cnt_bytes = static_cast<size_t>(d.sm_count) * 8 * sizeof(unsigned int);
  if (cudaMalloc(reinterpret_cast<void**>(&w.ws), ws_bytes) != cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&w.cnt), cnt_bytes) != cudaSuccess ||
      cudaMemsetAsync(w.cnt, 0, cnt_bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    if (w.ws) cudaFree(w.ws);
    if (w.cnt) cudaFree(w.cnt);
    return false;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto ins = d.split.emplace(stream, w);
    *out = ins.first->second;
    if (ins.second) return true;
  }
  // another thread made this stream's workspace meanwhile: use that one
  cudaFree(w.ws);
  cudaFree(w.cnt);
  cudaGetLastError();
  return true;
}

}  // namespace

namespace tkg {

tkg_status check_gemm_args(int kind, int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                           const tkg_scales* scales) {
  const int64_t kMax = 0x7FFFFFFF;
  if (M < 1 || N < 1 || K < 1 || M > kMax || N > kMax || K > kMax) return TKG_ERR_INVALID_ARG;
  const int64_t k_align = kind == 0 ? 8 : kind == 1 ? 16 : 32;
  if (K % k_align != 0) return TKG_ERR_INVALID_ARG;
  if (!A || !B || !C) return TKG_ERR_INVALID_ARG;
  if (kind == 0 && scales != nullptr) return TKG_ERR_INVALID_ARG;
  if (kind == 1 && (!scales || !scales->a_scale || !scales->b_scale || scales->a_block_scale ||
                    scales->b_block_scale))
    return TKG_ERR_INVALID_ARG;
  if (kind == 2 && (!scales || !scales->a_scale || !scales->b_scale || !scales->a_block_scale ||
                    !scales->b_block_scale))
    return TKG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return TKG_ERR_MISALIGNED;
  if (kind != 0 && ((reinterpret_cast<uintptr_t>(scales->a_scale) & 3u) ||
                    (reinterpret_cast<uintptr_t>(scales->b_scale) & 3u)))
    return TKG_ERR_MISALIGNED;
  if (kind == 2 && (!aligned16(scales->a_block_scale) || !aligned16(scales->b_block_scale)))
    return TKG_ERR_MISALIGNED;
  return TKG_OK;
}

tkg_status plan_gemm(int kind, int64_t M, int64_t N, int64_t K, int sm_count, GemmPlan* out) {
  GemmPlan g;
  g.id = pick_variant(kind, M, N, K, sm_count);
  g.v = variant_of(kind, g.id);
  if (!g.v) return TKG_ERR_INTERNAL;
  const int64_t tile_m = g.v->tile_m;
  g.tiles_m = (M + tile_m - 1) / tile_m;
  g.tiles_n = (N + g.v->bn - 1) / g.v->bn;
  if (g.tiles_m * g.tiles_n > 0x7FFFFFFF) return TKG_ERR_INVALID_ARG;
  const int64_t k_bytes = kind == 0 ? K * 2 : kind == 1 ? K : K / 2;
  g.num_kb = static_cast<int>((k_bytes + 127) / 128);
  if (kind == 2) {
    g.sf_blocks_a = static_cast<int>(g.tiles_m * g.v->cg);
    g.sf_blocks_b = static_cast<int>(g.tiles_n * (g.v->bn / 128));
    g.sf_bytes = nvfp4_scratch_bytes(g.sf_blocks_a, g.sf_blocks_b, g.num_kb);
    g.sf_b_off = static_cast<size_t>(g.sf_blocks_a) * g.num_kb * 2048;
  }
  *out = g;
  return TKG_OK;
}

tkg_status gemm_params(GemmParams* out, const GemmPlan& g, int kind, int64_t M, int64_t N, int64_t K, const void* A,
                       const void* B, void* C, const tkg_scales* scales, const uint8_t* sf_scratch, bool cached_maps) {
  DevState* d = nullptr;
  tkg_status st = current_device(&d);
  if (st != TKG_OK) return st;
  GemmParams& p = *out;
  std::memset(&p, 0, sizeof(p));
  const KernelVariant& v = *g.v;
  // Operand maps: rows of K elements, boxes of 128 bytes x (rows per CTA); rows of one B box: a
  // CTA's share of one MMA's N (512-wide tiles load two boxes per stage)
  const uint32_t b_rows = static_cast<uint32_t>((v.bn > 256 ? 256 : v.bn) / v.cg);
  if (kind == 0) {
    st = get_map(&p.tmap_a, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, K * 2, 64, 128, 128, cached_maps);
    if (st == TKG_OK)
      st = get_map(&p.tmap_b, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, K * 2, 64, b_rows, 128, cached_maps);
  } else {
    const int64_t row_bytes = kind == 1 ? K : K / 2;
    st = get_map(&p.tmap_a, A, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, M, row_bytes, 128, 128, 128, cached_maps);
    if (st == TKG_OK)
      st = get_map(&p.tmap_b, B, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, N, row_bytes, 128, b_rows, 128,
                   cached_maps);
  }
  if (st == TKG_OK && kind == 2) {
    // the staged scales: runs of 16 rows x 128 bytes, one box per (K stage, 128-row block) of A and
    // BN/128 boxes' worth for B
    p.sf_blocks_a = g.sf_blocks_a;
    p.sf_blocks_b = g.sf_blocks_b;
    st = get_map(&p.tmap_sfa, sf_scratch, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128,
                 static_cast<uint64_t>(g.sf_blocks_a) * g.num_kb * 16, 128, 128, 16, 0, cached_maps);
    if (st == TKG_OK)
      st = get_map(&p.tmap_sfb, sf_scratch + g.sf_b_off, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128,
                   static_cast<uint64_t>(g.sf_blocks_b) * g.num_kb * 16, 128, 128,
                   static_cast<uint32_t>(16 * (v.bn / 128)), 0, cached_maps);
  }
  p.c_via_tma = (N % 8 == 0) ? 1 : 0;
  if (st == TKG_OK && p.c_via_tma)
    st = get_map(&p.tmap_c, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, N * 2, static_cast<uint32_t>(v.epi_cols), 32,
                 static_cast<int>(select_swizzle(static_cast<uint32_t>(v.epi_cols) * 2)), cached_maps);
  if (st != TKG_OK) return st;
  p.c_ptr = C;
  if (kind != 0) {
    p.a_scale = scales->a_scale;
    p.b_scale = scales->b_scale;
  }
  p.status = d->status;
  p.timeout_ns = static_cast<unsigned long long>(opt_or(g_opt_timeout, kDefaultTimeoutNs));
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.tiles_m = static_cast<int>(g.tiles_m);
  p.tiles_n = static_cast<int>(g.tiles_n);
  p.num_kb = g.num_kb;
  p.group_m = static_cast<int>(opt_or(g_opt_group, kDefaultGroupM));
  p.split_s = 1;
  p.k_serpentine = opt_or(g_opt_k_order, TKG_K_ORDER_SERPENTINE) == TKG_K_ORDER_SERPENTINE ? 1 : 0;
  p.fault_mode = take_fault_mode(1);
  p.visits = g_visits.exchange(nullptr);
  const int64_t sched = opt_or(g_opt_schedule, TKG_SCHEDULE_STATIC);
  p.sched = sched == TKG_SCHEDULE_DYNAMIC ? kSchedDynamic : sched == TKG_SCHEDULE_SINGLE ? kSchedSingle : kSchedStatic;
  return TKG_OK;
}

tkg_status gemm_enqueue(int kind, const GemmPlan& g, GemmParams& p, void* stream, bool allow_split) {
  DevState* d = nullptr;
  tkg_status st = current_device(&d);
  if (st != TKG_OK) return st;
  const KernelVariant& v = *g.v;
  const int64_t cl = v.cg;  // CTAs per cluster
  const int64_t units = g.tiles_m * g.tiles_n;
  int clusters = 0;
  st = max_clusters(*d, kind, g.id, v, &clusters);
  if (st != TKG_OK) return st;
  int64_t grid_clusters = clusters;
  const int64_t cap = g_opt_max_ctas.load(std::memory_order_relaxed);
  if (cap > 0 && cap / cl < grid_clusters) grid_clusters = cap / cl > 0 ? cap / cl : 1;

  // split-K head (static schedule, tiles of one MMA per K step), planned for the clusters the grid
  // may use
  int64_t items = units;
  if (allow_split && p.sched == kSchedStatic && v.bn <= 256 && v.tile_m == 128 * v.cg &&
      opt_or(g_opt_split, TKG_SPLIT_ON) == TKG_SPLIT_ON) {
    int split_tiles = 0, split_s = 1;
    split_plan(units, grid_clusters, p.num_kb, &split_tiles, &split_s);
    DevState::SplitWs w;
    if (split_tiles > 0 && split_workspace(*d, static_cast<cudaStream_t>(stream), &w)) {
      p.split_tiles = split_tiles;
      p.split_s = split_s;
      p.split_ws = w.ws;
      p.split_cnt = w.cnt;
      items = units + static_cast<int64_t>(split_tiles) * (split_s - 1);
    }
  }
  if (items < grid_clusters) grid_clusters = items;
  // one cluster per tile: the hardware places them as SMs free up (and, in the
  // dynamic schedule, running clusters cancel and take over those not started)
  if (p.sched != kSchedStatic) grid_clusters = units;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid_clusters * cl), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(v.threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(v.smem_bytes);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: this grid's CTAs may start (and run their
  // set-up) before the previous kernel on the stream has finished; the kernel
  // waits for it before touching global memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap() ? 2 : 1;
  void* args[] = {&p};
  if (cudaLaunchKernelExC(&cfg, v.func, args) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}

bool launch_overlap() { return opt_or(g_opt_overlap, TKG_OVERLAP_ON) == TKG_OVERLAP_ON; }

}  // namespace tkg

namespace {

// Checks, the plan, the NVFP4 scale scratch (stream-ordered pool, freed after
// the GEMM in stream order) and its re-layout, the parameters, the launch.
tkg_status gemm_launch(int kind, int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                       const tkg_scales* scales, void* stream) {
  tkg_status st = check_gemm_args(kind, M, N, K, A, B, C, scales);
  if (st != TKG_OK) return st;
  DevState* d = nullptr;
  st = current_device(&d);
  if (st != TKG_OK) return st;
  GemmPlan g;
  st = plan_gemm(kind, M, N, K, d->sm_count, &g);
  if (st != TKG_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* scratch = nullptr;
  auto release = [&]() {
    if (scratch) cudaFreeAsync(scratch, cs);
  };
  if (kind == 2) {
    cudaMemPool_t pool = nullptr;
    st = device_pool(*d, &pool);
    if (st != TKG_OK) return st;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), g.sf_bytes, pool, cs) != cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    if (nvfp4_interleave_scales(scales->a_block_scale, scales->b_block_scale, static_cast<int>(M),
                                static_cast<int>(N), static_cast<int>(K), g.sf_blocks_a, g.sf_blocks_b, g.num_kb, scratch,
                                g.sf_b_off, cs, launch_overlap()) != cudaSuccess) {
      cudaGetLastError();
      release();
      return TKG_ERR_CUDA;
    }
  }
  GemmParams p;
  st = gemm_params(&p, g, kind, M, N, K, A, B, C, scales, scratch, true);
  if (st == TKG_OK) st = gemm_enqueue(kind, g, p, stream, true);
  release();
  return st;
}

}  // namespace

extern "C" {

tkg_status tkg_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                         const tkg_scales* scales, void* stream) {
  return gemm_launch(0, M, N, K, A, B, C, scales, stream);
}

tkg_status tkg_gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                        const tkg_scales* scales, void* stream) {
  return gemm_launch(1, M, N, K, A, B, C, scales, stream);
}

tkg_status tkg_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                          const tkg_scales* scales, void* stream) {
  return gemm_launch(2, M, N, K, A, B, C, scales, stream);
}

tkg_status tkg_check_status(void* stream) {
  DevState* d = nullptr;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  tkg_status st = current_device(&d);
  if (st != TKG_OK) return st;
  unsigned int word = 0;
  if (cudaMemcpy(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    // a GEMM that gave up may have left split-K piece counts behind: drop every split
    // workspace of the device (cudaFree waits for the device), the next use makes fresh ones
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& kv : d->split) {
      cudaFree(kv.second.ws);
      cudaFree(kv.second.cnt);
    }
    d->split.clear();
    cudaGetLastError();
  }
  return (word & kStatusTimeout) ? TKG_ERR_TIMEOUT : TKG_OK;
}

const char* tkg_status_string(tkg_status s) {
  switch (s) {
    case TKG_OK: return "ok";
    case TKG_ERR_INVALID_ARG: return "invalid argument";
    case TKG_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case TKG_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case TKG_ERR_CUDA: return "CUDA runtime or driver error";
    case TKG_ERR_TIMEOUT: return "device pipeline wait timed out";
    case TKG_ERR_INTERNAL: return "internal error";
  }
  return "unknown status";
}

void tkg_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_maps.clear();
  for (auto& d : g_dev) {
    cudaMemPool_t pool = d.pool;
    if (pool) cudaMemPoolTrimTo(pool, 0);  // hand cached scratch back; the pool itself is reused
    // split-K workspaces (cudaFree waits for work still using them); the status word is a
    // static device variable and stays
    for (auto& kv : d.split) {
      cudaFree(kv.second.ws);
      cudaFree(kv.second.cnt);
    }
    d = DevState{};
    d.pool = pool;
  }
  cudaGetLastError();  // a context already torn down at exit makes the frees fail; nothing to report
}

tkg_status tkg_set_option(tkg_option key, int64_t value) {
  if (value < 0) return TKG_ERR_INVALID_ARG;
  switch (key) {
    case TKG_OPT_TIMEOUT_NS: g_opt_timeout.store(value); return TKG_OK;
    case TKG_OPT_GROUP_M:
      if (value > 65536) return TKG_ERR_INVALID_ARG;
      g_opt_group.store(value);
      return TKG_OK;
    case TKG_OPT_VARIANT:
      if (value >= kNumVariants) return TKG_ERR_INVALID_ARG;
      g_opt_variant.store(value);
      return TKG_OK;
    case TKG_OPT_MAX_CTAS: g_opt_max_ctas.store(value); return TKG_OK;
    case TKG_OPT_LAUNCH_OVERLAP:
      if (value > TKG_OVERLAP_OFF) return TKG_ERR_INVALID_ARG;
      g_opt_overlap.store(value);
      return TKG_OK;
    case TKG_OPT_SCHEDULE:
      if (value > TKG_SCHEDULE_SINGLE) return TKG_ERR_INVALID_ARG;
      g_opt_schedule.store(value);
      return TKG_OK;
    case TKG_OPT_SPLIT_K:
      if (value > TKG_SPLIT_OFF) return TKG_ERR_INVALID_ARG;
      g_opt_split.store(value);
      return TKG_OK;
    case TKG_OPT_K_ORDER:
      if (value > TKG_K_ORDER_FORWARD) return TKG_ERR_INVALID_ARG;
      g_opt_k_order.store(value);
      return TKG_OK;
  }
  return TKG_ERR_INVALID_ARG;
}

int64_t tkg_get_option(tkg_option key) {
  switch (key) {
    case TKG_OPT_TIMEOUT_NS: return opt_or(g_opt_timeout, kDefaultTimeoutNs);
    case TKG_OPT_GROUP_M: return opt_or(g_opt_group, kDefaultGroupM);
    case TKG_OPT_VARIANT: return g_opt_variant.load();
    case TKG_OPT_MAX_CTAS: return g_opt_max_ctas.load();
    case TKG_OPT_LAUNCH_OVERLAP: return opt_or(g_opt_overlap, TKG_OVERLAP_ON);
    case TKG_OPT_SCHEDULE: return opt_or(g_opt_schedule, TKG_SCHEDULE_STATIC);
    case TKG_OPT_SPLIT_K: return opt_or(g_opt_split, TKG_SPLIT_ON);
    case TKG_OPT_K_ORDER: return opt_or(g_opt_k_order, TKG_K_ORDER_SERPENTINE);
  }
  return -1;
}

// ---------------------------------------------------------------- debug (host)

int tkg_debug_tile_coord(int t, int tiles_m, int tiles_n, int group_m, int* tm, int* tn) {
  if (tiles_m < 1 || tiles_n < 1 || group_m < 1 || t < 0 || !tm || !tn) return -1;
  if (static_cast<int64_t>(tiles_m) * tiles_n <= t) return -1;
  TileOrder{tiles_m, tiles_n, group_m}.coord(t, *tm, *tn);
  return 0;
}

uint32_t tkg_debug_swizzle_offset(uint32_t off, uint32_t s_bytes) { return swizzle_offset(off, s_bytes); }

uint32_t tkg_debug_select_swizzle(uint32_t row_bytes) { return select_swizzle(row_bytes); }

tkg_status tkg_debug_variant_info(int kind, int variant, int32_t info[7]) {
  const KernelVariant* v = variant_of(kind, variant);
  if (!v || !info) return TKG_ERR_INVALID_ARG;
  info[0] = v->cg;
  info[1] = v->bn;
  info[2] = v->stages;
  info[3] = v->epi_warps;
  info[4] = v->threads;
  info[5] = v->smem_bytes;
  info[6] = v->tile_m;
  return TKG_OK;
}

int tkg_debug_pick_variant(int kind, int64_t M, int64_t N, int64_t K, int sm_count) {
  if (sm_count <= 0) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
  }
  return pick_variant(kind, M, N, K, sm_count);
}

int tkg_debug_split_plan(int64_t tiles, int64_t clusters, int num_kb, int* split_tiles, int* split_s) {
  if (!split_tiles || !split_s || num_kb < 0) return -1;
  split_plan(tiles, clusters, num_kb, split_tiles, split_s);
  return 0;
}

int tkg_debug_work_item(int w, int split_tiles, int split_s, int num_kb, int out[4]) {
  if (!out || w < 0 || split_tiles < 0 || split_s < 1 || num_kb < 1) return -1;
  const WorkItem wk = work_item(w, split_tiles, split_s, num_kb);
  out[0] = wk.tile;
  out[1] = wk.kb0;
  out[2] = wk.kb1;
  out[3] = wk.piece;
  return 0;
}

tkg_status tkg_debug_set_visit_counter(unsigned int* counts) {
  g_visits.store(counts);
  return TKG_OK;
}

tkg_status tkg_debug_set_fault(int mode) {
  if (mode < 0 || mode > 2) return TKG_ERR_INVALID_ARG;
  g_fault.store(mode);
  return TKG_OK;
}

}  // extern "C"

// Used by the probe translation unit.
namespace tkg {
tkg_status debug_encode_map(CUtensorMap* out, const void* ptr, uint64_t d0, uint64_t d1, uint64_t pitch, uint32_t b0,
                            uint32_t b1, int swz) {
  return get_map(out, ptr, CU_TENSOR_MAP_DATA_TYPE_UINT8, d0, d1, pitch, b0, b1, swz);
}
tkg_status debug_device_ready() {
  DevState* d = nullptr;
  return current_device(&d);
}

tkg_status device_sm_count(int* out) {
  DevState* d = nullptr;
  const tkg_status st = current_device(&d);
  if (st == TKG_OK) *out = d->sm_count;
  return st;
}

int take_fault_mode(int mode) {
  int expected = mode;
  return g_fault.compare_exchange_strong(expected, 0) ? mode : 0;
}

tkg_status device_status_word(unsigned int** out) {
  DevState* d = nullptr;
  const tkg_status st = current_device(&d);
  if (st == TKG_OK) *out = d->status;
  return st;
}

tkg_status encode_tiled_map(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* ptr,
                            const uint64_t* dims, const uint64_t* strides, const uint32_t* box, int swz) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const tkg_status st = ensure_encode_locked();
    if (st != TKG_OK) return st;
  }
  CUtensorMapSwizzle sw = swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swz == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  std::memset(out, 0, sizeof(*out));
  const CUresult r = g_encode(out, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), d, st, b, e,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TKG_OK : TKG_ERR_INVALID_ARG;
}
}  // namespace tkg
