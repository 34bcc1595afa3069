// gemm_nvfp4.cu — NVFP4 block-scaled GEMM (kind::mxf4nvf4, scale_vec::4X):
// packed e2m1 operands, one e4m3 scale per 16 consecutive K elements of each
// row, fp32 per-tensor scales applied in the epilogue (the block-scaled 4-bit
// GEMM of "ThunderKittens reaches 22.4 PFLOPS on NVIDIA Rubin", NVFP4 and
// tiling paragraphs).
//
// The tensor core reads the scales of one MMA (64 K elements = 4 scales per
// row) from tensor memory: row m of A's 128-row block at lane m, column
// (base + m/32); row n of B at lane n % 32 of every lane quarter, column
// (base + n/32); byte j = the j-th 16-element slice.  The caller's row-major
// [rows][K/16] scales are first rewritten by interleave_scales_kernel into
// 2 KB runs, one per (256-deep K stage, 128-row block), the runs of one K
// stage contiguous, so that every ring stage loads one contiguous run per 128
// rows with a plain 2-D TMA box.  A run is four 512-byte atoms, one per MMA of
// the stage, holding the 4 scales of rows r, r + 32, r + 64, r + 96 at byte
// 16 r (r < 32): one tcgen05.cp.32x128b.warpx4 puts row r's 16 bytes at lane
// r of every lane quarter, columns c .. c + 3, which is both layouts above
// (gemm_kernel.cuh issues the copies).
#include <cuda_bf16.h>

#include "gemm_variants.h"

#ifndef TKG_NVFP4_REG_SPLIT
#define TKG_NVFP4_REG_SPLIT true
#endif

namespace tkg {

// five 38 KB ring stages, one accumulator, eight epilogue warps (two per TMEM lane quarter, each
// draining half of the columns, one staging tile each), four scale warps whose leader lanes copy
// the scales into tensor memory
using Nvfp4_2Sm_256 = GemmCfg<Kind::NVFP4, 2, 256, 5, 8, 1, false, 1, TKG_NVFP4_REG_SPLIT>;

const KernelVariant* nvfp4_variant(int id) {
  static const KernelVariant v14 = make_variant<Nvfp4_2Sm_256>("nvfp4_2sm_256x256_s5_epi8_sfcp");
  switch (id) {
    case kVariant2Sm256x256SfCopy: return &v14;
    default: return nullptr;
  }
}

namespace {

struct InterleaveArgs {
  const uint8_t* src;  // row-major [rows][k16] e4m3 scales
  uint8_t* dst;        // runs [kstages][blocks][4 MMAs][512-byte atom]
  int rows;            // valid rows
  int k16;             // scales per row (K / 16)
  int blocks;          // 128-row blocks in dst (rows padded with zero scales)
  int kstages;         // 256-element K stages in dst (padded with zero scales)
};

// One CTA rewrites one 128-row block for two consecutive K stages: thread t loads the 16 scales of
// row t % 128 for stage kb0 + t / 128 (one 16-byte load from the row-major source; the two halves of
// the CTA read each source row's 32 bytes, one sector, together) into shared memory, then writes
// the 16 bytes of atom (t % 128) / 32 at row t % 32, so a warp writes 512 contiguous bytes.  Scales
// of rows or K positions past the matrix are written as 0; a stage that runs past the last K
// position, or a row pitch that is not a multiple of 16 bytes, takes byte loads.
__global__ void __launch_bounds__(256) interleave_scales_kernel(InterleaveArgs a, InterleaveArgs b, int blocks_a) {
  // launched as a programmatic dependent: the previous GEMM may still read the
  // scratch this kernel rewrites, or a previous kernel still write the scales
  griddep_wait();
  griddep_launch_dependents();
  const bool is_a = static_cast<int>(blockIdx.x) < blocks_a;
  const InterleaveArgs& s = is_a ? a : b;
  const int local = is_a ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - blocks_a;
  const int rb = local % s.blocks;
  const int r_in = static_cast<int>(threadIdx.x) & 127;
  const int half = static_cast<int>(threadIdx.x) >> 7;
  const int kb = 2 * (local / s.blocks) + half;
  const bool live = kb < s.kstages;
  const int row = rb * 128 + r_in;
  const int col = kb * 16;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (live && row < s.rows && col < s.k16) {
    const uint8_t* src = s.src + static_cast<size_t>(row) * s.k16 + col;
    if ((s.k16 & 15) == 0 && col + 16 <= s.k16) {
      v = __ldg(reinterpret_cast<const uint4*>(src));
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (col + j < s.k16) w[j >> 2] |= static_cast<uint32_t>(__ldg(src + j)) << (8 * (j & 3));
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  const size_t run = static_cast<size_t>(kb) * s.blocks + rb;
  // thread t then writes the 16 bytes of atom t / 32 (the stage's MMA) at row r = t % 32: that MMA's 4
  // scales of rows r, r + 32, r + 64, r + 96
  __shared__ uint4 rows16[2][128];
  rows16[half][r_in] = v;
  __syncthreads();
  const int t = r_in >> 5, r = r_in & 31;
  auto word = [&](int row_in) -> uint32_t {
    const uint4& u = rows16[half][row_in];
    return t == 0 ? u.x : t == 1 ? u.y : t == 2 ? u.z : u.w;
  };
  if (live)
    *reinterpret_cast<uint4*>(s.dst + (run * 4 + t) * 512 + static_cast<size_t>(r) * 16) =
        make_uint4(word(r), word(r + 32), word(r + 64), word(r + 96));
}

}  // namespace

// Rewrites both operands' scales into `scratch` (see the layout above), B's
// runs at byte offset `b_offset`.
cudaError_t nvfp4_interleave_scales(const uint8_t* sfa, const uint8_t* sfb, int M, int N, int K, int blocks_a,
                                    int blocks_b, int kstages, uint8_t* scratch, size_t b_offset,
                                    cudaStream_t stream, bool overlap) {
  InterleaveArgs a{sfa, scratch, M, K / 16, blocks_a, kstages};
  InterleaveArgs b{sfb, scratch + b_offset, N, K / 16, blocks_b, kstages};
  const int kpairs = (kstages + 1) / 2;
  const int grid_a = blocks_a * kpairs;
  const int grid_b = blocks_b * kpairs;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid_a + grid_b), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, interleave_scales_kernel, a, b, grid_a);
}

size_t nvfp4_scratch_bytes(int blocks_a, int blocks_b, int kstages) {
  return (static_cast<size_t>(blocks_a) + blocks_b) * kstages * 2048;
}

}  // namespace tkg
