// gemm_variants.h — registry of compiled kernel variants (host side).
#pragma once

#include "gemm_kernel.cuh"
#include "tkg.h"

namespace tkg {

// Variant ids (also the values of TKG_OPT_VARIANT).  The ids are those of the
// kernel forms measured while the tile shape was chosen; the forms that lost
// (1-SM 128 x 256, 256 x 128 / 192 / 224 pair tiles, A multicast between two
// pairs, a 512 x 256 pair tile whose two MMAs share B, NVFP4 scales read from
// global memory, copied by the MMA-issuing thread or written into tensor
// memory with tcgen05.st by scale warps) are no longer compiled.
enum VariantId : int {
  kVariantAuto = 0,
  kVariant2Sm256x256 = 2,         // cta_group::2, 256 x 256 tile per CTA pair (bf16 / FP8)
  kVariant2Sm256x256SfCopy = 14,  // cta_group::2, 256 x 256, block scales through shared memory, copied into
                                  // tensor memory (tcgen05.cp) by four issuing threads, eight epilogue warps
                                  // (NVFP4)
  kVariant2Sm256x512 = 15,        // cta_group::2, 256 x 512 tile per CTA pair: two N = 256 MMAs per K step, the
                                  // second taking A from the tensor core's collector buffer; eight epilogue
                                  // warps given 192 registers by a warpgroup register split (bf16 / FP8)
  kNumVariants = 16
};

// Each returns the variant for `id`, or nullptr if that kind has no such variant.
const KernelVariant* bf16_variant(int id);
const KernelVariant* fp8_variant(int id);
const KernelVariant* nvfp4_variant(int id);

// NVFP4: rewrite row-major [rows][K/16] block scales of A and B into the
// 2 KB per (K stage, 128-row block) runs that the GEMM stages (A's at scratch,
// B's at scratch + b_offset), four 512-byte per-MMA atoms inside a run (see
// gemm_nvfp4.cu).  One kernel launch on `stream`, as a programmatic dependent
// of the previous kernel if `overlap` (it waits for that kernel before
// touching memory either way).
cudaError_t nvfp4_interleave_scales(const uint8_t* sfa, const uint8_t* sfb, int M, int N, int K, int blocks_a,
                                    int blocks_b, int kstages, uint8_t* scratch, size_t b_offset,
                                    cudaStream_t stream, bool overlap);
size_t nvfp4_scratch_bytes(int blocks_a, int blocks_b, int kstages);

// ---------------------------------------------------------------- launch (api.cu)

// What a GEMM launch runs: the variant (TKG_OPT_VARIANT, else the default for
// the shape), its tile counts and K stages and, NVFP4, the staged block-scale
// geometry (2 KB runs per (K stage, 128-row block); B's after A's).
struct GemmPlan {
  int id = 0;
  const KernelVariant* v = nullptr;
  int64_t tiles_m = 0, tiles_n = 0;
  int num_kb = 0;
  int sf_blocks_a = 0, sf_blocks_b = 0;
  size_t sf_bytes = 0, sf_b_off = 0;
};
// Host-only argument checks of the GEMM entry points (no CUDA call).
tkg_status check_gemm_args(int kind, int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                           const tkg_scales* scales);
// Host only (no CUDA call); `sm_count` decides between the bf16 / FP8 tiles.
tkg_status plan_gemm(int kind, int64_t M, int64_t N, int64_t K, int sm_count, GemmPlan* out);
// The kernel parameters of a planned GEMM on the current device: tensor maps
// (through the host-side map cache if `cached_maps`, else encoded on the
// stack), sizes, options, and (NVFP4) the staged scales at `sf_scratch`.
tkg_status gemm_params(GemmParams* out, const GemmPlan& g, int kind, int64_t M, int64_t N, int64_t K, const void* A,
                       const void* B, void* C, const tkg_scales* scales, const uint8_t* sf_scratch, bool cached_maps);
// Launches the planned GEMM on `stream`: the persistent grid (or one cluster
// per tile) sized by the variant's co-resident clusters (cached per device),
// the split-K head if `allow_split` and the options ask for it (it needs a
// per-stream workspace the library allocates), programmatic dependent launch
// per TKG_OPT_LAUNCH_OVERLAP.
tkg_status gemm_enqueue(int kind, const GemmPlan& g, GemmParams& p, void* stream, bool allow_split);
// TKG_OPT_LAUNCH_OVERLAP is on.
bool launch_overlap();

// The current device's SM count, after the library's device check (api.cu).
tkg_status device_sm_count(int* out);
// Fault injection for the timeout tests: returns `mode` and disarms it if it is the
// armed mode (tkg_debug_set_fault), else 0.
int take_fault_mode(int mode);
// The current device's status word (device address), after the same check.
tkg_status device_status_word(unsigned int** out);
// A tiled TMA tensor map of `rank` dimensions (innermost first): element
// counts `dims`, byte strides of dimensions 1.. in `strides`, box `box`,
// swizzle 0/32/64/128 bytes; zero fill out of bounds.
tkg_status encode_tiled_map(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* ptr,
                            const uint64_t* dims, const uint64_t* strides, const uint32_t* box, int swz);

}  // namespace tkg
