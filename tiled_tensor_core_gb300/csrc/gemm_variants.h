// gemm_variants.h — registry of compiled kernel variants (host side).
#pragma once

#include "gemm_kernel.cuh"
#include "tkg.h"

namespace tkg {

// Variant ids (also the values of TKG_OPT_VARIANT).
enum VariantId : int {
  kVariantAuto = 0,
  kVariant1Sm128x256 = 1,  // cta_group::1, 128 x 256 tile per CTA
  kVariant2Sm256x256 = 2,  // cta_group::2, 256 x 256 tile per CTA pair
  kVariant2Sm256x128 = 3,  // cta_group::2, 256 x 128 tile per CTA pair
  kVariant2Sm256x224 = 4,  // cta_group::2, 256 x 224 tile per CTA pair (bf16 / FP8)
  kVariant2Sm256x256Sfw = 5,  // cta_group::2, 256 x 256, block scales written by scale warps (NVFP4)
  kVariant2Sm256x256Hybrid = 6,  // cta_group::2, 256 x 256, A scales by scale warps, B by a copy warp (NVFP4)
  kVariant2Sm256x256Coupled = 7,  // as 5, with one TMEM scale slot per ring stage (NVFP4)
  kVariant2Sm256x256SfSmem = 8,   // as 7, the scales brought into shared memory by the ring's TMA (NVFP4)
  kVariant2Sm256x192 = 9,          // cta_group::2, 256 x 192 tile per CTA pair (bf16 / FP8)
  // clusters of two CTA pairs on horizontally adjacent tiles, A multicast between the pairs (bf16 / FP8)
  kVariantMc256x256 = 10,
  kVariantMc256x224 = 11,
  kVariantMc256x192 = 12,
  kVariant2Sm256x512 = 13,  // cta_group::2, 256 x 512 tile per CTA pair: two N = 256 MMAs per K step (bf16 / FP8)
  kNumVariants = 14
};

// Each returns the variant for `id`, or nullptr if that kind has no such variant.
const KernelVariant* bf16_variant(int id);
const KernelVariant* fp8_variant(int id);
const KernelVariant* nvfp4_variant(int id);

// NVFP4: rewrite row-major [rows][K/16] block scales of A and B into the
// 2 KB per (K stage, 128-row block) runs the GEMM stages (A's at scratch, B's
// at scratch + b_offset), laid out for the variant's `sf_mode`.  One kernel
// launch on `stream`, as a programmatic dependent of the previous kernel if
// `overlap` (it waits for that kernel before touching memory either way).
cudaError_t nvfp4_interleave_scales(const uint8_t* sfa, const uint8_t* sfb, int M, int N, int K, int blocks_a,
                                    int blocks_b, int kstages, int sf_mode, uint8_t* scratch, size_t b_offset,
                                    cudaStream_t stream, bool overlap);
size_t nvfp4_scratch_bytes(int blocks_a, int blocks_b, int kstages);

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
