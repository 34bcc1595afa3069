// gemm_variants.h — registry of compiled kernel variants (host side).
#pragma once

#include "gemm_kernel.cuh"

namespace tkg {

// Variant ids (also the values of TKG_OPT_VARIANT).
enum VariantId : int {
  kVariantAuto = 0,
  kVariant1Sm128x256 = 1,  // cta_group::1, 128 x 256 tile per CTA
  kVariant2Sm256x256 = 2,  // cta_group::2, 256 x 256 tile per CTA pair
  kVariant2Sm256x128 = 3,  // cta_group::2, 256 x 128 tile per CTA pair
  kNumVariants = 4
};

// Each returns the variant for `id`, or nullptr if that kind has no such variant.
const KernelVariant* bf16_variant(int id);
const KernelVariant* fp8_variant(int id);
const KernelVariant* nvfp4_variant(int id);

}  // namespace tkg
