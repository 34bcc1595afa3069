// gemm_bf16.cu — bf16 instantiations of the persistent tcgen05 GEMM.
#include <cuda_bf16.h>

#include "gemm_variants.h"

namespace tkg {

using Bf16_1Sm_256 = GemmCfg<Kind::BF16, 1, 256, 4, 4>;
using Bf16_2Sm_256 = GemmCfg<Kind::BF16, 2, 256, 6, 4>;
using Bf16_2Sm_128 = GemmCfg<Kind::BF16, 2, 128, 8, 4>;
using Bf16_2Sm_224 = GemmCfg<Kind::BF16, 2, 224, 6, 4>;
using Bf16_2Sm_192 = GemmCfg<Kind::BF16, 2, 192, 6, 4>;
using Bf16_Mc_256 = GemmCfg<Kind::BF16, 2, 256, 6, 4, 2, kSfCopy, 1, false, false, 2>;
using Bf16_Mc_224 = GemmCfg<Kind::BF16, 2, 224, 6, 4, 2, kSfCopy, 1, false, false, 2>;
using Bf16_Mc_192 = GemmCfg<Kind::BF16, 2, 192, 6, 4, 2, kSfCopy, 1, false, false, 2>;
using Bf16_2Sm_512 = GemmCfg<Kind::BF16, 2, 512, 4, 4, 1>;

const KernelVariant* bf16_variant(int id) {
  static const KernelVariant v1 = make_variant<Bf16_1Sm_256>("bf16_1sm_128x256_s4");
  static const KernelVariant v2 = make_variant<Bf16_2Sm_256>("bf16_2sm_256x256_s6");
  static const KernelVariant v3 = make_variant<Bf16_2Sm_128>("bf16_2sm_256x128_s8");
  static const KernelVariant v4 = make_variant<Bf16_2Sm_224>("bf16_2sm_256x224_s6");
  static const KernelVariant v9 = make_variant<Bf16_2Sm_192>("bf16_2sm_256x192_s6");
  static const KernelVariant v10 = make_variant<Bf16_Mc_256>("bf16_2x2sm_256x256_mca_s6");
  static const KernelVariant v11 = make_variant<Bf16_Mc_224>("bf16_2x2sm_256x224_mca_s6");
  static const KernelVariant v12 = make_variant<Bf16_Mc_192>("bf16_2x2sm_256x192_mca_s6");
  static const KernelVariant v13 = make_variant<Bf16_2Sm_512>("bf16_2sm_256x512_s4");
  switch (id) {
    case kVariant1Sm128x256: return &v1;
    case kVariant2Sm256x256: return &v2;
    case kVariant2Sm256x128: return &v3;
    case kVariant2Sm256x224: return &v4;
    case kVariant2Sm256x192: return &v9;
    case kVariantMc256x256: return &v10;
    case kVariantMc256x224: return &v11;
    case kVariantMc256x192: return &v12;
    case kVariant2Sm256x512: return &v13;
    default: return nullptr;
  }
}

}  // namespace tkg
