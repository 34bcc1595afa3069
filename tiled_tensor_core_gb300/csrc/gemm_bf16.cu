// gemm_bf16.cu — bf16 instantiations of the persistent tcgen05 GEMM.
#include <cuda_bf16.h>

#include "gemm_variants.h"

namespace tkg {

using Bf16_2Sm_256 = GemmCfg<Kind::BF16, 2, 256, 6, 4>;
// 256x512: two N = 256 MMAs per K step sharing A through the collector buffer; eight epilogue warps
// given 192 registers by a warpgroup register split
using Bf16_2Sm_512 = GemmCfg<Kind::BF16, 2, 512, 4, 8, 1, true, 1, true>;

const KernelVariant* bf16_variant(int id) {
  static const KernelVariant v2 = make_variant<Bf16_2Sm_256>("bf16_2sm_256x256_s6");
  static const KernelVariant v15 = make_variant<Bf16_2Sm_512>("bf16_2sm_256x512_s4_epi8_regsplit");
  switch (id) {
    case kVariant2Sm256x256: return &v2;
    case kVariant2Sm256x512: return &v15;
    default: return nullptr;
  }
}

}  // namespace tkg
