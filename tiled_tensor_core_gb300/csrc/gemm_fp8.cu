// gemm_fp8.cu — FP8 (e4m3 x e4m3, kind::f8f6f4) instantiations of the
// persistent tcgen05 GEMM.  Same byte geometry as bf16: a stage row is 128
// bytes = 128 K elements; each MMA consumes 32 of them.
#include <cuda_bf16.h>

#include "gemm_variants.h"

namespace tkg {

using Fp8_2Sm_256 = GemmCfg<Kind::FP8, 2, 256, 6, 4>;
// 256x512: two N = 256 MMAs per K step sharing A through the collector buffer; eight epilogue warps
// given 192 registers by a warpgroup register split
using Fp8_2Sm_512 = GemmCfg<Kind::FP8, 2, 512, 4, 8, 1, true, 1, true>;

const KernelVariant* fp8_variant(int id) {
  static const KernelVariant v2 = make_variant<Fp8_2Sm_256>("fp8_2sm_256x256_s6");
  static const KernelVariant v15 = make_variant<Fp8_2Sm_512>("fp8_2sm_256x512_s4_epi8_regsplit");
  switch (id) {
    case kVariant2Sm256x256: return &v2;
    case kVariant2Sm256x512: return &v15;
    default: return nullptr;
  }
}

}  // namespace tkg
