// gemm_nvfp4.cu — NVFP4 block-scaled GEMM variants (kind::mxf4nvf4).
#include <cuda_bf16.h>

#include "gemm_variants.h"

namespace tkg {

const KernelVariant* nvfp4_variant(int id) {
  (void)id;
  return nullptr;
}

}  // namespace tkg
