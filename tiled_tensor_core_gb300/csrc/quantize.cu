// quantize.cu — on-device FP8 and NVFP4 encoders: the step before the GEMM
// that turns fp32 data into the operands tkg_gemm_fp8 / tkg_gemm_nvfp4 take
// (the 8-bit and block-scaled 4-bit formats of "ThunderKittens reaches 22.4
// PFLOPS on NVIDIA Rubin", NVFP4 and FP8 paragraphs).
//
// Both encoders need the tensor's absolute maximum before any element can be
// encoded, so each is two passes over x (HBM-bound; x is far larger than L2 at
// the sizes that matter):
//   1. amax_kernel: max |x| into a 32-bit word (the caller's scale output,
//      zeroed first).  Non-negative floats order like their bit patterns, so
//      the reduction is an integer max (warp reduce, then one atomicMax per CTA).
//   2. encode kernel: every thread derives the tensor scale from that word and
//      encodes 16 consecutive elements per step, walking the tensor from its
//      end, so that it first re-reads what the amax pass read last and L2
//      still holds (up to the L2 size of the second read comes from L2, not
//      HBM); the fp32 arithmetic is the
//      one the format reading fixes (one IEEE rounding per multiply or divide,
//      written with __fmul_rn / __fdiv_rn so that nothing is contracted) and
//      the rounding to e4m3 / e2m1 is the hardware's cvt.rn.satfinite.
//   3. finish_kernel (one thread): the word becomes the scale the GEMM takes.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_variants.h"
#include "tkg.h"

namespace tkg {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float max4(float m, const float4& v) {
  return fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
}

// Two fp32 -> e4m3 codes, round to nearest even, saturating at +-448:
// `lo` in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight fp32 -> eight e2m1 codes packed in 32 bits, element i in bits 4i..4i+3
// (element 2j in the low nibble of byte j).
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Exact value of an e4m3 code (sign | exponent, bias 7 | 3-bit mantissa; no NaN codes reach here).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0x1p-9f;
  return (c & 0x80u) ? -mag : mag;
}

__global__ void __launch_bounds__(kThreads) amax_kernel(const float4* __restrict__ x, int64_t n4,
                                                        unsigned int* __restrict__ amax_bits) {
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    const float4 a = ld_stream(x + i), b = ld_stream(x + i + stride), c = ld_stream(x + i + 2 * stride),
                 d = ld_stream(x + i + 3 * stride);
    m = max4(max4(max4(max4(m, a), b), c), d);
  }
  for (; i < n4; i += stride) m = max4(m, ld_stream(x + i));
  unsigned int bits = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  __shared__ unsigned int warp_max[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = bits;
  __syncthreads();
  if (threadIdx.x < 32) {
    bits = threadIdx.x < kThreads / 32 ? warp_max[threadIdx.x] : 0u;
    bits = __reduce_max_sync(0xffffffffu, bits);
    if (threadIdx.x == 0) atomicMax(amax_bits, bits);
  }
}

// FP8: s = 448 / amax (1 if amax == 0); q = e4m3(x * s).  16 elements per thread step.
__global__ void __launch_bounds__(kThreads) fp8_encode_kernel(const float4* __restrict__ x, uint4* __restrict__ q,
                                                              int64_t n16, const unsigned int* __restrict__ amax_bits) {
  const float amax = __uint_as_float(*amax_bits);
  const float s = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < n16; t += stride) {
    const int64_t i = n16 - 1 - t;
    const float4 a = ld_stream(x + 4 * i), b = ld_stream(x + 4 * i + 1), c = ld_stream(x + 4 * i + 2),
                 d = ld_stream(x + 4 * i + 3);
    uint4 o;
    o.x = e4m3x2(__fmul_rn(a.x, s), __fmul_rn(a.y, s)) | (e4m3x2(__fmul_rn(a.z, s), __fmul_rn(a.w, s)) << 16);
    o.y = e4m3x2(__fmul_rn(b.x, s), __fmul_rn(b.y, s)) | (e4m3x2(__fmul_rn(b.z, s), __fmul_rn(b.w, s)) << 16);
    o.z = e4m3x2(__fmul_rn(c.x, s), __fmul_rn(c.y, s)) | (e4m3x2(__fmul_rn(c.z, s), __fmul_rn(c.w, s)) << 16);
    o.w = e4m3x2(__fmul_rn(d.x, s), __fmul_rn(d.y, s)) | (e4m3x2(__fmul_rn(d.z, s), __fmul_rn(d.w, s)) << 16);
    q[i] = o;
  }
}

// NVFP4: g = amax / 2688 (1 if amax == 0); per block of 16: sb = e4m3(b / (6 g)),
// d = dec(sb) * g, q = e2m1(x / d) (0 when d == 0).  One block per thread step;
// blocks are consecutive along rows, so consecutive threads read consecutive 64 B.
__global__ void __launch_bounds__(kThreads) nvfp4_encode_kernel(const float4* __restrict__ x, uint2* __restrict__ q,
                                                                uint8_t* __restrict__ sf, int64_t nblocks,
                                                                const unsigned int* __restrict__ amax_bits) {
  const float amax = __uint_as_float(*amax_bits);
  const float g = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  const float six_g = __fmul_rn(6.0f, g);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < nblocks; t += stride) {
    const int64_t i = nblocks - 1 - t;
    float v[16];
    {
      const float4 a = ld_stream(x + 4 * i), b = ld_stream(x + 4 * i + 1), c = ld_stream(x + 4 * i + 2),
                   d = ld_stream(x + 4 * i + 3);
      v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
      v[8] = c.x, v[9] = c.y, v[10] = c.z, v[11] = c.w, v[12] = d.x, v[13] = d.y, v[14] = d.z, v[15] = d.w;
    }
    float bmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(v[j]));
    const uint32_t sb = e4m3x2(__fdiv_rn(bmax, six_g), 0.0f) & 0xFFu;
    const float dq = __fmul_rn(e4m3_value(sb), g);
    uint2 o = make_uint2(0u, 0u);
    if (dq != 0.0f) {
      float h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = __fdiv_rn(v[j], dq);
      o.x = e2m1x8(h);
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = __fdiv_rn(v[8 + j], dq);
      o.y = e2m1x8(h);
    }
    q[i] = o;
    sf[i] = static_cast<uint8_t>(sb);
  }
}

// mode 0: FP8 dequantisation scale amax / 448; mode 1: NVFP4 global scale amax / 2688 (1 if amax == 0).
__global__ void finish_kernel(unsigned int* word, int mode) {
  const float amax = __uint_as_float(*word);
  const float out = amax > 0.0f ? __fdiv_rn(amax, mode == 0 ? 448.0f : 2688.0f) : 1.0f;
  *word = __float_as_uint(out);
}

tkg_status encode(int mode, int64_t rows, int64_t cols, const float* x, void* q, uint8_t* sf, float* scale,
                  void* stream) {
  if (rows <= 0 || cols <= 0 || cols % 16 != 0 || !x || !q || !scale || (mode == 1 && !sf))
    return TKG_ERR_INVALID_ARG;
  if (rows > (int64_t(1) << 40) / cols) return TKG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return TKG_ERR_MISALIGNED;
  int sms = 0;
  const tkg_status st = device_sm_count(&sms);
  if (st != TKG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t n = rows * cols;
  unsigned int* word = reinterpret_cast<unsigned int*>(scale);
  const int grid = sms * kCtasPerSm;
  if (cudaMemsetAsync(word, 0, sizeof(unsigned int), s) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  amax_kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(x), n / 4, word);
  if (mode == 0)
    fp8_encode_kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(x), static_cast<uint4*>(q), n / 16,
                                                word);
  else
    nvfp4_encode_kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(x), static_cast<uint2*>(q), sf,
                                                  n / 16, word);
  finish_kernel<<<1, 1, 0, s>>>(word, mode);
  if (cudaGetLastError() != cudaSuccess) return TKG_ERR_CUDA;
  return TKG_OK;
}

}  // namespace
}  // namespace tkg

extern "C" {

tkg_status tkg_quantize_fp8(int64_t rows, int64_t cols, const float* x, uint8_t* q, float* dequant_scale,
                            void* stream) {
  return tkg::encode(0, rows, cols, x, q, nullptr, dequant_scale, stream);
}

tkg_status tkg_quantize_nvfp4(int64_t rows, int64_t cols, const float* x, uint8_t* q_packed, uint8_t* block_scales,
                              float* global_scale, void* stream) {
  return tkg::encode(1, rows, cols, x, q_packed, block_scales, global_scale, stream);
}

}  // extern "C"
