// FP8 base weights for the LoRA-off draft pass.  The "LoRA Inference"
// glossary lists quantizing the base model's weights to 8 bits among the
// serving optimisations that go with LoRA; the draft pass of InvisibleLoRA
// runs the base model alone, so an E4M3 copy of W halves the bytes of that
// HBM-bound pass while the LoRA-on verify pass keeps bf16 and the accept step
// keeps the output distribution exact.
//
// Quantization is per row with one fp32 scale: scale = amax / 448 (IEEE
// division) and code = E4M3(v / scale) by cvt.rn.satfinite (nearest, ties to
// even, saturating at 448).  W is quantized once per output row; the draft
// call quantizes its activations per token row into the workspace, then the
// stream-K GEMM multiplies the codes with kind::f8f6f4 MMAs and scales in its
// epilogue (gemm_sk.cu).
#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int Q_THREADS = 256;
constexpr float E4M3_MAX = 448.0f;

// Two fp32 values to two E4M3 codes, `lo` in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int w = 0; w < Q_THREADS / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();  // red is reused by the next row
  return m;
}

// One CTA per row (grid-stride): the row's absolute maximum, then its codes,
// 8 values (one 16-byte load, one 8-byte store) per thread and step.  K % 8
// == 0 and 16-byte aligned rows (checked on the host).
__global__ void __launch_bounds__(Q_THREADS)
    quantize_rows_e4m3_kernel(const uint16_t *__restrict__ src, int R, int K, uint8_t *__restrict__ q,
                              float *__restrict__ scale) {
  __shared__ float red[Q_THREADS / 32];
  grid_launch_dependents();
  grid_dependency_wait();  // the rows come from the kernel just before
  const int n8 = K / 8;
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const uint4 *row = reinterpret_cast<const uint4 *>(src + (size_t)r * K);
    float amax = 0.f;
    for (int c = threadIdx.x; c < n8; c += Q_THREADS) {
      const uint4 v = __ldg(row + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
    amax = block_max(amax, red);
    const bool zero = !(amax > 0.f);
    const float s = zero ? 1.f : __fdiv_rn(amax, E4M3_MAX);
    if (threadIdx.x == 0) scale[r] = s;
    uint2 *out = reinterpret_cast<uint2 *>(q + (size_t)r * K);
    for (int c = threadIdx.x; c < n8; c += Q_THREADS) {
      uint2 o = make_uint2(0u, 0u);  // a zero row stores +0 codes
      if (!zero) {
        const uint4 v = __ldg(row + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          p[i] = cvt_e4m3x2(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                            __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), s));
        o = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
      }
      out[c] = o;
    }
  }
}

cudaError_t launch_quantize_rows_e4m3(const uint16_t *src, int R, int K, uint8_t *q, float *scale, int num_sms,
                                      cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const int grid = R < num_sms * 8 ? R : num_sms * 8;
  return launch_pdl(quantize_rows_e4m3_kernel, dim3((unsigned)grid), dim3(Q_THREADS), 0, s, src, R, K, q, scale);
}

}  // namespace mlora
