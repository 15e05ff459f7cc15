// The library's one definition of a probability from a logit, the softmax at
// temperature 1 (the plain reading of a language model's output: the
// InvisibleLoRA abstract has both passes end in a distribution over the
// vocabulary).  The softmax, the draft draw and the accept step on logits all
// compute it with these functions, so their values agree bit for bit:
//
//   p(v) = exp_of(z(v) - m) * R,    m = max_w z(w),
//   R = 1 / S rounded once per row,  S = the row's sum of exp_of(z(w) - m),
//
// in fp32, with exp_of(d) = 2^(d log2 e) from the identity e^d = 2^(d log2 e):
// d log2 e rounded once, then 2^y by the ex2.approx instruction of the PTX
// ISA.  A row's statistics are stored as the pair (m, R).
#pragma once

#include <cuda_runtime.h>

namespace mlora {

constexpr float LOG2_E = 1.44269504088896340736f;

// 2^y by the hardware's approximation (+0 for y = -inf, NaN for NaN).
__device__ __forceinline__ float exp2_hw(float y) {
  float r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// e^d.
__device__ __forceinline__ float exp_of(float d) { return exp2_hw(d * LOG2_E); }

// The probability of an entry from its logit z and its row's pair (m, R).
__device__ __forceinline__ float prob_from_logit(float z, float2 st) { return exp_of(z - st.x) * st.y; }

}  // namespace mlora
