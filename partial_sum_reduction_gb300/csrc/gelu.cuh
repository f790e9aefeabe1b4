// GeLU of the column-parallel matmul's epilogue ("The simple maths behind
// parallel training", MLP block), shared by the GEMM epilogue and the
// reduction kernels.
#pragma once

// The tanh form (Hendrycks & Gimpel 2016): 0.5 x (1 + tanh u) with
// u = sqrt(2/pi) (x + 0.044715 x^3), evaluated through the identity
// (1 + tanh u) / 2 = 1 / (1 + exp(-2u)), i.e. x / (1 + exp(-2u)), with the
// fast exponential and division intrinsics: a few instructions where a full
// tanhf took dozens, which made GeLU the slowest part of the epilogue.
// Relative error a few fp32 ulp (tested against tanhf), far below the bf16
// rounding of stored activations.  x -> +inf gives x; x -> -inf gives -0
// (exp overflows to inf).
__device__ __forceinline__ float gelu_tanh(float x) {
    const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);  // sqrt(2/pi) = 0.79788456...
    return __fdividef(x, 1.0f + __expf(-2.0f * u));
}
