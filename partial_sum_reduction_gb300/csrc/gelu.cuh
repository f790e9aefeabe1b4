// GeLU of the column-parallel matmul's epilogue ("The simple maths behind
// parallel training", MLP block), shared by the tensor-core GEMM epilogue,
// the CUDA-core GEMM and the reduction kernels.
#pragma once

// 2^v on the MUFU unit (PTX ex2.approx, subnormal results flushed to zero).
__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// 1/d for d in [1, 2], on the FMA pipe.  The seed subtracts d's bit
// pattern from a constant: a float's bits, read as an integer, are a
// piecewise-linear log2 of its value, so the difference approximates
// log2(1/d) (Blinn, "Floating-point tricks", IEEE CG&A 17(4), 1997).
// 0x7EF311C2 minimises the seed's relative error over [1, 2] (5.1 %,
// exhaustive search).  One third-order step, y (1 + t + t^2) with
// t = 1 - d y, cubes the error (1.3e-4); one Newton-Raphson step,
// y (1 + t), squares it (1.7e-8).  Within 0.78 ulp of 1/d on all of
// [1, 2]; exact at d = 1 and d = 2.
__device__ __forceinline__ float recip_1_2(float d) {
    float y = __int_as_float(0x7EF311C2 - __float_as_int(d));
    float t = fmaf(-d, y, 1.0f);
    y = fmaf(y, fmaf(t, t, t), y);
    t = fmaf(-d, y, 1.0f);
    return fmaf(y, t, y);
}

// The tanh form (Hendrycks & Gimpel 2016): 0.5 x (1 + tanh u) with
// u = sqrt(2/pi) (x + 0.044715 x^3).  Through (1 + tanh u) / 2 = s(2u),
// s the logistic function, GeLU is x s(2u) with s(2u) = 1 / (1 + 2^z),
// z = -2 u log2(e).  The exponential is taken of -|z|, so the denominator
// stays in [1, 2] for every x and the reciprocal needs no range handling:
//   z <= 0:  s = 1 / (1 + 2^-|z|)
//   z >  0:  s = 2^-|z| / (1 + 2^-|z|)
// One MUFU op per element (the exponential), the rest on the FMA pipe: a
// hardware reciprocal as well would make the MUFU unit, at a quarter of
// the FMA rate, the bound of a GeLU epilogue.  Relative error about 1e-6
// where |GeLU| > 1e-3 (the fp32 rounding of u dominates), far below the
// bf16 rounding of stored activations.  x -> +inf gives x; finite
// x -> -inf gives -0.
__device__ __forceinline__ float gelu_tanh(float x) {
    const float k0 = -2.0f * 0.7978845608028654f * 1.4426950408889634f;  // -2 sqrt(2/pi) log2(e)
    const float k1 = k0 * 0.044715f;
    const float z = x * fmaf(x * x, k1, k0);
    const float e = ex2_approx(-fabsf(z));
    const float y = recip_1_2(1.0f + e);
    return x * (z > 0.0f ? e * y : y);
}
