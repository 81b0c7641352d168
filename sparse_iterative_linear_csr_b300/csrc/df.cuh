// df.cuh -- double-float arithmetic (an unevaluated pair hi + lo of fp32
// values, |lo| <= ulp(hi)/2) for the fp32-storage path.
//
// On B300 the fp64 pipe issues at 1/64 of the fp32 rate, and conversions
// between fp32 and fp64 also occupy it, so the fp32-storage kernels do all
// element-wise arithmetic here, on the fp32 pipe.  Products of two fp32
// values are exact (FMA-based two-product); sums use Knuth's two-sum and
// Dekker's fast-two-sum (error-free transformations; see Ogita, Rump and
// Oishi, "Accurate sum and dot product", SIAM J. Sci. Comput. 2005).  The
// pair carries about 48 significant bits, far more than the fp32 values it
// rounds back to.
#pragma once

#include <cuda_runtime.h>

namespace sla {

struct DF {
    float hi, lo;
};

__device__ __forceinline__ DF df_make(float a) { return DF{a, 0.0f}; }

// s + e = a + b exactly (any magnitudes)
__device__ __forceinline__ DF two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return DF{s, e};
}

// s + e = a + b exactly when |a| >= |b| (or a == 0)
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return DF{s, __fsub_rn(b, __fsub_rn(s, a))};
}

// p + e = a * b exactly (barring underflow)
__device__ __forceinline__ DF two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return DF{p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ DF df_add(DF x, DF y) {
    DF s = two_sum(x.hi, y.hi);
    const DF t = two_sum(x.lo, y.lo);
    s.lo = __fadd_rn(s.lo, t.hi);
    s = fast_two_sum(s.hi, s.lo);
    s.lo = __fadd_rn(s.lo, t.lo);
    return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ DF df_add_f(DF x, float b) {
    DF s = two_sum(x.hi, b);
    s.lo = __fadd_rn(s.lo, x.lo);
    return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ DF df_neg(DF x) { return DF{-x.hi, -x.lo}; }

// (x.hi + x.lo) * b
__device__ __forceinline__ DF df_mul_f(DF x, float b) {
    DF p = two_prod(x.hi, b);
    p.lo = __fmaf_rn(x.lo, b, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

// (a.hi + a.lo) * (b.hi + b.lo)
__device__ __forceinline__ DF df_mul(DF a, DF b) {
    DF p = two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, p.lo);
    p.lo = __fmaf_rn(a.lo, b.hi, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

// x * x
__device__ __forceinline__ DF df_sqr(DF x) {
    DF p = two_prod(x.hi, x.hi);
    p.lo = __fmaf_rn(__fmul_rn(2.0f, x.hi), x.lo, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

// acc += a * b for fp32 a, b (exact product)
__device__ __forceinline__ DF df_fma_ff(float a, float b, DF acc) { return df_add(acc, two_prod(a, b)); }

// acc += (g.hi + g.lo) * b
__device__ __forceinline__ DF df_fma_df(DF g, float b, DF acc) {
    DF p = two_prod(g.hi, b);
    p.lo = __fmaf_rn(g.lo, b, p.lo);
    return df_add(acc, p);
}

// Nearest fp32 to hi + lo.
__device__ __forceinline__ float df_round(DF x) { return __fadd_rn(x.hi, x.lo); }

// fp64 <-> double-float (set-up and per-thread totals only: these use the
// fp64 pipe).
__device__ __forceinline__ DF df_from_double(double v) {
    const float hi = __double2float_rn(v);
    return DF{hi, __double2float_rn(v - (double)hi)};
}
__device__ __forceinline__ double df_to_double(DF x) { return (double)x.hi + (double)x.lo; }

}  // namespace sla
