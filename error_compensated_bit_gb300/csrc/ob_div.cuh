// Division helper for the Adam updates of the warm-up and LoCo passes.
#pragma once

namespace ob {

// x / d, bit-identical to __fdiv_rn(x, d). IEEE division takes a slow path for a zero
// numerator, and zero numerators are common in these passes (never-touched elements,
// averages of quantized zeros); for d > 0 the quotient of a zero is that zero (its sign
// kept), so it is selected instead, and the division is given a nonzero numerator.
__device__ __forceinline__ float div_rn_zero_fast(float x, float d)
{
    const bool zero = (x == 0.0f) & (d > 0.0f);
    const float q = __fdiv_rn(zero ? 1.0f : x, d);
    return zero ? x : q;
}

}  // namespace ob
