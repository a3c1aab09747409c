// bf16 vectors widened to fp32 pairs, for the packed .f32x2 arithmetic of
// sm_100 and later (__fadd2_rn / __fmul2_rn / __ffma2_rn): two lanes per
// instruction, each rounded as its scalar counterpart.  f[q] holds elements
// 2q (x) and 2q + 1 (y) of an 8-element vector.
#pragma once

#include "common.cuh"

namespace nf {

__device__ __forceinline__ void unpack8x2(uint4 v, float2 (&f)[4]) {
    f[0] = make_float2(bf_lo(v.x), bf_hi(v.x));
    f[1] = make_float2(bf_lo(v.y), bf_hi(v.y));
    f[2] = make_float2(bf_lo(v.z), bf_hi(v.z));
    f[3] = make_float2(bf_lo(v.w), bf_hi(v.w));
}

__device__ __forceinline__ uint4 pack8x2(const float2 (&o)[4]) {
    return make_uint4(pack2(o[0].x, o[0].y), pack2(o[1].x, o[1].y), pack2(o[2].x, o[2].y),
                      pack2(o[3].x, o[3].y));
}

}  // namespace nf
