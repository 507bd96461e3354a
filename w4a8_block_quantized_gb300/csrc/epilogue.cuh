// epilogue.cuh -- the store of one output, shared by the contraction kernels.
//
// "MNN LLM inference on the SpacemiT K3", section 4 step 3: the epilogue adds the bias and
// applies the optional clamp before writing the output directly; y is stored as fp32 or,
// for consumers that want it, bf16 (round to nearest even).
#pragma once

#include <cuda_bf16.h>

#include "w4a8_internal.h"

namespace w4a8 {

__device__ __forceinline__ void store_y(const OutSpec& o, int64_t idx, float v) {
    v = fminf(fmaxf(v, o.lo), o.hi);  // exact; the identity for the default bounds
    if (o.bf16)
        reinterpret_cast<__nv_bfloat16*>(o.y)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(o.y)[idx] = v;
}

}  // namespace w4a8
