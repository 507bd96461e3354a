// operand_codes.cuh -- the u4 weight code as the tensor cores' e4m3 operand, shared by the
// producers of that operand (the weight job of prep.cu and the converter warps of gemm.cu),
// so that both write the same bytes.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w4a8 {

// u4 pairs -> bytes in k order: nibbles k0..k7 of w become bytes of (o0: k0..k3, o1: k4..k7).
// A byte holding the code q is the e4m3 encoding of q * 2^-9 (the subnormal binade and the
// first normal binade share the step 2^-9), the GEMM's weight operand.
__device__ __forceinline__ void expand8(uint32_t w, uint32_t& o0, uint32_t& o1) {
    const uint32_t lo = w & 0x0F0F0F0Fu;         // k0 k2 k4 k6
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // k1 k3 k5 k7
    o0 = __byte_perm(lo, hi, 0x5140);
    o1 = __byte_perm(lo, hi, 0x7362);
}

// The weight side of the zero-point MMA for one row and block: the fp16 pair {-z_w, -z_w}
// (the sign bit flipped: exact), the low word of a 16-byte row whose other 12 bytes are 0.
__device__ __forceinline__ uint32_t neg_zero_pair(uint16_t z) {
    const uint32_t zb = static_cast<uint32_t>(z) ^ 0x8000u;
    return zb | (zb << 16);
}

}  // namespace w4a8
