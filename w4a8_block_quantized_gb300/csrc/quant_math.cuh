// quant_math.cuh -- the activation quantizer shared by the pre-pass (prep.cu) and the
// few-token kernel (gemv.cu), so that both produce the same codes bit for bit.
//
// "MNN LLM inference on the SpacemiT K3", section 4 step 1 (dynamic per-row INT8):
// s = absmax / 127 (fp32 IEEE division), code = clamp(round_half_away(x / s), -127, 127).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w4a8 {

// INT8 code of one activation: clamp(round_half_away(x / s), -127, 127), fp32 IEEE division.
__device__ __forceinline__ int quant1(float x, float s) {
    float r = roundf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

// The same code, as a float, without a division in the common case.  With r = RN(1/s),
// t = RN(x * r) lies within |x/s| * (2^-23 + 2^-48) of x/s, and the IEEE quotient
// RN(x/s) within |x/s| * 2^-24; for |x/s| <= 127.5 the two differ by less than 2^-15.  So
// unless t is within 2^-15 of a half-integer, round_half_away(t) equals round_half_away of
// the IEEE quotient.  near_tie() flags the rest, which are recomputed with the division.
__device__ __forceinline__ bool near_tie(float t) {
    const float a = fabsf(t);
    return fabsf((a - truncf(a)) - 0.5f) <= 0x1p-15f;
}

// t rounded to the nearest integer (ties to even), and whether t lies within 2^-15 of a
// half-integer.  |t - rint(t)| is exact (the two are within a factor two of each other, or
// the integer is 0) and equals the distance of frac(|t|) from the nearer integer, so the
// flag is the near_tie() test.  Away from the flagged values round-to-even and
// round-half-away agree; the flagged ones are recomputed by the caller.
// The rounding is done on the fp32 add pipe: for |t| <= 2^22, (t + 1.5 * 2^23) - 1.5 * 2^23
// is t rounded to the nearest integer, ties to even (the sum's unit in the last place is 1
// and the add rounds to nearest even), i.e. exactly rintf(t); |t| <= 127.5 here.
__device__ __forceinline__ float rint_flag(float t, bool& tie) {
    const float q = __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f);
    tie |= fabsf(t - q) >= 0.5f - 0x1p-15f;
    return q;
}

// One code by the definition (IEEE division, round half away from zero, clamp to +-127), for the
// rare elements next to a rounding boundary and for rows whose scale has no finite reciprocal.
// Out of line and scalar: the division's code is then not repeated in every quantizing loop
// body.  (For a scale with a finite reciprocal the clamp never binds: see quant_lane.)
static __device__ __noinline__ float requant(float x, float s) {
    return fminf(fmaxf(roundf(__fdiv_rn(x, s)), -127.0f), 127.0f);
}

// Quantize one lane's V float4 of a row to float codes; s > 0 is the row's scale and
// r = RN(1/s).  No clamp is applied on the fast path: for finite inputs |x| <= absmax and
// s = RN(absmax/127), so while s keeps at least 22 significant bits (s >= 2^-128, which covers
// every s with a finite r) |x/s| <= 127 (1 + 2^-22) and no code can exceed 127 in magnitude,
// exactly as the clamped definition gives.  The rare near-tie elements of the warp are
// recomputed with the IEEE division (warp-uniform branch).  A scale below 2^-128 (absmax below
// about 127 * 2^-128) has no finite reciprocal, and deep in the subnormal range so few
// significant bits that |x/s| can pass 127; such a row (uniform across the warp) takes the
// recompute for every element: IEEE division, round half away, clamp.
// Two fp32 lanes per instruction (mul / add / sub .rn.f32x2): each element is rounded exactly
// as the scalar operation rounds it.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// rint_flag on two elements at once: t = x * r, q = (t + 1.5 * 2^23) - 1.5 * 2^23, and the
// near-tie flag from |t - q| (the same roundings, element by element, as rint_flag).
__device__ __forceinline__ void rint_flag2(float x0, float x1, uint64_t rr, float& q0, float& q1, bool& tie) {
    const uint64_t kc = pk2(12582912.0f, 12582912.0f);
    const uint64_t t = mul2(pk2(x0, x1), rr);
    const uint64_t q = sub2(add2(t, kc), kc);
    float d0, d1;
    upk2(sub2(t, q), d0, d1);
    upk2(q, q0, q1);
    tie |= fmaxf(fabsf(d0), fabsf(d1)) >= 0.5f - 0x1p-15f;
}

template <int V>
__device__ __forceinline__ void quant_lane(const float4 (&x)[V], float4 (&q)[V], float s, float r) {
    const bool tiny = !(r < __int_as_float(0x7f800000));
    bool tie = tiny;
    const uint64_t rr = pk2(r, r);
#pragma unroll
    for (int i = 0; i < V; ++i) {
        rint_flag2(x[i].x, x[i].y, rr, q[i].x, q[i].y, tie);
        rint_flag2(x[i].z, x[i].w, rr, q[i].z, q[i].w, tie);
    }
    if (__any_sync(0xffffffffu, tie)) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            if (tiny || near_tie(x[i].x * r)) q[i].x = requant(x[i].x, s);
            if (tiny || near_tie(x[i].y * r)) q[i].y = requant(x[i].y, s);
            if (tiny || near_tie(x[i].z * r)) q[i].z = requant(x[i].z, s);
            if (tiny || near_tie(x[i].w * r)) q[i].w = requant(x[i].w, s);
        }
    }
}

}  // namespace w4a8
