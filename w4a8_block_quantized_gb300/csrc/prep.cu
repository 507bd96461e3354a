// prep.cu -- activation pre-pass (K1) and operand packing.
//
// "MNN LLM inference on the SpacemiT K3", section 4 step 1: one pass over the fp32
// activations produces absmax -> scale -> INT8 codes -> packed A + the per-block row
// sum ("srcKernelSum"), instead of an absmax scan, a second quantize/pack read and a
// separate sum.  Here one warp (or a few warps, for long rows) holds a row in
// registers after a single 128-bit streaming read, reduces absmax with warp shuffles,
// divides by absmax/127 with an IEEE fp32 division, rounds half away from zero,
// reduces the 64-element block sums with shuffles, and writes either
//   - the API layout: int8 a_q [M][K], fp32 s_a [M], int32 rowsum [M][K/64], or
//   - the tensor-core layout of the fused call: per row and 64-block the two e4m3
//     nibble planes of section 3 eq. (3) (16*(a>>4) and a&15), s_a, and the row sums
//     as the operand of the zero-point MMA.
// The same launch also prepares the weight side in its extra CTAs (the u4 codes expanded
// to the GEMM's e4m3 operand, the fp16 scales and zeros laid out for the epilogue and the
// zero-point MMA), so a call costs two launches in total.
#include "operand_codes.cuh"
#include "quant_math.cuh"
#include "sm103_ptx.cuh"
#include "w4a8_internal.h"

#include <atomic>
#include <cuda_fp16.h>

namespace w4a8 {
namespace {

// Two e4m3 codes in one 16-bit word, v0 in the low byte.  The inputs are small exact
// integers (|v| <= 128 with at most 4 significant bits), so the conversion is exact.
__device__ __forceinline__ uint32_t e4m3x2(float v0, float v1) {
    unsigned short d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(v1), "f"(v0));
    return d;
}

// Section 3 eq. (3) planes of four codes: hi word holds e4m3(16*(a>>4)) (signed high
// nibble, arithmetic shift), lo word holds e4m3(a & 15), element j in byte j.
__device__ __forceinline__ void planes4(int a0, int a1, int a2, int a3, uint32_t& hi, uint32_t& lo) {
    hi = e4m3x2(static_cast<float>(16 * (a0 >> 4)), static_cast<float>(16 * (a1 >> 4))) |
         (e4m3x2(static_cast<float>(16 * (a2 >> 4)), static_cast<float>(16 * (a3 >> 4))) << 16);
    lo = e4m3x2(static_cast<float>(a0 & 15), static_cast<float>(a1 & 15)) |
         (e4m3x2(static_cast<float>(a2 & 15), static_cast<float>(a3 & 15)) << 16);
}

// Zero-point operand of one token and block: rs = 64*rh + rl as the exact fp16 pair
// {rh / 8, rl / 512} (see the rx layout in w4a8_internal.h), then 12 zero bytes.
__device__ __forceinline__ uint4 rx_entry(int rs) {
    const int rh = rs >> 6, rl = rs & 63;
    const __half2 p = __floats2half2_rn(static_cast<float>(rh) * 0.125f, static_cast<float>(rl) * (1.0f / 512.0f));
    return make_uint4(*reinterpret_cast<const uint32_t*>(&p), 0u, 0u, 0u);
}

// Token record of row m, block b, for records of 2^ts tokens (the layout in w4a8_internal.h).
__device__ __forceinline__ uint8_t* token_rec(uint8_t* trec, int64_t m, int64_t b, int64_t nb, int ts) {
    return trec + ((m >> ts) * nb + b) * (static_cast<int64_t>(144) << ts);
}

// Byte offset, inside a token record, of the 4 codes k = 4j .. 4j+3 of the block (j < 16) of
// row r in plane p (0 = high nibbles, 1 = low nibbles): 128-byte swizzle of 16-byte chunks.
__device__ __forceinline__ int plane_off(int r, int j, int p) {
    const int c = (j >> 2) + 4 * p;
    return r * 128 + ((c ^ (r & 7)) << 4) + ((j & 3) << 2);
}

// Section 3 eq. (3) planes of four float codes (exact integers in [-127, 127]): hi word holds
// e4m3(16 * floor(q / 16)) (the signed high nibble times 16), lo word e4m3(q - that) (the
// unsigned low nibble), element j in byte j.  Two elements per mul / sub .rn.f32x2; every
// product and difference here is exact (q is an integer in [-127, 127]).
__device__ __forceinline__ void planes4f(float4 q, uint32_t& hi, uint32_t& lo) {
    const uint64_t k16 = pk2(0.0625f, 0.0625f), k1 = pk2(16.0f, 16.0f);
    float a0, a1, a2, a3;
    upk2(mul2(pk2(q.x, q.y), k16), a0, a1);
    upk2(mul2(pk2(q.z, q.w), k16), a2, a3);
    const uint64_t h01 = mul2(pk2(floorf(a0), floorf(a1)), k1), h23 = mul2(pk2(floorf(a2), floorf(a3)), k1);
    float h0, h1, h2, h3, l0, l1, l2, l3;
    upk2(h01, h0, h1);
    upk2(h23, h2, h3);
    upk2(sub2(pk2(q.x, q.y), h01), l0, l1);
    upk2(sub2(pk2(q.z, q.w), h23), l2, l3);
    hi = e4m3x2(h0, h1) | (e4m3x2(h2, h3) << 16);
    lo = e4m3x2(l0, l1) | (e4m3x2(l2, l3) << 16);
}

// Four float codes as int8 bytes: adding 1.5 * 2^23 puts the integer, in two's complement,
// in the low mantissa bits, whose low byte is the code.
__device__ __forceinline__ uint32_t bytes4f(float4 q) {
    const uint32_t b0 = __float_as_uint(q.x + 12582912.0f), b1 = __float_as_uint(q.y + 12582912.0f);
    const uint32_t b2 = __float_as_uint(q.z + 12582912.0f), b3 = __float_as_uint(q.w + 12582912.0f);
    return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Weight-job items a thread loads before it expands any.  The job has one item per thread up
// to 152 * 8 CTAs; past that cap each thread loops over several, and loading two at a time
// overlaps their latencies.  Measured on the 7B-class pair's fused calls (2.9 items per thread):
// 814 -> 802 and 939 -> 911 us.  (Halving the CTAs to give every thread two items had cost the
// 512-row linears of a decoder layer 0.6 us each.)
constexpr int kWeightItems = 2;

__device__ __forceinline__ float h2f(uint16_t bits) { return __half2float(__ushort_as_half(bits)); }

// The sums of H values (H in {1, 2, 4}) over each 16-lane half of the warp, reduced together:
// every halving step sends half of a lane's remaining values to its partner and keeps the
// other half, so H sums cost log2(H) + 4 shuffle steps instead of 4 H.  Lane l then holds
// value j = jsel(l) of its half's sums; lanes with (l & (16 / H - 1)) == 0 hold distinct j.
// The values are exact small integers, so every order gives the same bits.
template <int H>
__device__ __forceinline__ float half_warp_sums(const float (&p)[H], int lane, int& j) {
    float v;
    if constexpr (H == 4) {
        const bool u8 = lane & 8, u4 = lane & 4;
        float a0 = u8 ? p[2] : p[0], a1 = u8 ? p[3] : p[1];
        const float s0 = u8 ? p[0] : p[2], s1 = u8 ? p[1] : p[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, 8);
        a1 += __shfl_xor_sync(0xffffffffu, s1, 8);
        v = u4 ? a1 : a0;
        v += __shfl_xor_sync(0xffffffffu, u4 ? a0 : a1, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        j = (u8 ? 2 : 0) + (u4 ? 1 : 0);
    } else if constexpr (H == 2) {
        const bool u8 = lane & 8;
        v = u8 ? p[1] : p[0];
        v += __shfl_xor_sync(0xffffffffu, u8 ? p[0] : p[1], 8);
#pragma unroll
        for (int o = 4; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        j = u8 ? 1 : 0;
    } else {
        v = p[0];
#pragma unroll
        for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        j = 0;
    }
    return v;
}

// Weight job (the weight records of w4a8_internal.h), spread over the CTAs past the row
// CTAs.  One thread per (row n, block b), rows padded to a multiple of 128: the 32 packed
// bytes expanded to 64 e4m3 bytes in 64-byte-swizzled order; then {-z_w, -z_w} (fp16 pair,
// exact) with 12 zero bytes, and 512 s_w[n,b] (fp32, into the scale array; the power of two
// undoes the 2^-9 scale of the e4m3 weight operand); zeros for rows past N.
__device__ void weights_job(const PrepArgs& a, int64_t cta, int64_t ctas) {
    constexpr int U = kWeightItems;
    const int64_t nb = a.K / kBlock;
    const int64_t tiles = (a.N + kTileW - 1) / kTileW;
    const int64_t total = tiles * nb * kTileW;
    const int64_t stride = ctas * blockDim.x;
    // U items per thread, i0 + u * stride: every load of the U items goes out before the first
    // expansion, so their latencies overlap
    for (int64_t i0 = cta * blockDim.x + threadIdx.x; i0 < total; i0 += stride * U) {
        uint4 w0[U], w1[U];
        uint16_t sh[U], zh[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + u * stride;
            const int64_t rb = i >> 7;
            const int64_t n = (rb / nb) * kTileW + (i & 127);
            const int64_t b = rb - (rb / nb) * nb;
            w0[u] = w1[u] = make_uint4(0u, 0u, 0u, 0u);
            sh[u] = zh[u] = 0;
            if (i < total && n < a.N) {
                const uint4* src = reinterpret_cast<const uint4*>(a.wq + (a.n_first + n) * (a.K / 2) + b * 32);
                w0[u] = __ldcs(src);
                w1[u] = __ldcs(src + 1);
                if (a.s_w) {
                    const int64_t sidx = (a.n_first + n) * nb + b;
                    sh[u] = a.s_w[sidx];
                    zh[u] = a.z_w[sidx];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + u * stride;
            if (i >= total) break;
            const int64_t rb = i >> 7;
            const int r = static_cast<int>(i & 127);
            const int64_t n = (rb / nb) * kTileW + r;
            uint8_t* rec = a.wrec + rb * kWRec;
            uint4 o[4];
            expand8(w0[u].x, o[0].x, o[0].y);
            expand8(w0[u].y, o[0].z, o[0].w);
            expand8(w0[u].z, o[1].x, o[1].y);
            expand8(w0[u].w, o[1].z, o[1].w);
            expand8(w1[u].x, o[2].x, o[2].y);
            expand8(w1[u].y, o[2].z, o[2].w);
            expand8(w1[u].z, o[3].x, o[3].y);
            expand8(w1[u].w, o[3].z, o[3].w);
            const int sw = (r >> 1) & 3;
#pragma unroll
            for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(rec + r * 64 + ((c ^ sw) << 4)) = o[c];
            if (a.s_w) {
                const bool live = n < a.N;
                *reinterpret_cast<uint4*>(rec + kWZx + r * 16) =
                    make_uint4(live ? neg_zero_pair(zh[u]) : 0u, 0u, 0u, 0u);
                a.sc[i] = live ? 512.0f * h2f(sh[u]) : 0.0f;  // [tile][b][r]: the item's linear index
            }
        }
    }
}

// Register-resident pre-pass: G warps per row, V float4 per lane (row length K <= 128*G*V).
// With V <= 8 the next iteration's row is loaded while the current one is quantized.
template <int G, int V, bool PLANES, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 2 : 1) quant_kernel(const PrepArgs a, int row_ctas) {
    // the next kernel in the stream (the contraction, a programmatic dependent) may launch and
    // run its set-up now; it waits for this whole grid to complete before reading its outputs
    griddep_launch_dependents();
    if (static_cast<int>(blockIdx.x) >= row_ctas) {
        if (a.wrec) weights_job(a, blockIdx.x - row_ctas, gridDim.x - row_ctas);
        return;
    }
    constexpr bool kPrefetch = V <= 8;
    const int ts = a.tw == 256 ? 8 : 7;  // token record width 2^ts
    __shared__ float red[2][NW];
    constexpr int RPC = NW / G;  // rows per CTA iteration
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = warp % G, rsub = warp / G;
    const int64_t K = a.K, n4 = K / 4, nb = K / kBlock;
    const int64_t step = static_cast<int64_t>(row_ctas) * RPC;
    auto load = [&](float4 (&v)[V], int64_t m) {
        const bool active = m < a.M;
        const float4* xr = reinterpret_cast<const float4*>(a.x) + (active ? (a.row0 + m) * n4 : 0);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int64_t f = static_cast<int64_t>(i * G + wg) * 32 + lane;
            v[i] = (active && f < n4) ? __ldcs(xr + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float4 v[V], nv[V];
    int par = 0;
    int64_t base = static_cast<int64_t>(blockIdx.x) * RPC;
    if (base < a.M) load(v, base + rsub);
    for (; base < a.M; base += step) {
        const int64_t m = base + rsub;
        const bool active = m < a.M;
        if (kPrefetch && base + step < a.M) load(nv, base + step + rsub);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i)
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (G > 1) {
            if (lane == 0) red[par][warp] = amax;
            // only the G warps of this row meet (measured at 8192 x 4096, two rows per CTA: the
            // record pre-pass 43.0 -> 41.0 us, the API layout 34.8 -> 30.7 us against one
            // barrier for the whole CTA).  A group reads only its own warps' slots, and red[par]
            // alternates between iterations: a warp writes this slot again only after passing
            // the group's next barrier, which every reader of it reaches first.
            if constexpr (RPC > 1) named_bar_sync(1 + rsub, G * 32);
            else __syncthreads();
            float t = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j) t = fmaxf(t, red[par][rsub * G + j]);
            amax = t;
            par ^= 1;
        }
        const float s = __fdiv_rn(amax, 127.0f);
        const float r = __frcp_rn(s);
        if (active && wg == 0 && lane == 0 && a.s_a_out) a.s_a_out[m] = s;
        // the lane's V float4 in parts of H (bounded register pressure), each: quantize, write
        // the operand or codes, then the 64-element block sums with the chains interleaved
        constexpr int H = V > 8 ? V / 4 : (V >= 2 ? V / 2 : 1);
#pragma unroll
        for (int h0 = 0; h0 < V; h0 += H) {
            float4 xh[H], q[H];
#pragma unroll
            for (int j = 0; j < H; ++j) xh[j] = v[h0 + j];
            if (s > 0.0f) {  // s = 0 (absmax 0, or absmax / 127 below the smallest subnormal): codes 0
                quant_lane<H>(xh, q, s, r);
            } else {
#pragma unroll
                for (int j = 0; j < H; ++j) q[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float part[H];
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const int64_t f = static_cast<int64_t>((h0 + j) * G + wg) * 32 + lane;
                part[j] = (q[j].x + q[j].y) + (q[j].z + q[j].w);  // exact
                if (active && f < n4) {
                    if (PLANES) {
                        uint32_t hi, lo;
                        planes4f(q[j], hi, lo);
                        uint8_t* rec = token_rec(a.trec, m, f >> 4, nb, ts);
                        const int row = static_cast<int>(m & ((1 << ts) - 1)), j = static_cast<int>(f & 15);
                        *reinterpret_cast<uint32_t*>(rec + plane_off(row, j, 0)) = hi;
                        *reinterpret_cast<uint32_t*>(rec + plane_off(row, j, 1)) = lo;
                    } else {
                        *reinterpret_cast<uint32_t*>(a.a_q_out + m * K + 4 * f) = bytes4f(q[j]);
                    }
                }
            }
            int jj;
            const float bsum = half_warp_sums<H>(part, lane, jj);
            if (active && (lane & (16 / H - 1)) == 0) {
                const int64_t f = static_cast<int64_t>((h0 + jj) * G + wg) * 32 + lane;
                if (f < n4) {
                    const int64_t b = f >> 4;
                    const int rs = static_cast<int>(bsum);
                    if (PLANES)
                        *reinterpret_cast<uint4*>(token_rec(a.trec, m, b, nb, ts) + (128 << ts) + (m & ((1 << ts) - 1)) * 16) =
                            rx_entry(rs);
                    else a.rs_out[m * nb + b] = rs;
                }
            }
        }
        if (kPrefetch) {
#pragma unroll
            for (int i = 0; i < V; ++i) v[i] = nv[i];
        } else if (base + step < a.M) {
            load(v, base + step + rsub);
        }
    }
}

// Long rows (K > 16384): one CTA per row, absmax pass then a quantize pass that re-reads
// the row (from L2 in practice; HBM traffic stays one read).
template <bool PLANES>
__global__ void __launch_bounds__(256) quant_long_kernel(const PrepArgs a, int row_ctas) {
    // the next kernel in the stream (the contraction, a programmatic dependent) may launch and
    // run its set-up now; it waits for this whole grid to complete before reading its outputs
    griddep_launch_dependents();
    if (static_cast<int>(blockIdx.x) >= row_ctas) {
        if (a.wrec) weights_job(a, blockIdx.x - row_ctas, gridDim.x - row_ctas);
        return;
    }
    __shared__ float red[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t K = a.K, n4 = K / 4, nb = K / kBlock;
    const int ts = a.tw == 256 ? 8 : 7;  // token record width 2^ts
    for (int64_t m = blockIdx.x; m < a.M; m += row_ctas) {
        const float4* xr = reinterpret_cast<const float4*>(a.x) + (a.row0 + m) * n4;
        float amax = 0.0f;
        for (int64_t f = threadIdx.x; f < n4; f += 256) {
            const float4 v = xr[f];
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, red[j]);
        __syncthreads();
        const float s = __fdiv_rn(amax, 127.0f);
        if (threadIdx.x == 0 && a.s_a_out) a.s_a_out[m] = s;
        const bool nz = s > 0.0f;  // s = 0: every code 0
        // n4 is a multiple of 16, so every warp iteration covers whole blocks.
        for (int64_t f0 = 0; f0 < n4; f0 += 256) {
            const int64_t f = f0 + threadIdx.x;
            const bool in = f < n4;
            float4 v = in ? __ldcs(xr + f) : make_float4(0.f, 0.f, 0.f, 0.f);
            int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
            if (nz) {
                c0 = quant1(v.x, s);
                c1 = quant1(v.y, s);
                c2 = quant1(v.z, s);
                c3 = quant1(v.w, s);
            }
            int part = c0 + c1 + c2 + c3;
            part += __shfl_xor_sync(0xffffffffu, part, 8);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            if (in) {
                const int64_t b = f >> 4;
                if (PLANES) {
                    uint32_t hi, lo;
                    planes4(c0, c1, c2, c3, hi, lo);
                    uint8_t* rec = token_rec(a.trec, m, b, nb, ts);
                    const int r = static_cast<int>(m & ((1 << ts) - 1)), j = static_cast<int>(f & 15);
                    *reinterpret_cast<uint32_t*>(rec + plane_off(r, j, 0)) = hi;
                    *reinterpret_cast<uint32_t*>(rec + plane_off(r, j, 1)) = lo;
                    if ((lane & 15) == 0) *reinterpret_cast<uint4*>(rec + (128 << ts) + r * 16) = rx_entry(part);
                } else {
                    const uint32_t w = (c0 & 0xff) | ((c1 & 0xff) << 8) | ((c2 & 0xff) << 16) |
                                       (static_cast<uint32_t>(c3 & 0xff) << 24);
                    *reinterpret_cast<uint32_t*>(a.a_q_out + m * K + 4 * f) = w;
                    if ((lane & 15) == 0) a.rs_out[m * nb + b] = part;
                }
            }
        }
    }
}

// Pack pre-quantized int8 codes into the tensor-core planes; transpose the row sums;
// re-lay out the weight scales.  Rows row0 .. row0 + M - 1 of a_q_in.
__global__ void __launch_bounds__(256) pack_kernel(const PrepArgs a, int row_ctas) {
    // the next kernel in the stream (the contraction, a programmatic dependent) may launch and
    // run its set-up now; it waits for this whole grid to complete before reading its outputs
    griddep_launch_dependents();
    if (static_cast<int>(blockIdx.x) >= row_ctas) {
        if (a.wrec) weights_job(a, blockIdx.x - row_ctas, gridDim.x - row_ctas);
        return;
    }
    const int64_t K = a.K, nb = K / kBlock, c16 = K / 16;
    const int64_t total = a.M * c16;
    const int ts = a.tw == 256 ? 8 : 7;  // token record width 2^ts
    const int64_t stride = static_cast<int64_t>(row_ctas) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t m = i / c16, c = i - m * c16;
        const int4 w = *reinterpret_cast<const int4*>(a.a_q_in + (a.row0 + m) * K + 16 * c);
        const uint32_t words[4] = {static_cast<uint32_t>(w.x), static_cast<uint32_t>(w.y),
                                   static_cast<uint32_t>(w.z), static_cast<uint32_t>(w.w)};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t u = words[j];
            planes4(static_cast<int8_t>(u & 0xff), static_cast<int8_t>((u >> 8) & 0xff),
                    static_cast<int8_t>((u >> 16) & 0xff), static_cast<int8_t>(u >> 24), hi[j], lo[j]);
        }
        uint8_t* rec = token_rec(a.trec, m, c >> 2, nb, ts);
        const int r = static_cast<int>(m & ((1 << ts) - 1)), j4 = static_cast<int>(c & 3);
        *reinterpret_cast<uint4*>(rec + r * 128 + ((j4 ^ (r & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(rec + r * 128 + (((j4 + 4) ^ (r & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (a.rs_in) {
        const int64_t tot = a.M * nb;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < tot; i += stride) {
            const int64_t m = i / nb, b = i - m * nb;
            *reinterpret_cast<uint4*>(token_rec(a.trec, m, b, nb, ts) + (128 << ts) + (m & ((1 << ts) - 1)) * 16) =
                rx_entry(a.rs_in[(a.row0 + m) * nb + b]);
        }
    }
}

// CTAs for the weight job: one (row, block) item per thread up to eight CTAs per SM, then
// a few items per thread (each item is an independent 32-byte read, so many threads in
// flight hide the latency).
int weight_ctas(const PrepArgs& a) {
    if (!a.wrec) return 0;
    const int64_t items = ((a.N + kTileW - 1) / kTileW) * (a.K / kBlock) * kTileW;
    const int64_t c = (items + 255) / 256;
    return static_cast<int>(c < 152 * 8 ? c : 152 * 8);
}

// CTAs of quant_kernel<G, V, PLANES, NW> resident on one SM (its register use decides), asked
// once per instantiation.
template <int G, int V, bool PLANES, int NW = 8>
int ctas_per_sm() {
    static std::atomic<int> n{0};
    int v = n.load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, quant_kernel<G, V, PLANES, NW>, NW * 32, 0) !=
                cudaSuccess ||
            v < 1) {
            // not remembered, and cleared, so that the launch that follows reports only its own
            // status: two per SM, what these kernels' launch bounds guarantee for 256 threads
            (void)cudaGetLastError();
            return NW == 8 ? 2 : 1;
        }
        n.store(v, std::memory_order_relaxed);
    }
    return v;
}

template <int G, int V, bool PLANES, int NW = 8>
cudaError_t run_quant(const PrepArgs& a, cudaStream_t s) {
    constexpr int RPC = NW / G;
    const int64_t need = (a.M + RPC - 1) / RPC;
    // as many row CTAs as fit on the GPU at once (two 256-thread or one 512-thread CTA per
    // SM), with the rows spread evenly: each CTA walks its rows with the next one in flight
    constexpr int64_t cap = NW == 8 ? 152 * 2 : 152;
    const int64_t iters = (need + cap - 1) / cap;
    const int row_ctas = static_cast<int>(iters > 0 ? (need + iters - 1) / iters : 1);
    const int grid = row_ctas + weight_ctas(a);
    quant_kernel<G, V, PLANES, NW><<<grid, NW * 32, 0, s>>>(a, row_ctas);
    return cudaGetLastError();
}

// The row CTAs run_quant launches for G warps per row (8-warp CTAs).
int64_t quant_row_ctas(int64_t M, int G) {
    const int64_t rpc = 8 / G, need = (M + rpc - 1) / rpc, cap = 152 * 2;
    const int64_t iters = (need + cap - 1) / cap;
    return iters > 0 ? (need + iters - 1) / iters : 1;
}

template <bool PLANES>
cudaError_t dispatch_quant(const PrepArgs& a, cudaStream_t s) {
    const int64_t n4 = a.K / 4;
    // Short rows: more warps per row (shorter chains per lane, more SMs) while the whole launch,
    // the weight job's CTAs included, still fits one wave (as many 256-thread CTAs per SM as the
    // instantiation's registers allow: three for four warps per row).  Measured at 128 and 512
    // rows of 1024: the pre-pass alone 8.2 -> 6.1 us with four warps per row; the fused pp512
    // call (512 rows, 192 weight-job CTAs: 448 CTAs in all) 18.1 -> 17.0 us per step.
    if (n4 <= 128 * 2 && quant_row_ctas(a.M, 4) + weight_ctas(a) <= 152 * ctas_per_sm<4, 2, PLANES>())
        return run_quant<4, 2, PLANES>(a, s);
    if (n4 <= 64 * 4 && quant_row_ctas(a.M, 2) + weight_ctas(a) <= 152 * ctas_per_sm<2, 4, PLANES>())
        return run_quant<2, 4, PLANES>(a, s);
    // smallest warp group G whose lanes hold the row in at most 8 float4 each (so the next
    // row can be prefetched): 1-8 warps of a 256-thread CTA, then the 16 warps of a 512-thread
    // CTA; past that, the two-pass kernel
    if (n4 <= 32 * 2) return run_quant<1, 2, PLANES>(a, s);
    if (n4 <= 32 * 4) return run_quant<1, 4, PLANES>(a, s);
    if (n4 <= 32 * 8) return run_quant<1, 8, PLANES>(a, s);
    if (n4 <= 64 * 8) return run_quant<2, 8, PLANES>(a, s);
    if (n4 <= 128 * 8) return run_quant<4, 8, PLANES>(a, s);
    if (n4 <= 256 * 8) return run_quant<8, 8, PLANES>(a, s);
    if (n4 <= 512 * 8) return run_quant<16, 8, PLANES, 16>(a, s);  // 512-thread CTAs, one row each
    const int row_ctas = static_cast<int>(a.M < 152 * 4 ? a.M : 152 * 4);
    quant_long_kernel<PLANES><<<row_ctas + weight_ctas(a), 256, 0, s>>>(a, row_ctas);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant(const PrepArgs& a, cudaStream_t s) {
    return a.trec ? dispatch_quant<true>(a, s) : dispatch_quant<false>(a, s);
}

cudaError_t launch_pack(const PrepArgs& a, cudaStream_t s) {
    const int64_t work = a.M * (a.K / 16);
    const int64_t need = (work + 255) / 256;
    int row_ctas = static_cast<int>(need < 152 * 8 ? need : 152 * 8);
    if (row_ctas < 1) row_ctas = 1;
    pack_kernel<<<row_ctas + weight_ctas(a), 256, 0, s>>>(a, row_ctas);
    return cudaGetLastError();
}

}  // namespace w4a8
