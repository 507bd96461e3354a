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
// The same launch also re-lays out the fp16 weight scales and zeros for the epilogue
// (extra CTAs), so a call costs two launches in total.
#include "sm103_ptx.cuh"
#include "w4a8_internal.h"

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

// Position of weight row n in a prepared-scale row (see the wsc layout in w4a8_internal.h).
__device__ __forceinline__ int64_t perm32(int64_t n) {
    const int r = static_cast<int>(n & 31);
    return (n & ~static_cast<int64_t>(31)) + ((r & 7) << 2) + (r >> 3);
}

// INT8 code of one activation: clamp(round_half_away(x / s), -127, 127), fp32 IEEE division.
__device__ __forceinline__ int quant1(float x, float s) {
    float r = roundf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

__device__ __forceinline__ float h2f(uint16_t bits) { return __half2float(__ushort_as_half(bits)); }

// Weight-scale job: per block b, 512 s_w[n,b] (fp32, rows permuted by perm32; the power
// of two undoes the 2^-9 scale of the e4m3 weight operand) and {-z_w, -z_w} (fp16x2, row
// order) for the zero-point MMA; zeros past N.
__device__ void scales_job(const PrepArgs& a, int64_t cta, int64_t ctas) {
    const int64_t nb = a.K / kBlock;
    const int64_t total = nb * a.N_pad;
    for (int64_t i = cta * blockDim.x + threadIdx.x; i < total; i += ctas * blockDim.x) {
        const int64_t b = i / a.N_pad;
        const int64_t n = i - b * a.N_pad;
        float sv = 0.0f;
        uint32_t zz = 0u;
        if (n < a.N) {
            sv = 512.0f * h2f(a.s_w[n * nb + b]);
            const uint32_t zb = static_cast<uint32_t>(a.z_w[n * nb + b]) ^ 0x8000u;  // -z_w, exact
            zz = zb | (zb << 16);
        }
        float* row = a.wsc + b * 2 * a.N_pad;
        row[perm32(n)] = sv;
        reinterpret_cast<uint32_t*>(row + a.N_pad)[n] = zz;
    }
}

// Register-resident pre-pass: G warps per row, V float4 per lane (row length K <= 128*G*V).
template <int G, int V, bool PLANES>
__global__ void __launch_bounds__(256) quant_kernel(const PrepArgs a, int row_ctas) {
    if (static_cast<int>(blockIdx.x) >= row_ctas) {
        if (a.wsc) scales_job(a, blockIdx.x - row_ctas, gridDim.x - row_ctas);
        return;
    }
    __shared__ float red[2][8];
    constexpr int RPC = 8 / G;  // rows per CTA iteration
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = warp % G, rsub = warp / G;
    const int64_t K = a.K, n4 = K / 4, nb = K / kBlock;
    int par = 0;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * RPC; base < a.M;
         base += static_cast<int64_t>(row_ctas) * RPC) {
        const int64_t m = base + rsub;
        const bool active = m < a.M;
        const float4* xr = reinterpret_cast<const float4*>(a.x) + (active ? (a.row0 + m) * n4 : 0);
        float4 v[V];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int64_t f = static_cast<int64_t>(i * G + wg) * 32 + lane;
            if (active && f < n4) {
                v[i] = __ldcs(xr + f);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
            } else {
                v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (G > 1) {
            if (lane == 0) red[par][warp] = amax;
            __syncthreads();
            float t = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j) t = fmaxf(t, red[par][rsub * G + j]);
            amax = t;
            par ^= 1;
        }
        const float s = __fdiv_rn(amax, 127.0f);
        if (active && wg == 0 && lane == 0) {
            if (a.s_a_out) a.s_a_out[m] = s;
        }
        const bool nz = amax > 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int64_t f = static_cast<int64_t>(i * G + wg) * 32 + lane;
            int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
            if (nz) {
                c0 = quant1(v[i].x, s);
                c1 = quant1(v[i].y, s);
                c2 = quant1(v[i].z, s);
                c3 = quant1(v[i].w, s);
            }
            int part = c0 + c1 + c2 + c3;  // 16 lanes = one 64-element block
            part += __shfl_xor_sync(0xffffffffu, part, 8);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            if (active && f < n4) {
                const int64_t b = f >> 4;
                if (PLANES) {
                    uint32_t hi, lo;
                    planes4(c0, c1, c2, c3, hi, lo);
                    uint8_t* dst = a.apk + m * (2 * K) + b * 128 + ((f & 15) << 2);
                    *reinterpret_cast<uint32_t*>(dst) = hi;
                    *reinterpret_cast<uint32_t*>(dst + 64) = lo;
                    if ((lane & 15) == 0) a.rx[b * a.M_pad + m] = rx_entry(part);
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

// Long rows (K > 16384): one CTA per row, absmax pass then a quantize pass that re-reads
// the row (from L2 in practice; HBM traffic stays one read).
template <bool PLANES>
__global__ void __launch_bounds__(256) quant_long_kernel(const PrepArgs a, int row_ctas) {
    if (static_cast<int>(blockIdx.x) >= row_ctas) {
        if (a.wsc) scales_job(a, blockIdx.x - row_ctas, gridDim.x - row_ctas);
        return;
    }
    __shared__ float red[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t K = a.K, n4 = K / 4, nb = K / kBlock;
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
        const bool nz = amax > 0.0f;
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
                    uint8_t* dst = a.apk + m * (2 * K) + b * 128 + ((f & 15) << 2);
                    *reinterpret_cast<uint32_t*>(dst) = hi;
                    *reinterpret_cast<uint32_t*>(dst + 64) = lo;
                    if ((lane & 15) == 0) a.rx[b * a.M_pad + m] = rx_entry(part);
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
    if (static_cast<int>(blockIdx.x) >= row_ctas) {
        if (a.wsc) scales_job(a, blockIdx.x - row_ctas, gridDim.x - row_ctas);
        return;
    }
    const int64_t K = a.K, nb = K / kBlock, c16 = K / 16;
    const int64_t total = a.M * c16;
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
        const int64_t b = c >> 2;
        uint8_t* dst = a.apk + m * (2 * K) + b * 128 + ((c & 3) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(dst + 64) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (a.rs_in && a.rx) {
        const int64_t tot = a.M * nb;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < tot; i += stride) {
            const int64_t b = i / a.M, m = i - b * a.M;
            a.rx[b * a.M_pad + m] = rx_entry(a.rs_in[(a.row0 + m) * nb + b]);
        }
    }
}

int scale_ctas(const PrepArgs& a) {
    if (!a.wsc) return 0;
    const int64_t total = (a.K / kBlock) * a.N_pad;
    const int64_t c = (total + 255) / 256;
    return static_cast<int>(c < 304 ? c : 304);
}

template <int G, int V, bool PLANES>
cudaError_t run_quant(const PrepArgs& a, cudaStream_t s) {
    constexpr int RPC = 8 / G;
    const int64_t need = (a.M + RPC - 1) / RPC;
    const int row_ctas = static_cast<int>(need < 152 * 8 ? need : 152 * 8);
    const int grid = row_ctas + scale_ctas(a);
    quant_kernel<G, V, PLANES><<<grid, 256, 0, s>>>(a, row_ctas);
    return cudaGetLastError();
}

template <bool PLANES>
cudaError_t dispatch_quant(const PrepArgs& a, cudaStream_t s) {
    const int64_t n4 = a.K / 4;
    // smallest warp group G whose lanes hold the row in at most 16 float4 each
    if (n4 <= 32 * 2) return run_quant<1, 2, PLANES>(a, s);
    if (n4 <= 32 * 4) return run_quant<1, 4, PLANES>(a, s);
    if (n4 <= 32 * 8) return run_quant<1, 8, PLANES>(a, s);
    if (n4 <= 32 * 16) return run_quant<1, 16, PLANES>(a, s);
    if (n4 <= 64 * 16) return run_quant<2, 16, PLANES>(a, s);
    if (n4 <= 128 * 16) return run_quant<4, 16, PLANES>(a, s);
    if (n4 <= 256 * 16) return run_quant<8, 16, PLANES>(a, s);
    const int row_ctas = static_cast<int>(a.M < 152 * 4 ? a.M : 152 * 4);
    quant_long_kernel<PLANES><<<row_ctas + scale_ctas(a), 256, 0, s>>>(a, row_ctas);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant(const PrepArgs& a, cudaStream_t s) {
    return a.apk ? dispatch_quant<true>(a, s) : dispatch_quant<false>(a, s);
}

cudaError_t launch_pack(const PrepArgs& a, cudaStream_t s) {
    const int64_t work = a.M * (a.K / 16);
    const int64_t need = (work + 255) / 256;
    int row_ctas = static_cast<int>(need < 152 * 8 ? need : 152 * 8);
    if (row_ctas < 1) row_ctas = 1;
    pack_kernel<<<row_ctas + scale_ctas(a), 256, 0, s>>>(a, row_ctas);
    return cudaGetLastError();
}

}  // namespace w4a8
