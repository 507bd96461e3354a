// gemm.cu -- block-64 W4A8 contraction on the sm_103a tensor cores + direct epilogue.
//
// "MNN LLM inference on the SpacemiT K3", section 3 eqs. (2)-(3) and section 4 steps 2-3.
// There is no integer MMA kind on sm_103a, so the exact INT8 x U4 block products are
// carried on the fp8 kind (tcgen05.mma kind::f8f6f4, E4M3 x E4M3 -> fp32 in TMEM):
//   - activations arrive as the two nibble planes of eq. (3): e4m3(16*(a>>4)) and
//     e4m3(a&15), both exact;
//   - a u4 weight code q, zero-extended to a byte, is exactly the e4m3 encoding of
//     q * 2^-9 (subnormal + first normal binade share the step 2^-9), so the in-shared-
//     memory unpack is two masks and two byte permutes per 8 weights;
//   - one block = 4 MMAs of K = 32 (hi plane x q, then lo plane x q) into one TMEM
//     accumulator, which then holds acc * 2^-9 with |acc| <= 127*15*64 < 2^17: exact
//     in fp32 provided the tensor core does not drop low-order bits (checked bit-exactly
//     against the oracle by the debug call);
//   - every 64-block gets its own accumulator (two TMEM buffers, ping-pong), drained by
//     the epilogue warps: t = fma(-z/512, rs, acc') (one rounding of acc - z*rs),
//     y += (512 s) * t, then y_out = fma(s_a, y, bias) written straight to HBM.
//
// Warp roles (one CTA = one 128 x BN output tile, 12 warps):
//   warp 0      TMA producer: activation planes (128-byte swizzle), packed weights, and
//               (bulk copies) the block's scales and row sums
//   warp 1      TMEM allocation + single-thread MMA issue
//   warps 2-3   weight unpack u4 -> e4m3 into the 64-byte-swizzled K-major operand
//   warps 4-11  epilogue (two warps per 32-lane TMEM quarter, half of the columns each)
// Every wait is bounded (WaitCtl); a CTA that gives up records a timeout and unwinds.
#include "sm103_ptx.cuh"
#include "w4a8_internal.h"

namespace w4a8 {
namespace {

template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int kSc = kStages + 4;  // scale/row-sum ring (outlives the MMA stage)
    static constexpr int kABytes = kTileM * 128;
    static constexpr int kBunpBytes = BN * 64;
    static constexpr int kBpkBytes = BN * 32;
    static constexpr int kSzBytes = BN * 8;
    static constexpr int kRBytes = kTileM * 4;
    static constexpr int kOffA = 0;
    static constexpr int kOffBunp = kOffA + kStages * kABytes;
    static constexpr int kOffBpk = kOffBunp + kStages * kBunpBytes;
    static constexpr int kOffSz = kOffBpk + kStages * kBpkBytes;
    static constexpr int kOffR = kOffSz + kSc * kSzBytes;
    static constexpr int kOffBar = kOffR + kSc * kRBytes;
    static constexpr int kNumBars = 3 * kStages + 2 * kSc + 5;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static constexpr uint32_t kTmemCols = 2 * BN;
    static_assert(kOffBunp % 1024 == 0 && kOffBpk % 1024 == 0, "operand tiles must be 1024-aligned");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

constexpr int kThreads = 384;
constexpr uint32_t kLayoutSw128 = 2, kLayoutSw64 = 4;

// u4 pairs -> e4m3 bytes in k order: nibbles k0..k7 of w become bytes of (o0: k0..k3, o1: k4..k7).
__device__ __forceinline__ void expand8(uint32_t w, uint32_t& o0, uint32_t& o1) {
    const uint32_t lo = w & 0x0F0F0F0Fu;         // k0 k2 k4 k6
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // k1 k3 k5 k7
    o0 = __byte_perm(lo, hi, 0x5140);
    o1 = __byte_perm(lo, hi, 0x7362);
}

// Bounded wait that ignores the abort flag: used while unwinding to let copies and MMAs
// already in flight land before the CTA's shared memory and TMEM are released.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return;
    }
}

template <int BN, bool DEBUG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
    using C = Cfg<BN>;
    constexpr int S = C::kStages, SC = C::kSc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + S;
    uint64_t* unp = empty + S;
    uint64_t* scfull = unp + S;
    uint64_t* scempty = scfull + SC;
    uint64_t* tfull = scempty + SC;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_n = (args.n_cnt + BN - 1) / BN;
    const int64_t tm = blockIdx.x / tiles_n, tn = blockIdx.x - tm * tiles_n;
    const int64_t mt0 = tm * kTileM;            // first operand row of the tile
    const int64_t nt0 = args.n0 + tn * BN;      // first weight row (output column) of the tile
    const int nb = static_cast<int>(args.K / kBlock);
    const WaitCtl ctl{abort_flag, args.status, args.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&unp[s], 64);
        }
        for (int c = 0; c < SC; ++c) {
            mbar_init(&scfull[c], 1);
            mbar_init(&scempty[c], 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // BN = 256 needs 128 accumulator registers per epilogue thread: move registers from
    // the producer/MMA/unpack warpgroup (warps 0-3) to the two epilogue warpgroups.
    // 128 x 64 + 256 x 208 = 61440 <= 384 x 168 registers at launch.
    if (warp < 4) {
    if (BN == 256) regs_dec<64>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int nA = 0, nS = 0;  // blocks whose operand / scale copies were issued
            for (int b = 0; b < nb; ++b) {
                const int s = b % S, k = b / S;
                if (k > 0 && !mbar_wait(&empty[s], (k - 1) & 1, ctl)) break;
                mbar_arrive_expect_tx(&full[s], C::kABytes + C::kBpkBytes);
                tma_load_2d(smem + C::kOffA + s * C::kABytes, &tmA, &full[s], b * 128, static_cast<int32_t>(mt0));
                tma_load_2d(smem + C::kOffBpk + s * C::kBpkBytes, &tmB, &full[s], b * 32,
                            static_cast<int32_t>(nt0));
                nA = b + 1;
                if (!DEBUG) {
                    const int c = b % SC, kc = b / SC;
                    if (kc > 0 && !mbar_wait(&scempty[c], (kc - 1) & 1, ctl)) break;
                    mbar_arrive_expect_tx(&scfull[c], C::kSzBytes + C::kRBytes);
                    bulk_load(smem + C::kOffSz + c * C::kSzBytes,
                              args.sz + (static_cast<int64_t>(b) * args.N_pad + nt0) / 2, C::kSzBytes, &scfull[c]);
                    bulk_load(smem + C::kOffR + c * C::kRBytes, args.rT + static_cast<int64_t>(b) * args.M_pad + mt0,
                              C::kRBytes, &scfull[c]);
                    nS = b + 1;
                }
            }
            if (*abort_flag) {
                // let every copy already issued land before the CTA exits
                for (int j = (nA > S ? nA - S : 0); j < nA; ++j) drain_wait(&full[j % S], (j / S) & 1, 100000000ull);
                for (int j = (nS > SC ? nS - SC : 0); j < nS; ++j)
                    drain_wait(&scfull[j % SC], (j / SC) & 1, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kTileM, BN);
            for (int b = 0; b < nb; ++b) {
                const int s = b % S, k = b / S;
                if (!mbar_wait(&unp[s], k & 1, ctl)) break;
                if (!mbar_wait(&full[s], k & 1, ctl)) break;
                const int buf = b & 1, u = b >> 1;
                if (u > 0 && !mbar_wait(&tempty[buf], (u - 1) & 1, ctl)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
                const uint32_t a0 = smem_u32(smem + C::kOffA + s * C::kABytes);
                const uint32_t b0 = smem_u32(smem + C::kOffBunp + s * C::kBunpBytes);
                // hi plane x q (K 0..31, 32..63), then lo plane x q
                mma_f8f6f4(d, smem_desc(a0 + 0, 1024, kLayoutSw128), smem_desc(b0 + 0, 512, kLayoutSw64), idesc, 0u);
                mma_f8f6f4(d, smem_desc(a0 + 32, 1024, kLayoutSw128), smem_desc(b0 + 32, 512, kLayoutSw64), idesc, 1u);
                mma_f8f6f4(d, smem_desc(a0 + 64, 1024, kLayoutSw128), smem_desc(b0 + 0, 512, kLayoutSw64), idesc, 1u);
                mma_f8f6f4(d, smem_desc(a0 + 96, 1024, kLayoutSw128), smem_desc(b0 + 32, 512, kLayoutSw64), idesc, 1u);
                mma_commit(&empty[s]);
                mma_commit(&tfull[buf]);
            }
            mma_commit(drain);
            drain_wait(drain, 0, 100000000ull);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ weight unpack
        const int ut = threadIdx.x - 64;
        for (int b = 0; b < nb; ++b) {
            const int s = b % S, k = b / S;
            if (!mbar_wait(&full[s], k & 1, ctl)) break;
            const uint8_t* src = smem + C::kOffBpk + s * C::kBpkBytes;
            uint8_t* dst = smem + C::kOffBunp + s * C::kBunpBytes;
#pragma unroll 4
            for (int c = ut; c < BN * 2; c += 64) {
                const int row = c >> 1, half = c & 1;
                const uint4 w = *reinterpret_cast<const uint4*>(src + c * 16);
                uint4 o0, o1;
                expand8(w.x, o0.x, o0.y);
                expand8(w.y, o0.z, o0.w);
                expand8(w.z, o1.x, o1.y);
                expand8(w.w, o1.z, o1.w);
                const int sw = (row >> 1) & 3;  // 64-byte swizzle: chunk ^= address bits 7..8
                *reinterpret_cast<uint4*>(dst + row * 64 + (((2 * half) ^ sw) << 4)) = o0;
                *reinterpret_cast<uint4*>(dst + row * 64 + (((2 * half + 1) ^ sw) << 4)) = o1;
            }
            fence_proxy_async_smem();
            mbar_arrive(&unp[s]);
        }
    }
    } else {
        // ------------------------------------------------------------ epilogue
        if (BN == 256) regs_inc<208>();
        constexpr int G = BN / 16;  // 8-column groups per thread
        const int q = warp & 3, h = (warp - 4) >> 2;
        const int r8 = lane >> 2, cp = lane & 3;
        float2 yv[4][G];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g) yv[i][g] = make_float2(0.f, 0.f);
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * (BN / 2));
        for (int b = 0; b < nb; ++b) {
            const int buf = b & 1, u = b >> 1;
            const int c = b % SC, kc = b / SC;
            if (!mbar_wait(&tfull[buf], u & 1, ctl)) break;
            if (!DEBUG && !mbar_wait(&scfull[c], kc & 1, ctl)) break;
            tc_fence_after();
            float4 R4 = make_float4(0.f, 0.f, 0.f, 0.f);
            const float* szb = reinterpret_cast<const float*>(smem + C::kOffSz + c * C::kSzBytes);
            if (!DEBUG) R4 = *reinterpret_cast<const float4*>(smem + C::kOffR + c * C::kRBytes + (q * 32 + r8 * 4) * 4);
            const float Rr[4] = {R4.x, R4.y, R4.z, R4.w};
#pragma unroll
            for (int ch = 0; ch < G / 4; ++ch) {
                uint32_t v0[16], v1[16];
                const uint32_t ta = lane_addr + static_cast<uint32_t>(buf * BN + ch * 32);
                tmem_ld_16x256b_x4(ta, v0);
                tmem_ld_16x256b_x4(ta + (16u << 16), v1);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int g = ch * 4 + j;
                    const int col = h * (BN / 2) + g * 8 + 2 * cp;  // column within the tile
                    float2 a2[4];
                    a2[0] = make_float2(__uint_as_float(v0[4 * j + 0]), __uint_as_float(v0[4 * j + 1]));
                    a2[1] = make_float2(__uint_as_float(v0[4 * j + 2]), __uint_as_float(v0[4 * j + 3]));
                    a2[2] = make_float2(__uint_as_float(v1[4 * j + 0]), __uint_as_float(v1[4 * j + 1]));
                    a2[3] = make_float2(__uint_as_float(v1[4 * j + 2]), __uint_as_float(v1[4 * j + 3]));
                    if (DEBUG) {
                        const int64_t n = nt0 + col;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t m = mt0 + q * 32 + r8 + 8 * i;
                            if (m < args.m_cnt) {
                                int32_t* dst = args.acc + (m * args.n_cnt + (n - args.n0)) * nb + b;
                                if (n < args.n0 + args.n_cnt) dst[0] = static_cast<int32_t>(a2[i].x * 512.0f);
                                if (n + 1 < args.n0 + args.n_cnt) dst[nb] = static_cast<int32_t>(a2[i].y * 512.0f);
                            }
                        }
                    } else {
                        const float4 S4 = *reinterpret_cast<const float4*>(szb + col * 2);
                        const float2 sc = make_float2(S4.x, S4.y), mz = make_float2(S4.z, S4.w);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 t2 = __ffma2_rn(mz, make_float2(Rr[i], Rr[i]), a2[i]);
                            yv[i][g] = __ffma2_rn(sc, t2, yv[i][g]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tempty[buf]);
                if (!DEBUG) mbar_arrive(&scempty[c]);
            }
        }
        if (!DEBUG && !*abort_flag) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t m = mt0 + q * 32 + r8 + 8 * i;
                if (m >= args.M) continue;
                const float sa = args.s_a[m];
                float* yrow = args.y + m * args.N;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int64_t n = nt0 + h * (BN / 2) + g * 8 + 2 * cp;
                    if (n + 1 < args.N) {
                        const float b0 = args.bias ? args.bias[n] : 0.0f;
                        const float b1 = args.bias ? args.bias[n + 1] : 0.0f;
                        const float2 o = make_float2(fmaf(sa, yv[i][g].x, b0), fmaf(sa, yv[i][g].y, b1));
                        if ((args.N & 1) == 0) {
                            *reinterpret_cast<float2*>(yrow + n) = o;
                        } else {
                            yrow[n] = o.x;
                            yrow[n + 1] = o.y;
                        }
                    } else if (n < args.N) {
                        const float b0 = args.bias ? args.bias[n] : 0.0f;
                        yrow[n] = fmaf(sa, yv[i][g].x, b0);
                    }
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// A CTA that waits on a barrier nothing completes, to exercise the bounded-wait path.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    const WaitCtl ctl{&abort_flag, status, limit_ns};
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, ctl);
    __syncthreads();
}

template <int BN, bool DEBUG>
cudaError_t run(const GemmMaps& maps, const GemmArgs& a, cudaStream_t s) {
    using C = Cfg<BN>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, DEBUG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const int64_t tiles = ((a.m_cnt + kTileM - 1) / kTileM) * ((a.n_cnt + BN - 1) / BN);
    gemm_kernel<BN, DEBUG><<<static_cast<unsigned>(tiles), kThreads, C::kSmemBytes, s>>>(maps.a, maps.b, a);
    return cudaGetLastError();
}

}  // namespace

int pick_block_n(int64_t m_cnt, int64_t n_cnt, int num_sms) {
    // Estimated time ~ waves * (BN + fixed per-tile cost); ties go to the wider tile.
    int best = 256;
    int64_t best_cost = -1;
    const int cands[3] = {256, 128, 64};
    for (int bn : cands) {
        const int64_t tiles = ((m_cnt + kTileM - 1) / kTileM) * ((n_cnt + bn - 1) / bn);
        const int64_t waves = (tiles + num_sms - 1) / num_sms;
        const int64_t cost = waves * (bn + 48);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

cudaError_t launch_gemm(const GemmMaps& maps, const GemmArgs& a, int block_n, bool debug, int num_sms,
                        cudaStream_t s) {
    (void)num_sms;
    switch (block_n) {
        case 256: return debug ? run<256, true>(maps, a, s) : run<256, false>(maps, a, s);
        case 128: return debug ? run<128, true>(maps, a, s) : run<128, false>(maps, a, s);
        case 64: return debug ? run<64, true>(maps, a, s) : run<64, false>(maps, a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace w4a8
