// gemm.cu -- block-64 W4A8 contraction on the sm_103a tensor cores + direct epilogue.
//
// "MNN LLM inference on the SpacemiT K3", section 3 eqs. (2)-(3) and section 4 steps 2-3.
// There is no integer MMA kind on sm_103a, so the exact INT8 x U4 block products are
// carried on the fp8 kind (tcgen05.mma kind::f8f6f4, E4M3 x E4M3 -> fp32 in TMEM):
//   - the weights arrive expanded to one byte per u4 code q (the pre-pass does it), and
//     that byte is exactly the e4m3 encoding of q * 2^-9 (the subnormal binade and the
//     first normal binade share the step 2^-9);
//   - activations arrive as the two nibble planes of eq. (3): e4m3(16*(a>>4)) and
//     e4m3(a&15), both exact;
//   - one 64-block = 4 MMAs of K = 32 (q x hi plane, then q x lo plane) into one TMEM
//     accumulator, which then holds acc * 2^-9 with |acc| <= 128*15*64 < 2^17, exact in
//     fp32 (checked bit for bit against the oracle through the debug call);
//   - the zero-point term of eq. (2) is a fifth MMA on the same accumulator (kind::f16,
//     K = 16, two live K slots): weights {-z_w, -z_w}, tokens {rh/8, rl/512} with the row
//     sum rs = 64 rh + rl, all exact in fp16, so the accumulator ends the block holding
//     (acc - z_w rs) * 2^-9;
//   - every 64-block gets its own accumulator (four TMEM buffers of 128 columns), drained
//     by the epilogue warps two blocks at a time with one fma per output and block,
//     y += (512 s_w) * D; at the end of a tile y_out = fma(s_a, y, bias) goes straight
//     to HBM.
//
// Orientation: the weights are the MMA's M = 128 operand (TMEM lanes = output columns n)
// and the tokens its N = 128 operand.  An epilogue thread owns one weight row (its TMEM
// lane) and 32 token columns, so s_w is one scalar per thread and block.
//
// Every operand of a (tile, 64-block) pair sits in one record written by the pre-pass in
// shared-memory order (w4a8_internal.h): token planes + token zero-point rows, and e4m3
// weights + weight zero-point rows + scales.  A pipeline stage holds two consecutive
// blocks and is filled by two bulk copies: issuing an asynchronous copy or barrier
// operation costs a thread on the order of a hundred cycles, so the copy count per block,
// not the bytes, decides whether the producer keeps up with the tensor pipe.  The weight
// scales stay out of the records: the epilogue loads them from memory one stage ahead, so
// a stage is free as soon as its MMAs complete.
//
// Warp roles (one persistent CTA per SM walking 128 x 128 output tiles, 20 warps):
//   warp 0       producer: two bulk copies per stage
//   warps 1-3    MMA issue, one stage each in turn; one lane of the warp issues.  The
//                issue cost of one thread's MMA sequence exceeds the tensor time of a
//                stage, three warps' together do not.  Warp 1 also owns TMEM.
//   warps 4-19   epilogue: 4 warps per 32-lane TMEM quarter, 32 of the 128 columns each;
//                a stage's two blocks per drain keep four TMEM loads in flight per wait
//
// The barrier of a stage gates its MMAs: it completes once the stage's copies have landed
// (producer arrival + transaction bytes) and the epilogue has released the two TMEM
// buffers the stage overwrites (one arrival per epilogue warp), so an issuer waits once per
// block.  The epilogue drains a stage's two blocks together (four TMEM loads in flight per
// wait), releases their buffers as soon as the accumulators are in registers, then folds
// them into y; it frees a stage once its accumulators are complete.  Every wait is bounded (WaitCtl); a CTA
// that gives up records a timeout and unwinds.
#include "epilogue.cuh"
#include "sm103_ptx.cuh"
#include "w4a8_internal.h"

namespace w4a8 {
namespace {

constexpr int kThreads = 640;
constexpr int kEpiWarps = 16;
constexpr int kIssuers = 3;
constexpr int kStages = 3;    // stages of two blocks
constexpr int kNBuf = 4;      // TMEM accumulator buffers of kTileT columns (two per stage)
constexpr uint32_t kLayoutSw128 = 2, kLayoutSw64 = 4;
// Register split: launch = 640 x 96 (checked at build time); warps 0-3 drop to 32,
// the 16 epilogue warps rise to 112: 128*32 + 512*112 = 61440 = 640*96.
constexpr int kRegsLow = 32, kRegsHigh = 112;

constexpr int kStageTok = 2 * kTokRec;               // token records of a stage's two blocks
constexpr int kStageBytes = kStageTok + 2 * kWRec;   // + weight records
constexpr int kZeroBytes = 4096;                     // K 8..15 of both zero-point operands
constexpr int kOffZero = kStages * kStageBytes;
constexpr int kOffBar = kOffZero + kZeroBytes;
constexpr int kNumBars = 2 * kStages + 2 + kIssuers;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = kNBuf * kTileT;
static_assert(kTokRec % 1024 == 0 && kWRec % 1024 == 0 && kStageBytes % 1024 == 0,
              "swizzled operand tiles must stay 1024-aligned");
static_assert(kSmemBytes + 2 * 16 * 32 * 4 <= 227 * 1024, "shared memory budget (with the static epilogue slots)");
static_assert(kTmemCols == 512, "TMEM allocation");
static_assert(kNBuf / 2 <= kStages, "a stage barrier carries a buffer release only after its previous phase");
static_assert(kZeroBytes >= kTileW * 16 && kZeroBytes >= kTileT * 16, "zero half of the zero-point operands");
// An mbarrier wait on parity P returns at once while the phase before P is still open, so a
// warp that waits for phase k + 1 of a stage must itself have seen phase k complete.  With
// the work items 2j + k dealt round-robin to the issuers, the issuer of a stage's slot k is
// the same warp at every phase of that stage only if the issuer count divides the number of
// slots per round of the stages.
static_assert((2 * kStages) % kIssuers == 0, "each stage slot must have one issuer warp at every phase");

// Grouped raster over the output tiles: groups of kGroup token tiles, the token tile
// varying fastest inside a group, so the CTAs running at one time share token and weight
// tiles in L2.
constexpr int64_t kGroup = 8;
__device__ __forceinline__ void tile_at(int64_t t, int64_t tiles_t, int64_t tiles_w, int64_t& tt, int64_t& tw) {
    const int64_t per = kGroup * tiles_w;
    const int64_t grp = t / per, r = t - grp * per;
    const int64_t g0 = grp * kGroup;
    const int64_t gsz = tiles_t - g0 < kGroup ? tiles_t - g0 : kGroup;
    tt = g0 + r % gsz;
    tw = r / gsz;
}

// Named barrier 1 over the 16 epilogue warps (barrier 0 is __syncthreads).  Every epilogue
// warp reaches each of these at the same point of the same loop: a wait that fails is voted
// on with epi_all() first, so either all epilogue warps go on or all unwind together.
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kEpiWarps * 32)
        : "memory");
    return r != 0;
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

template <bool DEBUG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;   // one per pair of TMEM buffers
    uint64_t* drain = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    __shared__ float epi_sa[kEpiWarps][32];    // per epilogue warp: the tile's s_a of its columns
    __shared__ float epi_bias[kEpiWarps][32];  // per epilogue thread: the bias of its row

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_t = (args.M + kTileT - 1) / kTileT;
    const int64_t tiles_w = (args.N + kTileW - 1) / kTileW;
    const int64_t ntiles = tiles_t * tiles_w;
    const int64_t first = blockIdx.x;
    // the host keeps ntiles * K/64 below 2^31, so the stage counters below fit 32 bits
    const uint32_t my_tiles = ntiles > first ? static_cast<uint32_t>((ntiles - 1 - first) / gridDim.x + 1) : 0u;
    const uint32_t nb = static_cast<uint32_t>(args.K / kBlock);
    const uint32_t spt = (nb + 1) / 2;         // stages per tile
    const uint32_t total = my_tiles * spt;     // stages of this CTA, counted across its tiles
    const WaitCtl ctl{abort_flag, args.status, args.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 2);  // the producer and one epilogue thread
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&tfull[i], 2);  // one commit per block slot
        for (int i = 0; i < kIssuers; ++i) mbar_init(&drain[i], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (!DEBUG) {
        for (int i = threadIdx.x; i < kZeroBytes / 16; i += kThreads)
            reinterpret_cast<uint4*>(smem + kOffZero)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Launched as a programmatic dependent of the previous kernel in the stream (normally the
    // pre-pass that wrote the operand records): the set-up above overlaps its tail, and no
    // global memory is touched before it has completed.
    griddep_wait();

    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 0) {
            // -------------------------------------------------------- producer
            if (lane == 0) {
                uint32_t j = 0, issued = 0;  // stage counter; stages whose copies were issued
                bool ok = true;
                for (uint32_t i = 0; ok && i < my_tiles; ++i) {
                    int64_t tt, tw;
                    tile_at(first + static_cast<int64_t>(i) * gridDim.x, tiles_t, tiles_w, tt, tw);
                    const uint8_t* tsrc = args.trec + static_cast<int64_t>(tt) * nb * kTokRec;
                    const uint8_t* wsrc = args.wrec + static_cast<int64_t>(tw) * nb * kWRec;
                    for (uint32_t p = 0; p < spt; ++p, ++j) {
                        const int s = static_cast<int>(j % kStages);
                        const uint32_t k = j / kStages;
                        if (k > 0 && !mbar_wait(&empty[s], (k - 1) & 1, ctl)) {
                            ok = false;
                            break;
                        }
                        const uint32_t b0 = 2 * p, cnt = nb - b0 < 2 ? 1u : 2u;
                        uint8_t* st = smem + s * kStageBytes;
                        mbar_arrive_expect_tx(&full[s], cnt * (kTokRec + kWRec));
                        bulk_load(st, tsrc + static_cast<int64_t>(b0) * kTokRec, cnt * kTokRec, &full[s]);
                        bulk_load(st + kStageTok, wsrc + static_cast<int64_t>(b0) * kWRec, cnt * kWRec, &full[s]);
                        issued = j + 1;
                    }
                }
                if (*abort_flag) {
                    // let every copy already issued land before the CTA exits
                    for (uint32_t q = (issued > kStages ? issued - kStages : 0); q < issued; ++q)
                        drain_wait(&full[q % kStages], (q / kStages) & 1, 100000000ull);
                }
            }
        } else {
            // -------------------------------------------------------- MMA issue (warps 1-3)
            const int iw = warp - 1;
            constexpr uint32_t idesc = idesc_e4m3_f32(kTileW, kTileT);
            // Descriptors of stage 0, slot 0; a record at byte offset o adds o >> 4 to the
            // start-address field, and a K offset of 32 bytes adds 2.  The field never
            // overflows: every shared-memory address is below 2^18.  The zero-point operands
            // take K 8..15 from the zero block, one leading byte offset away, which shrinks
            // as the start address grows.
            const uint32_t zr = smem_u32(smem + kOffZero);
            const uint32_t t0a = smem_u32(smem), w0a = smem_u32(smem + kStageTok);
            const uint64_t dT0 = smem_desc(t0a, 1024, kLayoutSw128);
            const uint64_t dW0 = smem_desc(w0a, 512, kLayoutSw64);
            const uint64_t dBx0 = smem_desc(t0a + kTokRx, 128, 0, zr - (t0a + kTokRx));
            const uint64_t dAx0 = smem_desc(w0a + kWZx, 128, 0, zr - (w0a + kWZx));
            // Work item i = 2 j + k is block slot k of stage j; warp 1 + (i % 3) issues it, so the
            // two blocks of a stage go out from two warps at once.  Stage j accumulates in the
            // TMEM buffer pair j % 2 (slot k in buffer 2 (j % 2) + k).
            for (uint32_t i = iw; i < 2 * total; i += kIssuers) {
                const uint32_t j = i >> 1, k = i & 1u;
                const int s = static_cast<int>(j % kStages);
                const uint32_t pair = j & 1u;
                const uint32_t b0 = 2 * (j % spt), cnt = nb - b0 < 2 ? 1u : 2u;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (j / kStages) & 1, ctl))) break;
                tc_fence_after();
                if (elect_one()) {
                    if (k < cnt) {
                        const uint32_t d = tmem_base + (2 * pair + k) * kTileT;
                        const uint64_t ot = static_cast<uint64_t>((s * kStageBytes + static_cast<int>(k) * kTokRec) >> 4);
                        const uint64_t ow = static_cast<uint64_t>((s * kStageBytes + static_cast<int>(k) * kWRec) >> 4);
                        const uint64_t dT = dT0 + ot, dW = dW0 + ow;
                        // q x hi plane (K 0..31, 32..63), then q x lo plane
                        mma_f8f6f4(d, dW, dT, idesc, 0u);
                        mma_f8f6f4(d, dW + 2, dT + 2, idesc, 1u);
                        mma_f8f6f4(d, dW, dT + 4, idesc, 1u);
                        mma_f8f6f4(d, dW + 2, dT + 6, idesc, 1u);
                        // zero-point term: {-z, -z} x {rh/8, rl/512}
                        if (!DEBUG) mma_f16(d, dAx0 + ow - (ow << 16), dBx0 + ot - (ot << 16), idesc, 1u);
                    }
                    // a stage's accumulators are complete once both slots' commits have arrived
                    // (a slot without a block commits at once)
                    mma_commit(&tfull[pair]);
                }
                __syncwarp();
            }
            // this warp's MMAs complete before the CTA releases TMEM
            if (elect_one()) mma_commit(&drain[iw]);
            __syncwarp();
            drain_wait(&drain[iw], 0, 100000000ull);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        regs_inc<kRegsHigh>();
        const int q = warp & 3, h = (warp - 4) >> 2;  // TMEM lane quarter, column quarter
        const int row = q * 32 + lane;                // this thread's weight row in the tile
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 32);
        // the TMEM buffers start free: release the first two stages
        if (warp == 4 && lane == 0)
            for (uint32_t q0 = 0; q0 < 2 && q0 < total; ++q0) mbar_arrive(&full[q0]);
        uint32_t j = 0;  // stage counter of this CTA
        bool ok = true;
        for (uint32_t i = 0; ok && i < my_tiles; ++i) {
            int64_t tt, tw;
            tile_at(first + static_cast<int64_t>(i) * gridDim.x, tiles_t, tiles_w, tt, tw);
            const int64_t mt0 = tt * kTileT + h * 32;  // first token column of this warp
            const int64_t n = tw * kTileW + row;       // this thread's weight row
            // this row's scales, block after block; each stage's pair is loaded one stage ahead
            const float* sct = DEBUG ? nullptr : args.sc + static_cast<int64_t>(tw) * nb * kTileW + row;
            if (!DEBUG) {
                // this tile's s_a and bias, loaded now into the warp's own slots so the stores at
                // the end of the tile neither wait on memory nor hold registers through the loop
                epi_sa[warp - 4][lane] = mt0 + lane < args.M ? __ldg(args.s_a + mt0 + lane) : 0.0f;
                epi_bias[warp - 4][lane] = (args.bias && n < args.N) ? __ldg(args.bias + n) : 0.0f;
            }
            float ns0 = 0.0f, ns1 = 0.0f;
            if (!DEBUG) {
                ns0 = __ldg(sct);
                if (nb > 1) ns1 = __ldg(sct + kTileW);
            }
            float y[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] = 0.0f;
            for (uint32_t p = 0; p < spt; ++p, ++j) {
                const int s = static_cast<int>(j % kStages);
                const bool two = 2 * p + 1 < nb;
                const float s0 = ns0, s1 = ns1;
                if (!DEBUG && p + 1 < spt) {
                    ns0 = __ldg(sct + (2 * p + 2) * kTileW);
                    ns1 = 2 * p + 3 < nb ? __ldg(sct + (2 * p + 3) * kTileW) : 0.0f;
                }
                const uint32_t pair = j & 1u, b0 = 2 * pair, b1 = b0 + 1;
                if (!epi_all(mbar_wait(&tfull[pair], (j >> 1) & 1, ctl))) {
                    ok = false;
                    break;
                }
                // the stage's MMAs are complete: its operands are no longer needed
                if (warp == 4 && lane == 0) mbar_arrive(&empty[s]);
                tc_fence_after();
                uint32_t v[64];
                tmem_ld_32x32b_x16(tl + b0 * kTileT, v);
                tmem_ld_32x32b_x16(tl + b0 * kTileT + 16, v + 16);
                if (two) {
                    tmem_ld_32x32b_x16(tl + b1 * kTileT, v + 32);
                    tmem_ld_32x32b_x16(tl + b1 * kTileT + 16, v + 48);
                }
                tmem_wait_ld();
                // the accumulators are in registers: the buffers are free for the stage two later
                // (the epilogue warps meet on a named barrier, then one thread arrives: sixteen
                // arrivals on one mbarrier word would serialise)
                tc_fence_before();
                epi_bar_sync();
                if (warp == 4 && lane == 0 && j + 2 < total) mbar_arrive(&full[(j + 2) % kStages]);
                if (DEBUG) {
                    if (n < args.N) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (e == 1 && !two) break;
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const int64_t m = mt0 + c;
                                if (m < args.M)
                                    args.acc[(m * args.N + n) * nb + 2 * p + e] =
                                        static_cast<int32_t>(__uint_as_float(v[32 * e + c]) * 512.0f);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) y[c] = fmaf(s0, __uint_as_float(v[c]), y[c]);
                    if (two) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) y[c] = fmaf(s1, __uint_as_float(v[32 + c]), y[c]);
                    }
                }
            }
            if (!ok) break;
            if (!DEBUG) __syncwarp();  // every lane: the slots were written by other lanes of the warp
            if (!DEBUG && n < args.N) {
                const float bn = epi_bias[warp - 4][lane];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int64_t m = mt0 + c;
                    if (m < args.M) store_y(args.out, m * args.N + n, fmaf(epi_sa[warp - 4][c], y[c], bn));
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- 256-token tiles
// The large-M variant.  One MMA covers 128 weights x 256 tokens (N = 256), so the SM issues
// half as many tcgen05.mma instructions per unit of work as with 128-token tiles (the MMA
// issue rate of an SM, one instruction per ~50-90 cycles, is what bounds the 128-token
// kernel).  Two TMEM buffers of 256 columns; one block per shared-memory stage, filled by two
// bulk copies (a 256-token record and a weight record).  Roles, barriers and bounded waits
// follow gemm_kernel; an epilogue thread owns one weight row and 64 token columns, drained
// 32 at a time.
namespace wide {
constexpr int kTN = 256;
constexpr int kStages = 4;
constexpr int kNBuf = 2;
constexpr int kIssuers = 2;  // warps 1-2; each owns every other stage (warp 3 idles)
constexpr int kTok = 144 * kTN;                 // token record of one block
constexpr int kStageBytes = kTok + kWRec;
constexpr int kOffZero = kStages * kStageBytes;
constexpr int kOffBar = kOffZero + kZeroBytes;
constexpr int kNumBars = 2 * kStages + kNBuf + kIssuers;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kTok % 1024 == 0 && kStageBytes % 1024 == 0, "swizzled operand tiles must stay 1024-aligned");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kNBuf * kTN == 512, "TMEM allocation");
static_assert(kNBuf <= kStages, "a stage barrier carries a buffer release only after its previous phase");
static_assert(kZeroBytes >= kTN * 16, "zero half of the token-side zero-point operand");
// block g goes to issuer g % kIssuers: the same warp waits every phase of a stage, in order
static_assert(kStages % kIssuers == 0 && kIssuers <= 3, "each stage must have one issuer warp at every phase");
}  // namespace wide

// DEBUG: no zero-point MMA and no register split; the epilogue stores each block's exact
// integer accumulator (acc * 2^-9 in TMEM, times 512) instead of folding it into y.
template <bool DEBUG>
__global__ void __launch_bounds__(kThreads, 1) gemm_wide_kernel(const GemmArgs args) {
    namespace W = wide;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + W::kOffBar);
    uint64_t* empty = full + W::kStages;
    uint64_t* tfull = empty + W::kStages;
    uint64_t* drain = tfull + W::kNBuf;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + W::kOffMisc);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_t = (args.M + W::kTN - 1) / W::kTN;
    const int64_t tiles_w = (args.N + kTileW - 1) / kTileW;
    const int64_t ntiles = tiles_t * tiles_w;
    const int64_t first = blockIdx.x;
    // the host keeps ntiles * K/64 below 2^31, so the block counters below fit 32 bits
    const uint32_t my_tiles = ntiles > first ? static_cast<uint32_t>((ntiles - 1 - first) / gridDim.x + 1) : 0u;
    const uint32_t nb = static_cast<uint32_t>(args.K / kBlock);
    const uint32_t total = my_tiles * nb;  // blocks of this CTA, counted across its tiles
    const WaitCtl ctl{abort_flag, args.status, args.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < W::kStages; ++s) {
            mbar_init(&full[s], 2);  // the producer and one epilogue thread
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < W::kNBuf; ++i) mbar_init(&tfull[i], 1);
        for (int i = 0; i < W::kIssuers; ++i) mbar_init(&drain[i], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (!DEBUG) {
        for (int i = threadIdx.x; i < kZeroBytes / 16; i += kThreads)
            reinterpret_cast<uint4*>(smem + W::kOffZero)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();

    if (warp < 4) {
        if (!DEBUG) regs_dec<kRegsLow>();
        if (warp == 0) {
            // -------------------------------------------------------- producer
            if (lane == 0) {
                uint32_t g = 0, issued = 0;
                bool ok = true;
                for (uint32_t i = 0; ok && i < my_tiles; ++i) {
                    int64_t tt, tw;
                    tile_at(first + static_cast<int64_t>(i) * gridDim.x, tiles_t, tiles_w, tt, tw);
                    const uint8_t* tsrc = args.trec + static_cast<int64_t>(tt) * nb * W::kTok;
                    const uint8_t* wsrc = args.wrec + static_cast<int64_t>(tw) * nb * kWRec;
                    for (uint32_t b = 0; b < nb; ++b, ++g) {
                        const int s = static_cast<int>(g % W::kStages);
                        const uint32_t k = g / W::kStages;
                        if (k > 0 && !mbar_wait(&empty[s], (k - 1) & 1, ctl)) {
                            ok = false;
                            break;
                        }
                        uint8_t* st = smem + s * W::kStageBytes;
                        mbar_arrive_expect_tx(&full[s], W::kTok + kWRec);
                        bulk_load(st, tsrc + static_cast<int64_t>(b) * W::kTok, W::kTok, &full[s]);
                        bulk_load(st + W::kTok, wsrc + static_cast<int64_t>(b) * kWRec, kWRec, &full[s]);
                        issued = g + 1;
                    }
                }
                if (*abort_flag) {
                    for (uint32_t q = (issued > W::kStages ? issued - W::kStages : 0); q < issued; ++q)
                        drain_wait(&full[q % W::kStages], (q / W::kStages) & 1, 100000000ull);
                }
            }
        } else if (warp <= W::kIssuers) {
            // -------------------------------------------------------- MMA issue (warps 1-2)
            const int iw = warp - 1;
            constexpr uint32_t idesc = idesc_e4m3_f32(kTileW, W::kTN);
            const uint32_t zr = smem_u32(smem + W::kOffZero);
            const uint32_t t0a = smem_u32(smem), w0a = smem_u32(smem + W::kTok);
            const uint64_t dT0 = smem_desc(t0a, 1024, kLayoutSw128);
            const uint64_t dW0 = smem_desc(w0a, 512, kLayoutSw64);
            const uint64_t dBx0 = smem_desc(t0a + 128 * W::kTN, 128, 0, zr - (t0a + 128 * W::kTN));
            const uint64_t dAx0 = smem_desc(w0a + kWZx, 128, 0, zr - (w0a + kWZx));
            for (uint32_t g = iw; g < total; g += W::kIssuers) {
                const int s = static_cast<int>(g % W::kStages);
                const uint32_t buf = g & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (g / W::kStages) & 1, ctl))) break;
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t d = tmem_base + buf * W::kTN;
                    const uint64_t o = static_cast<uint64_t>((s * W::kStageBytes) >> 4);
                    const uint64_t dT = dT0 + o, dW = dW0 + o;
                    mma_f8f6f4(d, dW, dT, idesc, 0u);
                    mma_f8f6f4(d, dW + 2, dT + 2, idesc, 1u);
                    mma_f8f6f4(d, dW, dT + 4, idesc, 1u);
                    mma_f8f6f4(d, dW + 2, dT + 6, idesc, 1u);
                    if (!DEBUG) mma_f16(d, dAx0 + o - (o << 16), dBx0 + o - (o << 16), idesc, 1u);
                    mma_commit(&tfull[buf]);
                }
                __syncwarp();
            }
            if (elect_one()) mma_commit(&drain[iw]);
            __syncwarp();
            drain_wait(&drain[iw], 0, 100000000ull);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        if (!DEBUG) regs_inc<kRegsHigh>();
        const int q = warp & 3, h = (warp - 4) >> 2;  // TMEM lane quarter, 64-column quarter
        const int row = q * 32 + lane;
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 64);
        if (warp == 4 && lane == 0)
            for (uint32_t q0 = 0; q0 < W::kNBuf && q0 < total; ++q0) mbar_arrive(&full[q0]);
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t i = 0; ok && i < my_tiles; ++i) {
            int64_t tt, tw;
            tile_at(first + static_cast<int64_t>(i) * gridDim.x, tiles_t, tiles_w, tt, tw);
            const int64_t mt0 = tt * W::kTN + h * 64;
            const int64_t n = tw * kTileW + row;
            const float* sct = DEBUG ? nullptr : args.sc + static_cast<int64_t>(tw) * nb * kTileW + row;
            float ns = DEBUG ? 0.0f : __ldg(sct);
            float y[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) y[c] = 0.0f;
            // debug: this block's exact accumulators of 32 token columns starting at c0
            auto store_acc = [&](const uint32_t (&v)[32], int c0, uint32_t b) {
                if (n >= args.N) return;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int64_t m = mt0 + c0 + c;
                    if (m < args.M)
                        args.acc[(m * args.N + n) * nb + b] = static_cast<int32_t>(__uint_as_float(v[c]) * 512.0f);
                }
            };
            for (uint32_t b = 0; b < nb; ++b, ++g) {
                const float sb = ns;
                if (!DEBUG && b + 1 < nb) ns = __ldg(sct + (b + 1) * kTileW);
                const uint32_t buf = g & 1u;
                if (!epi_all(mbar_wait(&tfull[buf], (g >> 1) & 1, ctl))) {
                    ok = false;
                    break;
                }
                if (warp == 4 && lane == 0) mbar_arrive(&empty[g % W::kStages]);
                tc_fence_after();
                const uint32_t tb = tl + buf * W::kTN;
                uint32_t v[32];
                tmem_ld_32x32b_x16(tb, v);
                tmem_ld_32x32b_x16(tb + 16, v + 16);
                tmem_wait_ld();
                if (DEBUG) {
                    store_acc(v, 0, b);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) y[c] = fmaf(sb, __uint_as_float(v[c]), y[c]);
                }
                tmem_ld_32x32b_x16(tb + 32, v);
                tmem_ld_32x32b_x16(tb + 48, v + 16);
                tmem_wait_ld();
                // the accumulator is in registers: the buffer is free for block g + 2
                tc_fence_before();
                epi_bar_sync();
                if (warp == 4 && lane == 0 && g + W::kNBuf < total) mbar_arrive(&full[(g + W::kNBuf) % W::kStages]);
                if (DEBUG) {
                    store_acc(v, 32, b);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) y[32 + c] = fmaf(sb, __uint_as_float(v[c]), y[32 + c]);
                }
            }
            if (!ok) break;
            if (!DEBUG && n < args.N) {
                const float bn = args.bias ? args.bias[n] : 0.0f;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const int64_t m = mt0 + c;
                    if (m < args.M) store_y(args.out, m * args.N + n, fmaf(args.s_a[m], y[c], bn));
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
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

template <typename Kernel>
cudaError_t launch(Kernel kernel, int smem_bytes, bool* attr_done, int64_t tiles, const GemmArgs& a, int num_sms,
                   cudaStream_t s) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const int64_t grid = tiles < num_sms ? tiles : num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, bool debug, int num_sms, cudaStream_t s) {
    static bool attr_done[4][64] = {};
    if (num_sms < 1) return cudaErrorInvalidValue;
    const int64_t tiles_w = (a.N + kTileW - 1) / kTileW;
    if (a.tw == wide::kTN) {
        const int64_t tiles = ((a.M + wide::kTN - 1) / wide::kTN) * tiles_w;
        return debug ? launch(gemm_wide_kernel<true>, wide::kSmemBytes, attr_done[3], tiles, a, num_sms, s)
                     : launch(gemm_wide_kernel<false>, wide::kSmemBytes, attr_done[2], tiles, a, num_sms, s);
    }
    if (a.tw != kTileT) return cudaErrorInvalidValue;
    const int64_t tiles = ((a.M + kTileT - 1) / kTileT) * tiles_w;
    return debug ? launch(gemm_kernel<true>, kSmemBytes, attr_done[1], tiles, a, num_sms, s)
                 : launch(gemm_kernel<false>, kSmemBytes, attr_done[0], tiles, a, num_sms, s);
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace w4a8
