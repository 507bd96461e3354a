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
// (producer arrival + transaction bytes) and every epilogue warp has released the two TMEM
// buffers the stage overwrites (one arrival per epilogue warp), so an issuer waits once per
// block.  The epilogue drains a stage's two blocks together (four TMEM loads in flight per
// wait), releases their buffers as soon as the accumulators are in its registers, then folds
// them into y; it frees a stage once its accumulators are complete.  The epilogue warps wait
// and release each on their own: a rendezvous of all sixteen per stage (a vote on the wait,
// a named barrier before one release) cost the skew between the warps at every stage
// (measured on the 7B-class contraction: 4-7% of its time).  Every wait is bounded (WaitCtl); a
// thread that gives up raises the CTA's abort flag, so every role stops waiting and unwinds.
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "operand_codes.cuh"
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

// The same tile in 32-bit arithmetic, for the packed kernel, whose producer thread computed it
// on its critical path (three 64-bit divisions, a long software sequence, per copy).  The host
// keeps the tile count below 2^31 and tiles_w is at most 2^24.  The record kernels keep the
// 64-bit form: measured, the 32-bit one made the 256-token kernel about 4% slower.
__device__ __forceinline__ void tile_at32(int64_t t, int64_t tiles_t, int64_t tiles_w, int64_t& tt, int64_t& tw) {
    const uint32_t t32 = static_cast<uint32_t>(t), tt32 = static_cast<uint32_t>(tiles_t);
    const uint32_t per = static_cast<uint32_t>(kGroup) * static_cast<uint32_t>(tiles_w);
    const uint32_t grp = t32 / per, r = t32 - grp * per;
    const uint32_t g0 = grp * static_cast<uint32_t>(kGroup);
    const uint32_t gsz = tt32 - g0 < static_cast<uint32_t>(kGroup) ? tt32 - g0 : static_cast<uint32_t>(kGroup);
    const uint32_t q = r / gsz;
    tt = g0 + (r - q * gsz);
    tw = q;
}

// y[c] = fma(s, v[c], y[c]) for c < C, two columns per instruction (fma.rn.f32x2: the same
// single-rounding fp32 fma per element as fmaf, so the sums are unchanged bit for bit).
template <int C>
__device__ __forceinline__ void fma_cols(float* y, float s, const uint32_t* v) {
    uint64_t ss;
    asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(s));
#pragma unroll
    for (int c = 0; c < C; c += 2) {
        uint64_t yy, vv;
        asm("mov.b64 %0, {%1, %2};" : "=l"(yy) : "f"(y[c]), "f"(y[c + 1]));
        asm("mov.b64 %0, {%1, %2};" : "=l"(vv) : "r"(v[c]), "r"(v[c + 1]));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(yy) : "l"(ss), "l"(vv));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(y[c]), "=f"(y[c + 1]) : "l"(yy));
    }
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

// KS: CTAs (a cluster) per tile, each contracting 1/KS of K (1, or 2 for the K split).
template <bool DEBUG, int KS>
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
    // With a K split, a cluster of ks CTAs shares each tile (the host launches exactly one tile
    // per cluster): CTA kr of the cluster contracts blocks kb0 .. kb0 + nbl - 1 of K.
    constexpr uint32_t ks = static_cast<uint32_t>(KS);
    static_assert(KS == 1 || (KS == 2 && !DEBUG), "the K split is a two-CTA cluster, outside the debug form");
    const uint32_t kr = ks > 1 ? cluster_ctarank() : 0u;
    const int64_t first = blockIdx.x / ks;
    const uint32_t stride = gridDim.x / ks;
    // the host keeps ntiles * K/64 below 2^31, so the stage counters below fit 32 bits
    const uint32_t my_tiles = ntiles > first ? static_cast<uint32_t>((ntiles - 1 - first) / stride + 1) : 0u;
    const uint32_t nb = static_cast<uint32_t>(args.K / kBlock);  // blocks of a tile's records
    const uint32_t nbl = nb / ks, kb0 = kr * nbl;
    const uint32_t spt = (nbl + 1) / 2;        // stages per tile
    const uint32_t total = my_tiles * spt;     // stages of this CTA, counted across its tiles
    const WaitCtl ctl{abort_flag, args.status, args.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1 + kEpiWarps);  // the producer and every epilogue warp
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
                    tile_at(first + static_cast<int64_t>(i) * stride, tiles_t, tiles_w, tt, tw);
                    // this CTA's first block of the tile's records
                    const uint8_t* tsrc = args.trec + (static_cast<int64_t>(tt) * nb + kb0) * kTokRec;
                    const uint8_t* wsrc = args.wrec + (static_cast<int64_t>(tw) * nb + kb0) * kWRec;
                    // the tile's weight scales into L2 ahead of the epilogue's loads
                    if (!DEBUG)
                        bulk_prefetch_l2(args.sc + (static_cast<int64_t>(tw) * nb + kb0) * kTileW, nbl * kTileW * 4u);
                    for (uint32_t p = 0; p < spt; ++p, ++j) {
                        const int s = static_cast<int>(j % kStages);
                        const uint32_t k = j / kStages;
                        if (k > 0 && !mbar_wait(&empty[s], (k - 1) & 1, ctl)) {
                            ok = false;
                            break;
                        }
                        const uint32_t b0 = 2 * p, cnt = nbl - b0 < 2 ? 1u : 2u;
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
                const uint32_t b0 = 2 * (j % spt), cnt = nbl - b0 < 2 ? 1u : 2u;
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
        if (ks > 1) {  // the epilogue's two cluster barriers of the K split
            cluster_sync_all();
            cluster_sync_all();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        regs_inc<kRegsHigh>();
        const int q = warp & 3, h = (warp - 4) >> 2;  // TMEM lane quarter, column quarter
        const int row = q * 32 + lane;                // this thread's weight row in the tile
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 32);
        // the TMEM buffers start free: release the first two stages
        if (lane == 0)
            for (uint32_t q0 = 0; q0 < 2 && q0 < total; ++q0) mbar_arrive(&full[q0]);
        uint32_t j = 0;  // stage counter of this CTA
        bool ok = true;
        // this thread's sums and output position, kept past the tile loop for the K split
        float y[32];
        int64_t mt0 = 0, n = 0;
        for (uint32_t i = 0; ok && i < my_tiles; ++i) {
            int64_t tt, tw;
            tile_at(first + static_cast<int64_t>(i) * stride, tiles_t, tiles_w, tt, tw);
            mt0 = tt * kTileT + h * 32;  // first token column of this warp
            n = tw * kTileW + row;       // this thread's weight row
            // this row's scales, block after block (from this CTA's first block of K); each
            // stage's pair is loaded one stage ahead
            const float* sct = DEBUG ? nullptr : args.sc + (static_cast<int64_t>(tw) * nb + kb0) * kTileW + row;
            if (!DEBUG) {
                // this tile's s_a and bias, loaded now into the warp's own slots so the stores at
                // the end of the tile neither wait on memory nor hold registers through the loop
                epi_sa[warp - 4][lane] = mt0 + lane < args.M ? __ldcg(args.s_a + mt0 + lane) : 0.0f;
                epi_bias[warp - 4][lane] = (args.bias && n < args.N) ? __ldg(args.bias + n) : 0.0f;
            }
            float ns0 = 0.0f, ns1 = 0.0f;
            if (!DEBUG) {
                ns0 = __ldcg(sct);
                if (nbl > 1) ns1 = __ldcg(sct + kTileW);
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] = 0.0f;
            for (uint32_t p = 0; p < spt; ++p, ++j) {
                const int s = static_cast<int>(j % kStages);
                const bool two = 2 * p + 1 < nbl;
                const float s0 = ns0, s1 = ns1;
                if (!DEBUG && p + 1 < spt) {
                    ns0 = __ldcg(sct + (2 * p + 2) * kTileW);
                    ns1 = 2 * p + 3 < nbl ? __ldcg(sct + (2 * p + 3) * kTileW) : 0.0f;
                }
                const uint32_t pair = j & 1u, b0 = 2 * pair, b1 = b0 + 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&tfull[pair], (j >> 1) & 1, ctl))) {
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
                // this warp's accumulators are in registers: its part of the buffers is free for the
                // stage two later (the stage barrier completes once every epilogue warp has arrived)
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && j + 2 < total) mbar_arrive(&full[(j + 2) % kStages]);
                if (DEBUG) {
                    if (n < args.N) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (e == 1 && !two) break;
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const int64_t m = mt0 + c;
                                if (m < args.M)
                                    args.acc[(m * args.N + n) * nb + kb0 + 2 * p + e] =
                                        static_cast<int32_t>(__uint_as_float(v[32 * e + c]) * 512.0f);
                            }
                        }
                    }
                } else {
                    fma_cols<32>(y, s0, v);
                    if (two) {
                        fma_cols<32>(y, s1, v + 32);
                    }
                }
            }
            if (!ok) break;
            if (!DEBUG) __syncwarp();  // every lane: the slots were written by other lanes of the warp
            if (!DEBUG && ks == 1 && n < args.N) {
                const float bn = epi_bias[warp - 4][lane];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int64_t m = mt0 + c;
                    if (m < args.M) store_y(args.out, m * args.N + n, fmaf(epi_sa[warp - 4][c], y[c], bn));
                }
            }
        }
        if (ks > 1) {
            // K split (one tile per cluster): the second CTA leaves its partial sums in its own
            // stage memory, idle now that its MMAs are complete; the first adds them to its own,
            // in that order, and stores the tile.  Every thread of both CTAs takes part in both
            // cluster barriers (the other warps at the end of their roles), also after a wait gave
            // up (the outputs are then undefined; the status word says so): the second CTA's memory
            // stays until the first has read it.
            float* part = reinterpret_cast<float*>(smem) + (warp - 4) * 32 * 32 + lane;  // [warp][c][lane]
            if (kr == 1) {
#pragma unroll
                for (int c = 0; c < 32; ++c) part[c * 32] = y[c];
            }
            cluster_sync_all();
            if (kr == 0 && n < args.N) {
#pragma unroll
                for (int c = 0; c < 32; ++c) y[c] += ld_shared_cluster_f32(part + c * 32, 1);
                const float bn = epi_bias[warp - 4][lane];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int64_t m = mt0 + c;
                    if (m < args.M) store_y(args.out, m * args.N + n, fmaf(epi_sa[warp - 4][c], y[c], bn));
                }
            }
            cluster_sync_all();
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
// The large-M variant.  One MMA covers 128 weights x 256 tokens (N = 256), so per unit of work
// the SM issues half as many tcgen05.mma instructions, reads the weight operand from shared
// memory half as often and waits on half as many accumulator hand-offs as with 128-token tiles
// (measured at M = 8192: the 128-token kernel takes 25% longer).  Two TMEM buffers of 256
// columns; one block per shared-memory stage, filled by two bulk copies (a 256-token record and
// a weight record).  Roles, barriers and bounded waits follow gemm_kernel; an epilogue thread
// owns one weight row and 64 token columns, drained 32 at a time.
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
            mbar_init(&full[s], 1 + kEpiWarps);  // the producer and every epilogue warp
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
                    // the tile's weight scales (nb x 128 floats, contiguous) into L2 now, a few
                    // blocks before the epilogue reads the first of them: a scale load that misses
                    // L2 holds up the drain of its block's accumulator, and with it the MMAs that
                    // wait for that TMEM buffer
                    if (!DEBUG) bulk_prefetch_l2(args.sc + static_cast<int64_t>(tw) * nb * kTileW, nb * kTileW * 4u);
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
        if (lane == 0)
            for (uint32_t q0 = 0; q0 < W::kNBuf && q0 < total; ++q0) mbar_arrive(&full[q0]);
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t i = 0; ok && i < my_tiles; ++i) {
            int64_t tt, tw;
            tile_at(first + static_cast<int64_t>(i) * gridDim.x, tiles_t, tiles_w, tt, tw);
            const int64_t mt0 = tt * W::kTN + h * 64;
            const int64_t n = tw * kTileW + row;
            const float* sct = DEBUG ? nullptr : args.sc + static_cast<int64_t>(tw) * nb * kTileW + row;
            float ns = DEBUG ? 0.0f : __ldcg(sct);
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
                if (!DEBUG && b + 1 < nb) ns = __ldcg(sct + (b + 1) * kTileW);
                const uint32_t buf = g & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], (g >> 1) & 1, ctl))) {
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
                    fma_cols<32>(y, sb, v);
                }
                tmem_ld_32x32b_x16(tb + 32, v);
                tmem_ld_32x32b_x16(tb + 48, v + 16);
                tmem_wait_ld();
                // this warp's accumulators are in registers: its part of the buffer is free for
                // block g + 2 (the stage barrier completes once every epilogue warp has arrived)
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && g + W::kNBuf < total) mbar_arrive(&full[(g + W::kNBuf) % W::kStages]);
                if (DEBUG) {
                    store_acc(v, 32, b);
                } else {
                    fma_cols<32>(y + 32, sb, v);
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

// ---------------------------------------------------------------- 128-token tiles, packed weights
// The contraction of gemm_kernel, reading the caller's packed weights (section 4 step 2: each
// task reuses one staged B tile); it serves w4a8_linear_act.  The producer stages each stage's
// 2 x 32 packed bytes of the tile's 128 weight rows with one tiled TMA load (64-byte swizzle,
// rows past N filled with zeros), and the epilogue warps, between their drains, expand them in
// shared memory to the e4m3 operand and write the {-z_w, -z_w} rows of the zero-point MMA --
// the same bytes the weight job writes into a weight record, so the MMAs, and every output,
// are those of gemm_kernel bit for bit.  The epilogue reads 512 s_w from s_w itself.  No
// weight record is written to or read from device memory.
// Measured alone after an L2 flush, it takes 20.5 us on the pp512 linear (512 x 1024 -> 3072)
// against 14.3 us for gemm_kernel, and 59 / 88 us against 33 / 41 us on the M = 512 linears
// 2048 -> 6144 and 6144 -> 2048: while the expanding warps load and store shared memory, the
// tensor cores' stages stretch.  So the one-call entry points keep the weight records; this
// kernel is the form that needs neither a workspace nor expanded weights in memory.  Every
// epilogue warp arrives on the stage barrier itself, for its part of the expanded operand and
// for its part of the released TMEM buffers (a named barrier of all sixteen before one arrival
// cost 10-24% of this kernel's time).
//
// The packed weights have a ring of kPkSlots slots of their own, so their loads run ahead of the
// operand stages -- and, with `early` set (they do not depend on the previous kernel), start
// before the pre-pass has finished.  Operand stage s = j % kStages of stage j is expanded as soon
// as stage j - kStages has completed its MMAs, right after the epilogue has drained that stage's
// accumulators; the first kStages stages are expanded up front.  Each tile also prefetches the
// next tile's s_w / z_w rows into L2.
//
// Warp roles (20 warps, register split as in gemm_kernel):
//   warp 0       producer: per stage one TMA load (packed weights, into the ring) and one bulk
//                copy (token records of the stage's two blocks)
//   warps 1-3    MMA issue, as in gemm_kernel
//   warps 4-19   epilogue and expansion: thread t expands the 16 packed bytes (t & 3) of weight
//                row t >> 2 of a stage; the drain is gemm_kernel's
// Barriers: per operand stage full (token records landed, the operand expanded, the two TMEM
// buffers released) and empty (the stage's MMAs done: its operand buffers free); per ring slot
// wfull (the packed weights landed).  A ring slot is reloaded only after the stage that last
// used it has completed its MMAs (its expansion came before that stage's full barrier), so it
// needs no barrier of its own for that.
namespace packed {
constexpr int kStages = 3;                        // operand stages (token records + expanded weights)
constexpr int kPkSlots = 6;                       // staged packed weights: a deeper ring of their own
constexpr int kPk = kTileW * 64;                  // 128 rows x 64 packed bytes (two blocks)
constexpr int kOffWop = 2 * kTokRec;              // the stage's two expanded weight records
constexpr int kStageBytes = kOffWop + 2 * kWRec;
constexpr int kOffPk = kStages * kStageBytes;
constexpr int kOffZero = kOffPk + kPkSlots * kPk;
constexpr int kOffBar = kOffZero + kZeroBytes;
constexpr int kNumBars = 2 * kStages + kPkSlots + 2 + kIssuers;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kOffWop == kStageTok && kStages == ::w4a8::kStages,
              "the issuers' descriptors and the TMEM release schedule follow gemm_kernel's stage layout");
static_assert(kStageBytes % 1024 == 0 && kOffPk % 1024 == 0 && kPk % 1024 == 0, "swizzled tiles must stay 1024-aligned");
static_assert(kSmemBytes + 2 * kEpiWarps * 32 * 4 <= 227 * 1024, "shared memory budget");
static_assert(kPkSlots >= kStages, "the weights of stage j + kStages go out while stage j's operands are in use");
static_assert(kEpiWarps * 32 == 4 * kTileW, "one expanding thread per 16 packed bytes of a stage");
}  // namespace packed

// Prefetch [p, p + bytes) into L2, one instruction per 128-byte line.
__device__ __forceinline__ void prefetch_l2_span(const void* p, int64_t bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(127);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes);
    for (uintptr_t a = a0; a < a1; a += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// This CTA's share of the work: its tiles are first, first + stride, ...; of each tile's K it
// contracts blocks kb0 .. kb0 + nbl - 1 (all of them unless K is split over a cluster).
struct KPart {
    uint32_t stride, kb0, nbl;
};

// A walk over the (tile, stage of the tile) pairs of a CTA's stages.
struct StageCursor {
    uint32_t i, p;
    int64_t tt, tw;
};

__device__ __forceinline__ void cursor_tile(StageCursor& c, uint32_t my_tiles, int64_t first, int64_t tiles_t,
                                            int64_t tiles_w, uint32_t stride) {
    if (c.i < my_tiles) tile_at32(first + static_cast<int64_t>(c.i) * stride, tiles_t, tiles_w, c.tt, c.tw);
}

__device__ __forceinline__ void cursor_next(StageCursor& c, uint32_t spt, uint32_t my_tiles, int64_t first,
                                            int64_t tiles_t, int64_t tiles_w, uint32_t stride) {
    if (++c.p == spt) {
        c.p = 0;
        ++c.i;
        cursor_tile(c, my_tiles, first, tiles_t, tiles_w, stride);
    }
}

// The producer's TMA load of stage `wnext`'s packed weights (the stage `cw` points at) into its
// ring slot; advances both.
__device__ __forceinline__ void issue_weights(const GemmArgs& args, uint8_t* smem, uint64_t* wfull, StageCursor& cw,
                                              uint32_t& wnext, uint32_t spt, uint32_t my_tiles, int64_t first,
                                              int64_t tiles_t, int64_t tiles_w, const KPart& kp) {
    namespace P = packed;
    uint64_t* bar = &wfull[wnext % P::kPkSlots];
    mbar_arrive_expect_tx(bar, P::kPk);
    // x: the stage's first packed byte of a row (32 per block), a multiple of 64 bytes
    tma_load_2d(smem + P::kOffPk + (wnext % P::kPkSlots) * P::kPk, &args.wmap, static_cast<int>(64 * cw.p + 32 * kp.kb0),
                static_cast<int>(cw.tw * kTileW), bar);
    ++wnext;
    cursor_next(cw, spt, my_tiles, first, tiles_t, tiles_w, kp.stride);
}

// 512 s_w[n, b] from the caller's fp16 scales (row pointer swr, null past N), 0 past the last
// block: the power of two undoes the 2^-9 of the e4m3 weight operand (exact).
__device__ __forceinline__ float weight_scale(const uint16_t* swr, uint32_t b, uint32_t nb) {
    return (swr && b < nb) ? 512.0f * __half2float(__ushort_as_half(__ldg(swr + b))) : 0.0f;
}

// Expansion of stage jj's packed weights into operand stage jj % kStages, by the 512 epilogue
// threads (thread et: the 16 packed bytes (et & 3) of weight row et >> 2).  Every epilogue
// thread calls it for every stage in order, once that operand stage is free; false if a wait
// gave up (all threads alike).  A plain function, not a lambda: nothing of it may live in local
// memory, which with the shared-memory carve-out has next to no L1 behind it.
template <bool DEBUG>
__device__ __forceinline__ bool expand_stage(const GemmArgs& args, uint8_t* smem, uint64_t* wfull, uint64_t* full,
                                             uint32_t jj, uint32_t spt, uint32_t nb, int64_t first, int64_t tiles_t,
                                             int64_t tiles_w, int et, const WaitCtl& ctl, const KPart& kp) {
    namespace P = packed;
    const int xr = et >> 2, xc = et & 3, xsw = (xr >> 1) & 3;
    const uint32_t ti = jj / spt, p = jj - ti * spt;
    int64_t tt, tw;
    tile_at32(first + static_cast<int64_t>(ti) * kp.stride, tiles_t, tiles_w, tt, tw);
    const int64_t n = tw * kTileW + xr;
    const uint32_t b = 2 * p + (xc >> 1);  // block of this CTA's part of K
    const bool live = b < kp.nbl;
    // the zero point first: its latency overlaps the wait
    const uint32_t zz =
        (!DEBUG && live && (xc & 1) == 0 && n < args.N) ? neg_zero_pair(__ldg(args.z_w + n * nb + kp.kb0 + b)) : 0u;
    if (!__all_sync(0xffffffffu, mbar_wait(&wfull[jj % P::kPkSlots], (jj / P::kPkSlots) & 1, ctl))) return false;
    if (live) {
        const uint4 w =
            *reinterpret_cast<const uint4*>(smem + P::kOffPk + (jj % P::kPkSlots) * P::kPk + xr * 64 + ((xc ^ xsw) << 4));
        uint4 lo, hi;
        expand8(w.x, lo.x, lo.y);
        expand8(w.y, lo.z, lo.w);
        expand8(w.z, hi.x, hi.y);
        expand8(w.w, hi.z, hi.w);
        uint8_t* rec = smem + (jj % P::kStages) * P::kStageBytes + P::kOffWop + (xc >> 1) * kWRec;
        const int e0 = 2 * (xc & 1);
        *reinterpret_cast<uint4*>(rec + xr * 64 + ((e0 ^ xsw) << 4)) = lo;
        *reinterpret_cast<uint4*>(rec + xr * 64 + (((e0 + 1) ^ xsw) << 4)) = hi;
        if (!DEBUG && (xc & 1) == 0) *reinterpret_cast<uint4*>(rec + kWZx + xr * 16) = make_uint4(zz, 0u, 0u, 0u);
    }
    // the operand is written (generic proxy) before the tensor cores (async proxy) read it; the
    // stage barrier completes once every epilogue warp has arrived
    fence_proxy_async_smem();
    __syncwarp();
    if ((et & 31) == 0) mbar_arrive(&full[jj % P::kStages]);
    return true;
}

// KS: CTAs (a cluster) per tile, each contracting 1/KS of K, as in gemm_kernel.
template <bool DEBUG, int KS>
__global__ void __launch_bounds__(kThreads, 1) gemm_packed_kernel(const __grid_constant__ GemmArgs args) {
    namespace P = packed;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::kOffBar);
    uint64_t* empty = full + P::kStages;
    uint64_t* wfull = empty + P::kStages;   // per ring slot
    uint64_t* tfull = wfull + P::kPkSlots;  // one per pair of TMEM buffers
    uint64_t* drain = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::kOffMisc);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    __shared__ float epi_sa[kEpiWarps][32];
    __shared__ float epi_bias[kEpiWarps][32];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_t = (args.M + kTileT - 1) / kTileT;
    const int64_t tiles_w = (args.N + kTileW - 1) / kTileW;
    const int64_t ntiles = tiles_t * tiles_w;
    static_assert(KS == 1 || (KS == 2 && !DEBUG), "the K split is a two-CTA cluster, outside the debug form");
    const uint32_t kr = KS > 1 ? cluster_ctarank() : 0u;
    const int64_t first = blockIdx.x / KS;
    const uint32_t nb = static_cast<uint32_t>(args.K / kBlock);  // blocks of a row
    const KPart kp{gridDim.x / KS, kr * (nb / KS), nb / KS};
    const uint32_t my_tiles = ntiles > first ? static_cast<uint32_t>((ntiles - 1 - first) / kp.stride + 1) : 0u;
    const uint32_t nbl = kp.nbl;
    const uint32_t spt = (nbl + 1) / 2;        // stages per tile
    const uint32_t total = my_tiles * spt;
    const WaitCtl ctl{abort_flag, args.status, args.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::kStages; ++s) {
            // the producer, and two arrivals per epilogue warp (its part of the operand expanded,
            // its part of the TMEM buffers released)
            mbar_init(&full[s], 1 + 2 * kEpiWarps);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < P::kPkSlots; ++s) mbar_init(&wfull[s], 1);  // producer
        for (int i = 0; i < 2; ++i) mbar_init(&tfull[i], 2);
        for (int i = 0; i < kIssuers; ++i) mbar_init(&drain[i], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (!DEBUG) {
        for (int i = threadIdx.x; i < kZeroBytes / 16; i += kThreads)
            reinterpret_cast<uint4*>(smem + P::kOffZero)[i] = make_uint4(0u, 0u, 0u, 0u);
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

    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 0) {
            // -------------------------------------------------------- producer
            if (lane == 0) {
                tma_prefetch_map(&args.wmap);
                // two walks over (tile, stage of the tile): W for the weights (ahead), T for the
                // token records; each looks its tile up once
                StageCursor cw{}, ct{};
                cursor_tile(cw, my_tiles, first, tiles_t, tiles_w, kp.stride);
                cursor_tile(ct, my_tiles, first, tiles_t, tiles_w, kp.stride);
                uint32_t wnext = 0;  // stages whose weights were issued
                const uint32_t ahead = P::kPkSlots - P::kStages;
                const uint32_t pre = total < static_cast<uint32_t>(P::kPkSlots) ? total : static_cast<uint32_t>(P::kPkSlots);
                if (args.early)
                    while (wnext < pre) issue_weights(args, smem, wfull, cw, wnext, spt, my_tiles, first, tiles_t, tiles_w, kp);
                griddep_wait();
                while (wnext < pre) issue_weights(args, smem, wfull, cw, wnext, spt, my_tiles, first, tiles_t, tiles_w, kp);
                bool ok = true;
                uint32_t issued = 0;
                for (uint32_t j = 0; j < total; ++j) {
                    const uint32_t k = j / P::kStages;
                    if (k > 0 && !mbar_wait(&empty[j % P::kStages], (k - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    const uint32_t b0 = 2 * ct.p, cnt = nbl - b0 < 2 ? 1u : 2u;
                    uint64_t* bar = &full[j % P::kStages];
                    mbar_arrive_expect_tx(bar, cnt * kTokRec);
                    bulk_load(smem + (j % P::kStages) * P::kStageBytes,
                              args.trec + (static_cast<int64_t>(ct.tt) * nb + kp.kb0 + b0) * kTokRec, cnt * kTokRec, bar);
                    cursor_next(ct, spt, my_tiles, first, tiles_t, tiles_w, kp.stride);
                    issued = j + 1;
                    // stage j - kStages is complete, and so is every stage before it: W(j + ahead)
                    // may reuse the slot of stage j + ahead - kPkSlots = j - kStages
                    if (k > 0 && wnext == j + ahead && wnext < total)
                        issue_weights(args, smem, wfull, cw, wnext, spt, my_tiles, first, tiles_t, tiles_w, kp);
                }
                if (!ok || *abort_flag) {
                    // let every copy already issued land before the CTA exits
                    for (uint32_t q = (wnext > static_cast<uint32_t>(P::kPkSlots) ? wnext - P::kPkSlots : 0); q < wnext; ++q)
                        drain_wait(&wfull[q % P::kPkSlots], (q / P::kPkSlots) & 1, 100000000ull);
                    for (uint32_t q = (issued > static_cast<uint32_t>(P::kStages) ? issued - P::kStages : 0); q < issued; ++q)
                        drain_wait(&full[q % P::kStages], (q / P::kStages) & 1, 100000000ull);
                }
            }
        } else {
            // -------------------------------------------------------- MMA issue (warps 1-3)
            const int iw = warp - 1;
            constexpr uint32_t idesc = idesc_e4m3_f32(kTileW, kTileT);
            const uint32_t zr = smem_u32(smem + P::kOffZero);
            const uint32_t t0a = smem_u32(smem), w0a = smem_u32(smem + P::kOffWop);
            const uint64_t dT0 = smem_desc(t0a, 1024, kLayoutSw128);
            const uint64_t dW0 = smem_desc(w0a, 512, kLayoutSw64);
            const uint64_t dBx0 = smem_desc(t0a + kTokRx, 128, 0, zr - (t0a + kTokRx));
            const uint64_t dAx0 = smem_desc(w0a + kWZx, 128, 0, zr - (w0a + kWZx));
            for (uint32_t i = iw; i < 2 * total; i += kIssuers) {
                const uint32_t j = i >> 1, k = i & 1u;
                const int s = static_cast<int>(j % P::kStages);
                const uint32_t pair = j & 1u;
                const uint32_t b0 = 2 * (j % spt), cnt = nbl - b0 < 2 ? 1u : 2u;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (j / P::kStages) & 1, ctl))) break;
                tc_fence_after();
                if (elect_one()) {
                    if (k < cnt) {
                        const uint32_t d = tmem_base + (2 * pair + k) * kTileT;
                        const uint64_t ot = static_cast<uint64_t>((s * P::kStageBytes + static_cast<int>(k) * kTokRec) >> 4);
                        const uint64_t ow = static_cast<uint64_t>((s * P::kStageBytes + static_cast<int>(k) * kWRec) >> 4);
                        const uint64_t dT = dT0 + ot, dW = dW0 + ow;
                        mma_f8f6f4(d, dW, dT, idesc, 0u);
                        mma_f8f6f4(d, dW + 2, dT + 2, idesc, 1u);
                        mma_f8f6f4(d, dW, dT + 4, idesc, 1u);
                        mma_f8f6f4(d, dW + 2, dT + 6, idesc, 1u);
                        if (!DEBUG) mma_f16(d, dAx0 + ow - (ow << 16), dBx0 + ot - (ot << 16), idesc, 1u);
                    }
                    mma_commit(&tfull[pair]);
                }
                __syncwarp();
            }
            if (elect_one()) mma_commit(&drain[iw]);
            __syncwarp();
            drain_wait(&drain[iw], 0, 100000000ull);
        }
        if (KS > 1) {  // the epilogue's two cluster barriers of the K split
            cluster_sync_all();
            cluster_sync_all();
        }
    } else {
        // ------------------------------------------------------------ epilogue + expansion
        regs_inc<kRegsHigh>();
        const int et = threadIdx.x - 4 * 32;           // 0 .. 511
        const int q = warp & 3, h = (warp - 4) >> 2;   // TMEM lane quarter (warp id mod 4), column quarter
        const int row = q * 32 + lane;
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 32);
        const bool lead = et == 0;
        bool ok = true;
        // the first stages' operands (their buffers start free); with `early` before the previous
        // kernel has finished: nothing here reads what it writes
        if (!args.early) griddep_wait();
        for (uint32_t jj = 0; ok && jj < total && jj < static_cast<uint32_t>(P::kStages); ++jj)
            ok = expand_stage<DEBUG>(args, smem, wfull, full, jj, spt, nb, first, tiles_t, tiles_w, et, ctl, kp);
        if (args.early) griddep_wait();
        // the TMEM buffers start free: release the first two stages
        if (lane == 0)
            for (uint32_t q0 = 0; q0 < 2 && q0 < total; ++q0) mbar_arrive(&full[q0]);
        uint32_t j = 0;  // stage counter of this CTA
        // this thread's sums and output position, kept past the tile loop for the K split
        float y[32];
        int64_t mt0 = 0, n = 0;
        for (uint32_t i = 0; ok && i < my_tiles; ++i) {
            int64_t tt, tw;
            tile_at32(first + static_cast<int64_t>(i) * kp.stride, tiles_t, tiles_w, tt, tw);
            mt0 = tt * kTileT + h * 32;  // first token column of this warp
            n = tw * kTileW + row;       // this thread's weight row
            // this row's scales from this CTA's first block of K
            const uint16_t* swr = (!DEBUG && n < args.N) ? args.s_w + n * nb + kp.kb0 : nullptr;
            if (!DEBUG && i + 1 < my_tiles && h == 0) {
                // the next tile's scales and zero points into L2 while this tile runs
                int64_t tt1, tw1;
                tile_at32(first + static_cast<int64_t>(i + 1) * kp.stride, tiles_t, tiles_w, tt1, tw1);
                const int64_t n1 = tw1 * kTileW + row;
                if (n1 < args.N) {
                    prefetch_l2_span(args.s_w + n1 * nb, nb * 2);
                    prefetch_l2_span(args.z_w + n1 * nb, nb * 2);
                }
            }
            if (!DEBUG) {
                epi_sa[warp - 4][lane] = mt0 + lane < args.M ? __ldcg(args.s_a + mt0 + lane) : 0.0f;
                epi_bias[warp - 4][lane] = (args.bias && n < args.N) ? __ldg(args.bias + n) : 0.0f;
            }
            // 512 s_w: the power of two undoes the 2^-9 of the e4m3 weight operand (exact)
            float ns0 = weight_scale(swr, 0, nbl), ns1 = weight_scale(swr, 1, nbl);
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] = 0.0f;
            for (uint32_t p = 0; p < spt; ++p, ++j) {
                const int s = static_cast<int>(j % P::kStages);
                const bool two = 2 * p + 1 < nbl;
                const float s0 = ns0, s1 = ns1;
                if (!DEBUG && p + 1 < spt) {
                    ns0 = weight_scale(swr, 2 * p + 2, nbl);
                    ns1 = weight_scale(swr, 2 * p + 3, nbl);
                }
                const uint32_t pair = j & 1u, b0 = 2 * pair;
                if (!__all_sync(0xffffffffu, mbar_wait(&tfull[pair], (j >> 1) & 1, ctl))) {
                    ok = false;
                    break;
                }
                // the stage's MMAs are complete: its token records may be reloaded
                if (lead) mbar_arrive(&empty[s]);
                tc_fence_after();
                // one block's accumulators at a time (32 registers): the expansion's state stays in
                // registers beside them
                uint32_t v[32];
#pragma unroll 1
                for (int e = 0; e < 2; ++e) {
                    if (e == 1 && !two) break;
                    const uint32_t tb = tl + (b0 + e) * kTileT;
                    tmem_ld_32x32b_x16(tb, v);
                    tmem_ld_32x32b_x16(tb + 16, v + 16);
                    tmem_wait_ld();
                    if (e == 1 || !two) {
                        // this warp's accumulators are in registers: its part of the buffers serves
                        // the stage two later
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0 && j + 2 < total) mbar_arrive(&full[(j + 2) % P::kStages]);
                    }
                    if (DEBUG) {
                        if (n < args.N) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const int64_t m = mt0 + c;
                                if (m < args.M)
                                    args.acc[(m * args.N + n) * nb + kp.kb0 + 2 * p + e] =
                                        static_cast<int32_t>(__uint_as_float(v[c]) * 512.0f);
                            }
                        }
                    } else {
                        const float sb = e == 0 ? s0 : s1;
                        fma_cols<32>(y, sb, v);
                    }
                }
                // operand stage s is free too (the stage's MMAs are done): the weights of stage
                // j + kStages go in, with the accumulators already folded (their registers free)
                if (j + P::kStages < total &&
                    !expand_stage<DEBUG>(args, smem, wfull, full, j + P::kStages, spt, nb, first, tiles_t, tiles_w, et, ctl,
                                         kp)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            if (!DEBUG) __syncwarp();  // every lane: the slots were written by other lanes of the warp
            if (!DEBUG && KS == 1 && n < args.N) {
                const float bn = epi_bias[warp - 4][lane];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int64_t m = mt0 + c;
                    if (m < args.M) store_y(args.out, m * args.N + n, fmaf(epi_sa[warp - 4][c], y[c], bn));
                }
            }
        }
        if (KS > 1) {
            // K split: the hand-off of gemm_kernel (the second CTA's partial sums through its own
            // idle stage memory, added by the first in the same order), so every output equals
            // the record form's bit for bit
            float* part = reinterpret_cast<float*>(smem) + (warp - 4) * 32 * 32 + lane;  // [warp][c][lane]
            if (kr == 1) {
#pragma unroll
                for (int c = 0; c < 32; ++c) part[c * 32] = y[c];
            }
            cluster_sync_all();
            if (kr == 0 && n < args.N) {
#pragma unroll
                for (int c = 0; c < 32; ++c) y[c] += ld_shared_cluster_f32(part + c * 32, 1);
                const float bn = epi_bias[warp - 4][lane];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int64_t m = mt0 + c;
                    if (m < args.M) store_y(args.out, m * args.N + n, fmaf(epi_sa[warp - 4][c], y[c], bn));
                }
            }
            cluster_sync_all();
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
                   cudaStream_t s, int threads = kThreads, int cluster = 1) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    // a K split runs exactly one tile per cluster of `cluster` CTAs (the host checked that they
    // all fit on the SMs at once)
    const int64_t grid = cluster > 1 ? tiles * cluster : (tiles < num_sms ? tiles : num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, bool debug, int num_sms, cudaStream_t s) {
    static bool attr_done[5][64] = {};
    if (num_sms < 1) return cudaErrorInvalidValue;
    const int64_t tiles_w = (a.N + kTileW - 1) / kTileW;
    if (a.tw == wide::kTN) {
        const int64_t tiles = ((a.M + wide::kTN - 1) / wide::kTN) * tiles_w;
        return debug ? launch(gemm_wide_kernel<true>, wide::kSmemBytes, attr_done[2], tiles, a, num_sms, s)
                     : launch(gemm_wide_kernel<false>, wide::kSmemBytes, attr_done[1], tiles, a, num_sms, s);
    }
    if (a.tw != kTileT) return cudaErrorInvalidValue;
    const int64_t tiles = ((a.M + kTileT - 1) / kTileT) * tiles_w;
    // the per-block accumulators of the debug form do not depend on how K is shared
    if (debug) return launch(gemm_kernel<true, 1>, kSmemBytes, attr_done[3], tiles, a, num_sms, s);
    if (a.ksplit == 1) return launch(gemm_kernel<false, 1>, kSmemBytes, attr_done[0], tiles, a, num_sms, s);
    if (a.ksplit != 2 || tiles * 2 > num_sms || (a.K / kBlock) % 2 != 0) return cudaErrorInvalidValue;
    return launch(gemm_kernel<false, 2>, kSmemBytes, attr_done[4], tiles, a, num_sms, s, kThreads, 2);
}

int gemm_ksplit(int64_t M, int64_t N, int64_t K, int tw, int num_sms) {
    if (tw != kTileT || M <= 0 || N <= 0) return 1;
    const int64_t tiles = ((M + kTileT - 1) / kTileT) * ((N + kTileW - 1) / kTileW);
    const int64_t nb = K / kBlock;
    // Measured: at K = 1024 (8 tiles) the split lost ~2 us to the cluster's hand-off, at K = 6144
    // (64 tiles) it saved 12 us of 41; from K = 2048 on each CTA drops eight stages or more.
    return (tiles * 2 <= num_sms && nb >= 32 && nb % 2 == 0) ? 2 : 1;
}

namespace {
// cuTensorMapEncodeTiled, resolved once through the runtime (no link-time dependence on the
// driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}
}  // namespace

cudaError_t launch_gemm_packed(const GemmArgs& a0, bool debug, int num_sms, cudaStream_t s) {
    static bool attr_done[3][64] = {};
    if (num_sms < 1 || a0.tw != kTileT || !a0.wq || (!debug && (!a0.s_w || !a0.z_w))) return cudaErrorInvalidValue;
    const EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    GemmArgs a = a0;
    // wq [N][K/2] bytes; a box is the 64 packed bytes (two 64-blocks) of 128 rows, 64-byte
    // swizzled as the converters read it; rows past N read as zeros
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K / 2), static_cast<cuuint64_t>(a.N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K / 2)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTileW)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&a.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t tiles = ((a.M + kTileT - 1) / kTileT) * ((a.N + kTileW - 1) / kTileW);
    if (debug) return launch(gemm_packed_kernel<true, 1>, packed::kSmemBytes, attr_done[1], tiles, a, num_sms, s);
    if (a.ksplit == 1) return launch(gemm_packed_kernel<false, 1>, packed::kSmemBytes, attr_done[0], tiles, a, num_sms, s);
    if (a.ksplit != 2 || tiles * 2 > num_sms || (a.K / kBlock) % 2 != 0) return cudaErrorInvalidValue;
    return launch(gemm_packed_kernel<false, 2>, packed::kSmemBytes, attr_done[2], tiles, a, num_sms, s, kThreads, 2);
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace w4a8
