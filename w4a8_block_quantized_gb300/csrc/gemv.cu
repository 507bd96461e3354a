// gemv.cu -- the few-token (decode) form of the block-64 W4A8 linear.
//
// "MNN LLM inference on the SpacemiT K3", section 3 eqs. (2)-(3) for the arithmetic; section
// 4's decode discussion for the shape of the work: one token per step, so the cost is one
// read of the packed weights with their block scales and zeros (tokens/s = bandwidth /
// weight bytes), streamed through a small on-chip buffer in ping-pong fashion while the
// previous piece is reduced, and the output written directly in fp32.
//
// With M <= kGemvMaxM tokens the contraction has no reuse worth a tensor-core tile: every
// weight is read once from HBM and used M times.  The weights are streamed as given (4 bits
// per weight + one fp16 s_w and one fp16 z_w per 64 weights = 4.5 bits per weight).
//
// Persistent CTAs, one per SM, each walking row tiles t = blockIdx.x, blockIdx.x + grid, ...
// (a launch of several linears: a contiguous range of tiles per CTA instead, so that each CTA
// stages the activations of only the one or two linears its range touches)
//   warp 8       producer: per tile three bulk copies into a ring of shared-memory stages --
//                the tile's packed rows (contiguous: rows are K/2 bytes apart) and the
//                16-byte-aligned interiors of its s_w and z_w rows (the few elements before
//                and after an interior are copied from global memory by the consumers, so
//                nothing outside the caller's arrays is touched).
//   warps 0-7    consumers.  A tile of TR >= 8 rows gives each warp TR/8 rows; a tile of
//                TR < 8 rows gives each row 8/TR warps that split its K chunks.  A lane owns
//                one 64-block of a row in every chunk of 32 blocks (2048 weights).
// The activations are staged once per CTA in shared memory, per token and chunk as four
// planes of 16 bytes per lane (plane p: codes 16p .. 16p+15 of the lane's block, each group
// of 8 codes as its even-k bytes then its odd-k bytes -- the order of the packed weight
// nibbles), with the block row sums as floats.  Either the CTA quantizes the rows itself
// from x (few tokens of moderate depth: the pre-pass's quantizer, quant_math.cuh, so the
// codes equal the pre-pass's bit for bit; the producer's first bulk copy brings x in, ahead
// of the weights) or it reads the pre-pass's outputs.  Per weight
// word: the low nibbles masked give the even codes for a signed dp4a; the high nibbles
// masked (16 q, kept unshifted) go through an unsigned x signed dp4a, the sum shifted right
// by 4 once per block; four independent accumulators.  A block's int32 product is exact;
// the epilogue forms t = acc - z_w rs with one fma and adds s_w t.  Sums: lane, then warp,
// then (split rows) the row's warps in a fixed order; y = s_a sum + bias.
//
// Every wait is bounded; a CTA that gives up records a timeout and unwinds.
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "quant_math.cuh"
#include "sm103_ptx.cuh"
#include "w4a8_internal.h"

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

namespace w4a8 {
namespace {

constexpr int kCW = 8;                     // consumer warps
constexpr int kGThreads = (kCW + 1) * 32;  // + the producer warp
constexpr int kChunkBlocks = 32;           // 64-blocks per row per warp step (one per lane)
constexpr int kChunkAct = kChunkBlocks * 64;  // staged activation bytes per token and chunk
constexpr int kMaxStages = 8;
constexpr int kSmemCap = 226 * 1024;  // dynamic; the static arrays fit in the last KiB
constexpr int kBarStage = 9;          // named barrier: the consumers while staging
// named barriers 1..4: the warps sharing one row of a tile of fewer than 8 rows

// One linear of a launch as the kernel sees it: the caller's arrays, and where its staged
// activations (token-major planes), block row sums (floats) and fp32 rows (quantizing launch)
// sit in shared memory.  Its row tiles are tiles tile0 .. tile0 + ceil(N / tr) - 1 of the
// launch.
struct GemvLin {
    const float* x;
    const int8_t* a_q;
    const float* s_a;
    const int32_t* rs;
    const uint8_t* wq;
    const uint16_t* s_w;
    const uint16_t* z_w;
    const float* bias;
    OutSpec out;
    int64_t N, K;
    int64_t tile0;
    uint32_t act_off, rs_off, x_off;
    uint32_t act_stride;  // staged activation bytes per token (chunks * 2048)
    int chunks;           // ceil(K / 2048)
    int tr;               // rows per tile of this linear
};

// The linears of a launch (one M), read by the kernel from parameter space.
struct GemvBatch {
    GemvLin lin[kGemvMaxLinears];
    int count = 0;
    int quantize = 0;  // every linear's rows are quantized in the kernel (x), else read (a_q, s_a, rs)
    int early = 0;     // the previous kernel in the stream writes none of the weights
};

// Shared-memory plan of one launch (computed on the host; identical for every CTA).  The tile
// heights (GemvLin::tr) are one for all linears, or, for a launch of several, may be one per
// linear chosen so that every tile holds about the same bytes (a stage slot holds the largest
// tile, so a deep linear's tiles no longer size the slots of the shallow ones).  Measured on a
// 2048-hidden decoder layer's seven linears in one launch: per-linear heights with contiguous
// ranges cut the step from 23.8 to 20.5 us (every CTA had quantized all seven rows, and the
// slots sized for the 6144-deep linear left two stages).  `tr` below is the largest height.
struct GemvPlan {
    int tr = 8;               // rows per tile
    int wpr = 1;              // warps per row (tr < 8)
    int ns = 2;               // stages
    uint32_t bar_off = 0, stage_off = 0;
    uint32_t stage_bytes = 0, w_bytes = 0, sz_bytes = 0;  // a stage; its weight part; one s_w / z_w slot
    uint32_t smem = 0;
    int64_t tiles = 0;
    int grid = 0;
    int contig = 0;           // each CTA takes a contiguous range of tiles (else every grid-th tile)
};

constexpr uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// One candidate of a plan: tile height trs[i] for linear i; a stage slot holds the largest tile.
// Replaces *best when its cost is lower.
void consider_plan(const GemvArgs* a, int count, const int* trs, uint32_t bar_off, uint32_t stage_off, int num_sms,
                   GemvPlan* best, int64_t* best_cost, int* best_tr) {
    uint32_t wb = 0, sz = 0;
    int64_t tiles = 0;
    int trmax = 0;
    for (int i = 0; i < count; ++i) {
        const int64_t K = a[i].K, nb = K / kBlock;
        wb = std::max(wb, align_up(static_cast<uint32_t>(trs[i] * K / 2), 16));
        sz = std::max(sz, align_up(static_cast<uint32_t>(trs[i] * nb * 2 + 32), 16));
        tiles += (a[i].N + trs[i] - 1) / trs[i];
        trmax = std::max(trmax, trs[i]);
    }
    const uint32_t stage = align_up(wb + 2 * sz, 128);
    const int64_t room = kSmemCap - 1024 - static_cast<int64_t>(stage_off);
    int64_t ns = room / stage;
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 2) return;
    const int64_t grid = tiles < num_sms ? tiles : num_sms;
    const int64_t waves = (tiles + grid - 1) / grid;
    // bytes streamed by the busiest CTA, plus a fixed cost per tile (barriers, sums), counted as
    // 16 KiB of streaming.  Measured on the 7B-class decode pair: with a 4 KiB charge the planner
    // split the 14336-deep rows over two warps (4-row tiles, seven waves); one warp per row (8-row
    // tiles, four waves) made the pair's step 7% faster, and the decoder-layer and single-linear
    // steps were unchanged.
    const int64_t cost = waves * (static_cast<int64_t>(stage) + 16384);
    if (*best_cost >= 0 && cost >= *best_cost) return;
    *best_cost = cost;
    best->tr = trmax;
    best->wpr = trmax >= 8 ? 1 : 8 / trmax;
    best->ns = static_cast<int>(ns);
    best->bar_off = bar_off;
    best->stage_off = stage_off;
    best->stage_bytes = stage;
    best->w_bytes = wb;
    best->sz_bytes = sz;
    best->smem = stage_off + static_cast<uint32_t>(ns) * stage + 1024;  // + base alignment slack
    best->tiles = tiles;
    best->grid = static_cast<int>(grid);
    // a batch: contiguous tile ranges, so that a CTA stages only the linears of its range
    best->contig = count > 1 ? 1 : 0;
    for (int i = 0; i < count; ++i) best_tr[i] = trs[i];
}

// Lays out the linears' staging areas (into b) and picks the tile height; false if they do not
// fit one CTA's shared memory next to two weight stages.
// `min_tr`: the smallest tile height allowed.  Heights of 8 rows and more give every output row
// one warp, whose sum runs in the same order whatever the height; a launch of several linears
// uses only those, so its outputs equal each linear's own launch bit for bit when that launch
// also has one warp per row.
bool plan_uncached(const GemvArgs* a, int count, bool quantize, int num_sms, GemvBatch* b, GemvPlan* out,
                  int min_tr) {
    if (count < 1 || count > kGemvMaxLinears) return false;
    const int64_t M = a[0].M;
    int64_t off = 0;
    for (int i = 0; i < count; ++i) {  // activations, then row sums, then fp32 rows
        const int64_t nb = a[i].K / kBlock;
        const int chunks = static_cast<int>((nb + kChunkBlocks - 1) / kChunkBlocks);
        b->lin[i].chunks = chunks;
        b->lin[i].act_stride = static_cast<uint32_t>(chunks) * kChunkAct;
        b->lin[i].act_off = static_cast<uint32_t>(off);
        off = align_up(static_cast<uint32_t>(off + M * chunks * kChunkAct), 128);
        if (off > kSmemCap) return false;
    }
    for (int i = 0; i < count; ++i) {
        b->lin[i].rs_off = static_cast<uint32_t>(off);
        off = align_up(static_cast<uint32_t>(off + M * (a[i].K / kBlock) * 4), 128);
        if (off > kSmemCap) return false;
    }
    for (int i = 0; i < count; ++i) {
        b->lin[i].x_off = static_cast<uint32_t>(off);
        if (quantize) off = align_up(static_cast<uint32_t>(off + M * a[i].K * 4), 128);
        if (off > kSmemCap) return false;
    }
    const uint32_t bar_off = static_cast<uint32_t>(off);
    const uint32_t stage_off = align_up(bar_off + (2 * kMaxStages + 1) * 8 + 16, 1024);
    GemvPlan best;
    int64_t best_cost = -1;
    int best_tr[kGemvMaxLinears];
    int trs[kGemvMaxLinears];
    for (int tr : {32, 16, 8, 4, 2, 1}) {  // one height for every linear
        if (tr > 8 && M > 2) continue;  // more rows per warp only for one or two tokens
        if (tr < min_tr) continue;
        for (int i = 0; i < count; ++i) trs[i] = tr;
        consider_plan(a, count, trs, bar_off, stage_off, num_sms, &best, &best_cost, best_tr);
    }
    if (count > 1) {
        // A height per linear (multiples of 8, so every row keeps one warp), for tiles of about
        // `target` bytes in every linear: the stage slots then fit the tiles of a deep linear and
        // of a shallow one alike, and more of them fit.
        const int hmax = M > 2 ? 8 : 32;
        for (int64_t target : {8192, 12288, 16384, 24576, 32768, 49152, 65536}) {
            for (int i = 0; i < count; ++i) {
                const int64_t row = a[i].K / 2;
                const int64_t t = 8 * std::max<int64_t>(1, (target + 4 * row) / (8 * row));
                trs[i] = static_cast<int>(std::max<int64_t>(std::min<int64_t>(t, hmax), std::max(min_tr, 8)));
            }
            consider_plan(a, count, trs, bar_off, stage_off, num_sms, &best, &best_cost, best_tr);
        }
    }
    if (best_cost < 0) return false;
    int64_t t0 = 0;
    for (int i = 0; i < count; ++i) {
        b->lin[i].tile0 = t0;
        b->lin[i].tr = best_tr[i];
        t0 += (a[i].N + best_tr[i] - 1) / best_tr[i];
    }
    *out = best;
    return true;
}

// make_plan remembers its answers: one call of the API plans the same shapes several times
// (the support checks, the batch's own plan, its launch), and a decode step is short enough
// that host time shows in it.  A small direct-mapped table keyed by everything the plan reads.
struct PlanKey {
    int32_t count, quantize, num_sms, min_tr;
    int64_t M, K[kGemvMaxLinears], N[kGemvMaxLinears];
};
struct PlanMemo {
    bool used = false, ok = false;
    PlanKey key;
    GemvPlan plan;
    GemvLin lin[kGemvMaxLinears];  // the layout fields make_plan sets
};
constexpr int kPlanSlots = 64;
PlanMemo g_plan_memo[kPlanSlots];
std::mutex g_plan_mu;

bool make_plan(const GemvArgs* a, int count, bool quantize, int num_sms, GemvBatch* b, GemvPlan* out,
               int min_tr = 1) {
    if (count < 1 || count > kGemvMaxLinears) return false;
    if (count == 1) return plan_uncached(a, count, quantize, num_sms, b, out, min_tr);  // cheaper than a lookup
    PlanKey k;
    std::memset(&k, 0, sizeof(k));
    k.count = count;
    k.quantize = quantize ? 1 : 0;
    k.num_sms = num_sms;
    k.min_tr = min_tr;
    k.M = a[0].M;
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
    mix(static_cast<uint64_t>(count) | static_cast<uint64_t>(k.quantize) << 8 | static_cast<uint64_t>(min_tr) << 16);
    mix(static_cast<uint64_t>(num_sms));
    mix(static_cast<uint64_t>(k.M));
    for (int i = 0; i < count; ++i) {
        k.K[i] = a[i].K;
        k.N[i] = a[i].N;
        mix(static_cast<uint64_t>(a[i].K));
        mix(static_cast<uint64_t>(a[i].N));
    }
    PlanMemo& m = g_plan_memo[h % kPlanSlots];
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        if (m.used && std::memcmp(&m.key, &k, sizeof(k)) == 0) {
            for (int i = 0; i < count; ++i) {
                GemvLin& L = b->lin[i];
                L.chunks = m.lin[i].chunks;
                L.act_stride = m.lin[i].act_stride;
                L.act_off = m.lin[i].act_off;
                L.rs_off = m.lin[i].rs_off;
                L.x_off = m.lin[i].x_off;
                L.tile0 = m.lin[i].tile0;
                L.tr = m.lin[i].tr;
            }
            if (m.ok) *out = m.plan;
            return m.ok;
        }
    }
    GemvPlan P;
    const bool ok = plan_uncached(a, count, quantize, num_sms, b, &P, min_tr);
    if (ok) *out = P;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    m.used = true;
    m.ok = ok;
    m.key = k;
    m.plan = P;
    for (int i = 0; i < count; ++i) m.lin[i] = b->lin[i];
    return ok;
}

// The linear that global tile g belongs to.
__device__ __forceinline__ int lin_of(const GemvBatch& B, int64_t g) {
    int li = 0;
    while (li + 1 < B.count && g >= B.lin[li + 1].tile0) ++li;
    return li;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}
// unsigned bytes of a x signed bytes of b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Elements [e0, e1) of a fp16 array, staged with one bulk copy of their 16-byte-aligned
// interior.  The slot keeps the array's alignment: element e0 sits `skew` bytes into it
// (its address mod 16), and the interior -- bytes [lo, hi) counted from element e0 -- lands
// at slot offset skew + lo.  The at most 7 elements before and 7 after the interior (byte
// offsets outside [lo, hi)) are not copied; readers load them from global memory, so no copy
// touches memory outside the caller's array.  An interior shorter than 16 bytes is empty
// (lo == hi, bytes == 0).
struct HalfSpan {
    const uint8_t* src;  // the interior's first byte
    uint32_t bytes, skew, lo, hi;
};

__device__ __forceinline__ HalfSpan half_span(const uint16_t* base, int64_t e0, int64_t e1) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(base + e0), a1 = reinterpret_cast<uintptr_t>(base + e1);
    const uintptr_t i0 = (a0 + 15) & ~uintptr_t(15), i1 = a1 & ~uintptr_t(15);
    HalfSpan h;
    h.src = reinterpret_cast<const uint8_t*>(i0);
    h.bytes = i1 > i0 ? static_cast<uint32_t>(i1 - i0) : 0u;
    h.skew = static_cast<uint32_t>(a0 & 15);
    h.lo = static_cast<uint32_t>(i0 - a0);
    h.hi = h.lo + h.bytes;
    return h;
}

// Whether the span of elements [e0, e1) of `base` begins and ends on a 16-byte boundary (its
// interior copy is then the whole span).
__device__ __forceinline__ bool span_whole(const uint16_t* base, int64_t e0, int64_t e1) {
    return ((reinterpret_cast<uintptr_t>(base + e0) | reinterpret_cast<uintptr_t>(base + e1)) & 15) == 0;
}

// The elements of a staged span that its interior copy left out (the at most 7 before and 7
// after the interior, when the span does not begin or end on a 16-byte boundary), loaded from
// global memory into the slot by consumer thread t < 32: threads 0-15 for the scales, 16-31 for
// the zero points.  The caller synchronizes the consumers afterwards.
__device__ __forceinline__ void fill_ragged(uint32_t s_slot, uint32_t z_slot, const uint16_t* s_w, const uint16_t* z_w,
                                            int64_t e0, int64_t e1, int t) {
    if (t >= 32) return;
    const bool zs = t >= 16;
    const uint16_t* base = zs ? z_w : s_w;
    const HalfSpan h = half_span(base, e0, e1);
    const uint32_t span = static_cast<uint32_t>((e1 - e0) * 2);
    const uint32_t k = static_cast<uint32_t>(t & 15), head = h.lo / 2;
    // head elements at byte offsets 0, 2, .., lo - 2; then the tail from hi on
    const uint32_t eo = k < head ? 2 * k : h.hi + 2 * (k - head);
    if (eo < span && (k < head || eo >= h.hi)) {
        const uint16_t v = __ldg(base + e0 + eo / 2);
        asm volatile("st.shared.u16 [%0], %1;" ::"r"((zs ? z_slot : s_slot) + h.skew + eo), "h"(v) : "memory");
    }
}

// A float code (an exact integer in [-127, 127]) as a word whose low byte is the code in two's
// complement: adding 1.5 * 2^23 puts the integer in the low mantissa bits.  One fp32 add, not
// a conversion instruction.
__device__ __forceinline__ int code_bits(float q) { return static_cast<int>(__float_as_uint(__fadd_rn(q, 12582912.0f))); }

// Low bytes of four int codes, c0 in byte 0.
__device__ __forceinline__ uint32_t pack4(int c0, int c1, int c2, int c3) {
    return __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
}

// Staged plane of 16 codes k = 16p .. 16p+15 of a block: {E, O} of codes 0-7 then of 8-15
// (E: the even codes of the group of 8, O: the odd ones), from four words of codes in k order.
__device__ __forceinline__ uint4 plane_of(uint32_t n0, uint32_t n1, uint32_t n2, uint32_t n3) {
    return make_uint4(__byte_perm(n0, n1, 0x6420), __byte_perm(n0, n1, 0x7531), __byte_perm(n2, n3, 0x6420),
                      __byte_perm(n2, n3, 0x7531));
}

// Exact product of one block: W0 / W1 the block's 32 packed bytes (codes 0-31 / 32-63 of
// the block, even k in the low nibbles), P the four staged planes of the token.
__device__ __forceinline__ int block_dot(const uint4& W0, const uint4& W1, const uint4 (&P)[4]) {
    constexpr uint32_t kLo = 0x0F0F0F0Fu, kHi = 0xF0F0F0F0u;
    int la = dp4a_ss(W0.x & kLo, P[0].x, 0), ha = dp4a_us(W0.x & kHi, P[0].y, 0);
    int lb = dp4a_ss(W0.y & kLo, P[0].z, 0), hb = dp4a_us(W0.y & kHi, P[0].w, 0);
    la = dp4a_ss(W0.z & kLo, P[1].x, la);
    ha = dp4a_us(W0.z & kHi, P[1].y, ha);
    lb = dp4a_ss(W0.w & kLo, P[1].z, lb);
    hb = dp4a_us(W0.w & kHi, P[1].w, hb);
    la = dp4a_ss(W1.x & kLo, P[2].x, la);
    ha = dp4a_us(W1.x & kHi, P[2].y, ha);
    lb = dp4a_ss(W1.y & kLo, P[2].z, lb);
    hb = dp4a_us(W1.y & kHi, P[2].w, hb);
    la = dp4a_ss(W1.z & kLo, P[3].x, la);
    ha = dp4a_us(W1.z & kHi, P[3].y, ha);
    lb = dp4a_ss(W1.w & kLo, P[3].z, lb);
    hb = dp4a_us(W1.w & kHi, P[3].w, hb);
    return (la + lb) + ((ha + hb) >> 4);  // the high sums are 16 x (odd-code products), exact
}

// The producer's copies of one row tile (global tile g, of linear L) into stage s: the packed
// rows, and the 16-byte-aligned interiors of the scale and zero spans.
__device__ __forceinline__ void issue_tile(const GemvLin& L, const GemvPlan& P, uint8_t* smem, uint64_t* full,
                                           int64_t g, int s) {
    const int64_t K = L.K, nb = K / kBlock;
    const int64_t n0 = (g - L.tile0) * L.tr;
    const int64_t rows = L.N - n0 < L.tr ? L.N - n0 : L.tr;
    const uint32_t wbytes = static_cast<uint32_t>(rows * (K / 2));
    const HalfSpan hs = half_span(L.s_w, n0 * nb, (n0 + rows) * nb);
    const HalfSpan hz = half_span(L.z_w, n0 * nb, (n0 + rows) * nb);
    uint8_t* st = smem + P.stage_off + s * P.stage_bytes;
    mbar_arrive_expect_tx(&full[s], wbytes + hs.bytes + hz.bytes);
    bulk_load(st, L.wq + n0 * (K / 2), wbytes, &full[s]);
    if (hs.bytes) bulk_load(st + P.w_bytes + hs.skew + hs.lo, hs.src, hs.bytes, &full[s]);
    if (hz.bytes) bulk_load(st + P.w_bytes + P.sz_bytes + hz.skew + hz.lo, hz.src, hz.bytes, &full[s]);
}

template <int MT, int RW>
__global__ void __launch_bounds__(kGThreads, 1)
    gemv_kernel(const __grid_constant__ GemvBatch B, const GemvPlan P, uint32_t* status, uint64_t wait_limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + P.bar_off);
    uint64_t* empty = full + kMaxStages;
    uint64_t* xbar = empty + kMaxStages;  // the fp32 rows (quantizing kernel)
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(xbar + 1);
    __shared__ float red[2][kCW][MT];
    __shared__ float amax_red[2][kCW];
    __shared__ float sa_sm[kGemvMaxLinears][MT];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = P.ns;
    // this CTA's tiles g_lo, g_lo + g_step, ...: a contiguous range (a batch: the CTA then stages
    // only the one or two linears its range touches) or every gridDim.x-th tile
    int64_t g_lo = blockIdx.x, g_step = gridDim.x;
    uint32_t my_tiles;
    if (P.contig) {
        g_lo = P.tiles * blockIdx.x / gridDim.x;
        my_tiles = static_cast<uint32_t>(P.tiles * (blockIdx.x + 1) / gridDim.x - g_lo);
        g_step = 1;
    } else {
        my_tiles = P.tiles > blockIdx.x ? static_cast<uint32_t>((P.tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0u;
    }
    // the linears those tiles belong to (tiles are numbered linear after linear)
    const int li_lo = my_tiles ? lin_of(B, g_lo) : 0;
    const int li_hi = my_tiles ? lin_of(B, g_lo + static_cast<int64_t>(my_tiles - 1) * g_step) : -1;
    const WaitCtl ctl{abort_flag, status, wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        mbar_init(xbar, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // The weights are read-only inputs: when the previous kernel cannot have written them
            // (`early`), the first stages' copies go out before it has finished, so this kernel's
            // weight stream overlaps its tail.  Everything else waits for it.
            uint32_t i = 0;
            if (B.early)
                for (; i < my_tiles && i < static_cast<uint32_t>(ns); ++i) {
                    const int64_t g = g_lo + static_cast<int64_t>(i) * g_step;
                    issue_tile(B.lin[lin_of(B, g)], P, smem, full, g, static_cast<int>(i));
                }
            griddep_wait();
            if (B.quantize) {
                // the rows to quantize, every linear's: every CTA reads them
                uint32_t xbytes = 0;
                for (int li = li_lo; li <= li_hi; ++li) xbytes += static_cast<uint32_t>(MT * B.lin[li].K * 4);
                mbar_arrive_expect_tx(xbar, xbytes);
                for (int li = li_lo; li <= li_hi; ++li)
                    bulk_load(smem + B.lin[li].x_off, B.lin[li].x, static_cast<uint32_t>(MT * B.lin[li].K * 4), xbar);
            }
            bool ok = true;
            for (; i < my_tiles; ++i) {
                const int s = static_cast<int>(i % ns);
                const uint32_t k = i / ns;
                if (k > 0 && !mbar_wait(&empty[s], (k - 1) & 1, ctl)) {
                    ok = false;
                    break;
                }
                const int64_t g = g_lo + static_cast<int64_t>(i) * g_step;
                issue_tile(B.lin[lin_of(B, g)], P, smem, full, g, s);
            }
            if (!ok || *abort_flag) {
                // let the copies already issued land before the CTA exits
                for (uint32_t q = (i > static_cast<uint32_t>(ns) ? i - ns : 0); q < i; ++q) {
                    const uint32_t bar = smem_u32(&full[q % ns]), par = (q / ns) & 1;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(bar, par) && globaltimer_ns() - t0 < 100000000ull) {
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        griddep_wait();
        // Stage every linear's activations: token m, block b = 32 c + l -> four 16-byte planes at
        // act_off + m * act_stride + 2048 c + 512 p + 16 l; the block row sums as floats; s_a.
        const bool got = !B.quantize || __all_sync(0xffffffffu, mbar_wait(xbar, 0, ctl));
        int par = 0;  // alternates the amax slots from row to row
        for (int li = li_lo; li <= li_hi; ++li) {
            const GemvLin& L = B.lin[li];
            const int64_t K = L.K, nb = K / kBlock;
            float* rsf_sm = reinterpret_cast<float*>(smem + L.rs_off);
            auto plane_addr = [&](int64_t m, int64_t b, int p) {
                return smem + L.act_off + m * L.act_stride + (b >> 5) * kChunkAct + p * 512 + (b & 31) * 16;
            };
            if (B.quantize) {
                // Quantize here, from the rows the producer copied in (nb <= 256).  The units are
                // 16 codes (a block's plane): lane group 4b .. 4b+3 of a warp holds block b.
                const uint32_t xs_base = smem_u32(smem + L.x_off);
                for (int m = 0; m < MT; ++m, par ^= 1) {
                    const uint32_t xr = xs_base + static_cast<uint32_t>(m * K * 4);
                    float amax = 0.0f;
                    for (int64_t f = threadIdx.x; got && f < K / 4; f += kCW * 32) {
                        const uint4 v = lds128(xr + static_cast<uint32_t>(f * 16));
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(__uint_as_float(v.x)), fabsf(__uint_as_float(v.y))),
                                                 fmaxf(fabsf(__uint_as_float(v.z)), fabsf(__uint_as_float(v.w)))));
                    }
#pragma unroll
                    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    if (lane == 0) amax_red[par][warp] = amax;
                    named_bar_sync(kBarStage, kCW * 32);
                    amax = 0.0f;
#pragma unroll
                    for (int w = 0; w < kCW; ++w) amax = fmaxf(amax, amax_red[par][w]);
                    const float s = __fdiv_rn(amax, 127.0f);
                    const float r = __frcp_rn(s);
                    if (threadIdx.x == 0) sa_sm[li][m] = s;
                    const int units = static_cast<int>(4 * nb);
                    for (int u0 = warp * 32; u0 < units; u0 += kCW * 32) {  // warp-uniform trip count
                        const int u = u0 + lane, b = u >> 2, p = u & 3;
                        const bool on = got && u < units;
                        // slot j holds float4 (j + rot) % 4 of the unit: consecutive lanes sit 64 bytes
                        // apart, and the rotation spreads each 8-lane phase of the loads over all banks
                        const int rot = (lane >> 1) & 3;
                        float4 xs[4], q[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int jj = (j + rot) & 3;
                            const uint4 v = on ? lds128(xr + static_cast<uint32_t>((64 * b + 16 * p + 4 * jj) * 4))
                                               : make_uint4(0, 0, 0, 0);
                            xs[j] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                                                __uint_as_float(v.w));
                        }
                        if (s > 0.0f) {  // s = 0: every code 0
                            quant_lane<4>(xs, q, s, r);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) q[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        uint32_t nr[4];
                        float part = 0.0f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            part += (q[j].x + q[j].y) + (q[j].z + q[j].w);  // exact
                            nr[j] = pack4(code_bits(q[j].x), code_bits(q[j].y), code_bits(q[j].z), code_bits(q[j].w));
                        }
                        // back to k order: n[k] = nr[(k - rot) % 4], a rotation by rot in two select steps
                        uint32_t h[4], n[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) h[k] = (rot & 1) ? nr[(k + 3) & 3] : nr[k];
#pragma unroll
                        for (int k = 0; k < 4; ++k) n[k] = (rot & 2) ? h[(k + 2) & 3] : h[k];
                        if (on) *reinterpret_cast<uint4*>(plane_addr(m, b, p)) = plane_of(n[0], n[1], n[2], n[3]);
                        part += __shfl_xor_sync(0xffffffffu, part, 1);
                        part += __shfl_xor_sync(0xffffffffu, part, 2);
                        if (on && p == 0) rsf_sm[m * nb + b] = part;
                    }
                }
            } else {
                for (int64_t u = threadIdx.x; u < MT * nb; u += kCW * 32) {
                    const int64_t m = u / nb, b = u - m * nb;
                    const int4* src = reinterpret_cast<const int4*>(L.a_q + m * K + 64 * b);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int4 v = __ldcg(src + p);
                        *reinterpret_cast<uint4*>(plane_addr(m, b, p)) =
                            plane_of(static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y), static_cast<uint32_t>(v.z),
                                     static_cast<uint32_t>(v.w));
                    }
                    rsf_sm[u] = static_cast<float>(__ldcg(L.rs + u));
                }
                if (threadIdx.x < MT) sa_sm[li][threadIdx.x] = __ldcg(L.s_a + threadIdx.x);
            }
        }
        named_bar_sync(kBarStage, kCW * 32);
        // the next kernel in the stream may start its prologue as this CTA's SM frees up; it
        // still waits for this whole grid (and its memory) before it touches data
        griddep_launch_dependents();

        const int wpr = P.wpr;
        const int rslot = warp / wpr, sidx = warp - rslot * wpr;
        for (uint32_t i = 0; i < my_tiles; ++i) {
            const int s = static_cast<int>(i % ns);
            const int64_t g = g_lo + static_cast<int64_t>(i) * g_step;
            const int li = lin_of(B, g);
            const GemvLin& L = B.lin[li];
            const int64_t N = L.N, nb = L.K / kBlock;
            const int tr = L.tr;
            const int64_t n0 = (g - L.tile0) * tr;
            const uint32_t act_base = smem_u32(smem + L.act_off), rs_base = smem_u32(smem + L.rs_off);
            const uint32_t krow = static_cast<uint32_t>(L.K / 2), nbu = static_cast<uint32_t>(nb);
            const int chunks = L.chunks;
            const uint32_t act_stride = L.act_stride;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (i / ns) & 1, ctl));
            const uint32_t st = smem_u32(smem + P.stage_off + s * P.stage_bytes);
            const int64_t rows = N - n0 < tr ? N - n0 : tr;
            // each span's element e0 sits at its slot offset `skew`; a span that does not begin
            // and end on a 16-byte boundary (possible when K is not a multiple of 512, or for
            // arrays that do not start on one) has its ragged ends filled in from global memory
            const int64_t e0 = n0 * nb, e1 = (n0 + rows) * nb;
            const uint32_t s_slot = st + P.w_bytes, z_slot = st + P.w_bytes + P.sz_bytes;
            const uint32_t swb = s_slot + static_cast<uint32_t>(reinterpret_cast<uintptr_t>(L.s_w + e0) & 15);
            const uint32_t zwb = z_slot + static_cast<uint32_t>(reinterpret_cast<uintptr_t>(L.z_w + e0) & 15);
            if (!(span_whole(L.s_w, e0, e1) && span_whole(L.z_w, e0, e1))) {  // the same for every consumer
                fill_ragged(s_slot, z_slot, L.s_w, L.z_w, e0, e1, static_cast<int>(threadIdx.x));
                // the slot is reloaded by a bulk copy (async proxy) after the stage is released
                fence_proxy_async_smem();
                named_bar_sync(kBarStage, kCW * 32);
            }
            // the rows of this warp in the tile: r_j = warp + 8 j (tr >= 8) or rslot (tr < 8)
            int rrow[RW];
            bool rok[RW];
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                rrow[j] = tr >= 8 ? warp + 8 * j : rslot;
                rok[j] = ok && rrow[j] < tr && n0 + rrow[j] < N;
            }
            float sum[RW][MT];
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int m = 0; m < MT; ++m) sum[j][m] = 0.0f;
            if (ok) {
                for (int c = sidx; c < chunks; c += wpr) {
                    const uint32_t b = static_cast<uint32_t>(c * kChunkBlocks + lane);
                    const bool live = b < nbu;
                    uint4 W0[RW], W1[RW];
                    float sw[RW], nz[RW];
#pragma unroll
                    for (int j = 0; j < RW; ++j) {
                        const bool on = rok[j] && live;
                        const uint32_t wa = st + rrow[j] * krow + b * 32;
                        W0[j] = on ? lds128(wa) : make_uint4(0, 0, 0, 0);
                        W1[j] = on ? lds128(wa + 16) : make_uint4(0, 0, 0, 0);
                        const uint32_t e = (rrow[j] * nbu + b) * 2;
                        sw[j] = on ? __half2float(__ushort_as_half(lds16(swb + e))) : 0.0f;
                        nz[j] = on ? -__half2float(__ushort_as_half(lds16(zwb + e))) : 0.0f;
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        uint4 Pl[4];
                        const uint32_t ad = act_base + m * act_stride + c * kChunkAct + 16 * lane;
#pragma unroll
                        for (int p = 0; p < 4; ++p) Pl[p] = lds128(ad + p * 512);
                        const float rsf = live ? lds_f32(rs_base + (m * nbu + b) * 4) : 0.0f;
#pragma unroll
                        for (int j = 0; j < RW; ++j) {
                            const int acc = block_dot(W0[j], W1[j], Pl);
                            sum[j][m] = fmaf(sw[j], fmaf(nz[j], rsf, static_cast<float>(acc)), sum[j][m]);
                        }
                    }
                }
            }
            // the stage has been read
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            // the warp sums (a full butterfly: every lane ends with the total; lane m stores token m)
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = sum[j][m];
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    sum[j][m] = v;
                }
            if (wpr == 1) {
#pragma unroll
                for (int j = 0; j < RW; ++j) {
                    const int64_t n = n0 + rrow[j];
                    float v = sum[j][0];
#pragma unroll
                    for (int m = 1; m < MT; ++m)
                        if (lane == m) v = sum[j][m];
                    if (rok[j] && lane < MT)
                        store_y(L.out, static_cast<int64_t>(lane) * N + n,
                                fmaf(sa_sm[li][lane], v, L.bias ? L.bias[n] : 0.0f));
                }
            } else {
                // the row's warps meet (every warp meets once per tile, whatever its waits gave)
                if (lane == 0)
#pragma unroll
                    for (int m = 0; m < MT; ++m) red[i & 1][warp][m] = sum[0][m];
                named_bar_sync(1 + rslot, wpr * 32);
                const int64_t n = n0 + rslot;
                if (sidx == 0 && rok[0] && lane < MT) {
                    float v = 0.0f;
                    for (int q = 0; q < wpr; ++q) v += red[i & 1][rslot * wpr + q][lane];
                    store_y(L.out, static_cast<int64_t>(lane) * N + n,
                            fmaf(sa_sm[li][lane], v, L.bias ? L.bias[n] : 0.0f));
                }
            }
        }
    }
    __syncthreads();
}

template <int MT, int RW>
cudaError_t launch_one(const GemvBatch& b, const GemvPlan& P, uint32_t* status, cudaStream_t s) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(gemv_kernel<MT, RW>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(P.grid));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = P.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MT, RW>, b, P, status, uint64_t(1000000000ull));
}

template <int MT>
cudaError_t launch_mt(const GemvBatch& b, const GemvPlan& P, uint32_t* status, cudaStream_t s) {
    if constexpr (MT <= 2) {
        if (P.tr == 32) return launch_one<MT, 4>(b, P, status, s);
        if (P.tr == 24) return launch_one<MT, 3>(b, P, status, s);
        if (P.tr == 16) return launch_one<MT, 2>(b, P, status, s);
    }
    return launch_one<MT, 1>(b, P, status, s);
}

GemvArgs shape_only(int64_t M, int64_t K) {
    GemvArgs a;
    a.M = M;
    a.N = 1;
    a.K = K;
    return a;
}

// The checks of a batch launch, and its plan: one M (1 .. kGemvMaxM), every linear quantized in
// the kernel or none, every row short enough for the kernel, the staging areas within one CTA.
bool plan_batch(const GemvArgs* a, int count, int num_sms, GemvBatch* b, GemvPlan* P) {
    if (count < 1 || count > kGemvMaxLinears) return false;
    const int64_t M = a[0].M;
    const bool quantize = a[0].x != nullptr;
    if (M < 1 || M > kGemvMaxM) return false;
    for (int i = 0; i < count; ++i) {
        if (a[i].M != M || a[i].N < 1 || (a[i].x != nullptr) != quantize || !gemv_supported(M, a[i].K)) return false;
        if (quantize && !gemv_quantizes(M, a[i].K)) return false;
    }
    *b = GemvBatch{};
    return make_plan(a, count, quantize, num_sms, b, P, count > 1 ? 8 : 1);
}

}  // namespace

namespace {
// Both answers for one (M, K), remembered: the API asks them for every entry of every call.
// One word per slot -- valid bit, M, K / 64, the two answers -- so readers need no lock.
constexpr int kFitSlots = 256;
std::atomic<uint64_t> g_fit[kFitSlots];

uint64_t fits_uncached(int64_t M, int64_t K) {
    const GemvArgs a = shape_only(M, K);
    GemvBatch b{};
    GemvPlan P;
    const bool sup = M >= 1 && M <= kGemvMaxM && K >= kBlock && make_plan(&a, 1, false, 1, &b, &P);
    const bool quant = sup && M * K <= kGemvFuseElems && make_plan(&a, 1, true, 1, &b, &P);
    return (sup ? 1u : 0u) | (quant ? 2u : 0u);
}

// bit 0: the few-token kernel takes (M, K); bit 1: it also quantizes such rows itself
uint64_t fits(int64_t M, int64_t K) {
    if (M < 1 || M > kGemvMaxM || K < kBlock || K % kBlock != 0 || K / kBlock >= (int64_t(1) << 40))
        return fits_uncached(M, K);
    const uint64_t tag = (uint64_t(1) << 63) | static_cast<uint64_t>(M) << 48 | static_cast<uint64_t>(K / kBlock) << 2;
    std::atomic<uint64_t>& slot = g_fit[(static_cast<uint64_t>(K / kBlock) * 8 + static_cast<uint64_t>(M)) % kFitSlots];
    const uint64_t v = slot.load(std::memory_order_relaxed);
    if ((v & ~uint64_t(3)) == tag) return v & 3;
    const uint64_t r = fits_uncached(M, K);
    slot.store(tag | r, std::memory_order_relaxed);
    return r;
}
}  // namespace

bool gemv_supported(int64_t M, int64_t K) { return (fits(M, K) & 1) != 0; }

bool gemv_quantizes(int64_t M, int64_t K) { return (fits(M, K) & 2) != 0; }

bool gemv_batch_fits(const GemvArgs* a, int count) {
    GemvBatch b{};
    GemvPlan P;
    return plan_batch(a, count, 1, &b, &P);
}

int gemv_tile_rows(const GemvArgs& a, int num_sms) {
    GemvBatch b{};
    GemvPlan P;
    return plan_batch(&a, 1, num_sms, &b, &P) ? P.tr : 0;
}

cudaError_t launch_gemv_batch(const GemvArgs* a, int count, int num_sms, uint32_t* status, cudaStream_t s) {
    GemvBatch b{};
    GemvPlan P;
    if (!plan_batch(a, count, num_sms, &b, &P)) return cudaErrorInvalidValue;
    for (int i = 0; i < count; ++i) {
        GemvLin& L = b.lin[i];
        L.x = a[i].x;
        L.a_q = a[i].a_q;
        L.s_a = a[i].s_a;
        L.rs = a[i].rs;
        L.wq = a[i].wq;
        L.s_w = a[i].s_w;
        L.z_w = a[i].z_w;
        L.bias = a[i].bias;
        L.out = a[i].out;
        L.N = a[i].N;
        L.K = a[i].K;
    }
    b.count = count;
    b.quantize = a[0].x != nullptr;
    b.early = a[0].early;
    switch (a[0].M) {
        case 1: return launch_mt<1>(b, P, status, s);
        case 2: return launch_mt<2>(b, P, status, s);
        case 3: return launch_mt<3>(b, P, status, s);
        case 4: return launch_mt<4>(b, P, status, s);
        case 5: return launch_mt<5>(b, P, status, s);
        case 6: return launch_mt<6>(b, P, status, s);
        case 7: return launch_mt<7>(b, P, status, s);
        default: return launch_mt<8>(b, P, status, s);
    }
}

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, uint32_t* status, cudaStream_t s) {
    return launch_gemv_batch(&a, 1, num_sms, status, s);
}

}  // namespace w4a8
