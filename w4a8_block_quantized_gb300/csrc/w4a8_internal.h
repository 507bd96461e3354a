// w4a8_internal.h -- declarations shared by the CUDA translation units of the library
// (host side: workspace layout, kernel argument blocks, launchers).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4a8 {

// Where and how an epilogue stores y: clamp(s_a * sum + bias, lo, hi) as fp32 or bf16
// (round to nearest even).  lo = -inf, hi = +inf store the value unchanged.
struct OutSpec {
    void* y = nullptr;  // [M][N] fp32 or bf16
    int bf16 = 0;
    float lo = -__builtin_huge_valf(), hi = __builtin_huge_valf();
};

// Bits of the per-device status word (a kernel ORs them in; the host reads and clears).
constexpr uint32_t kStatusTimeout = 1u;

constexpr int kBlock = 64;     // weights per (s_w, z_w) pair along K
constexpr int kTileW = 128;    // GEMM tile weight rows (output columns n) = TMEM lanes = MMA M
constexpr int kTileT = 128;    // GEMM tile tokens = MMA N

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline size_t align_ws(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Operand records: the GEMM moves each (tile, 64-block) operand with one bulk copy, so the
// producers write it in shared-memory order.
//
// Token record (144 TW bytes) for tokens TW t .. TW t + TW - 1 and block b, row r = m % TW:
//   [0, 128 TW)         the two e4m3 nibble planes of section 3 eq. (3) in the 128-byte-swizzled
//                       K-major layout: row r at 128 r; its 16-byte chunk c (c < 4: e4m3(16*(a>>4))
//                       for k = 16c .. 16c+15 of the block, c >= 4: e4m3(a & 15) for k = 16(c-4) ..)
//                       stored at chunk position c ^ (r % 8)
//   [128 TW, 144 TW)    row r at 128 TW + 16 r: the block row sum rs = 64*rh + rl (rh = rs >> 6,
//                       rl = rs & 63) as the fp16 pair {rh / 8, rl / 512} then 12 zero bytes, the
//                       token side of the zero-point MMA (exact: |rh| <= 127, 0 <= rl <= 63)
// The record width TW is a function of M alone (token_tile), so the pre-pass and the GEMM
// agree on it without knowing each other's other dimensions.
// Weight record (kWRec bytes) for weight rows 128t .. 128t+127 and block b, row r = n % 128:
//   [0, 8192)       the e4m3 weight operand in the 64-byte-swizzled K-major layout: row r at
//                   64 r, its 16-byte chunk c (k = 16c .. 16c+15) at chunk position c ^ ((r/2) % 4);
//                   the byte of a weight is its u4 code q, the e4m3 encoding of q * 2^-9
//                   (subnormals and the first normal binade share the step 2^-9)
//   [8192, 10240)   row r at 8192 + 16 r: the fp16 pair {-z_w, -z_w} then 12 zero bytes, the
//                   weight side of the zero-point MMA
// Weight scales (read by the epilogue straight from memory): fp32 512 s_w[n,b] (the power
// of two undoes the 2^-9) at [tile][b][r].
// Rows past M or N are not read into any stored output; the weight side writes them as 0.
constexpr int kTokRec = 18432;    // a 128-token record
constexpr int kTokRx = 16384;     // its zero-point rows

// Token tile width: 256 for the large-M contraction (N = 256 MMAs), 128 otherwise.
inline int token_tile(int64_t M) { return M >= 4096 ? 256 : 128; }
constexpr int kWRec = 10240;
constexpr int kWZx = 8192;

// Prepared activations (a caller-owned buffer): token records [ceil(M/TW)][K/64], then
// s_a fp32 [M] (omitted when the caller passes s_a).
struct ActLayout {
    size_t rec = 0, s_a = 0, total = 0;
    int64_t tiles = 0;
    int tw = 128;
};

inline ActLayout act_layout(int64_t M, int64_t K, bool with_sa, int tw) {
    ActLayout L;
    L.tw = tw;
    L.tiles = (M + tw - 1) / tw;
    size_t off = align_ws(static_cast<size_t>(L.tiles) * static_cast<size_t>(K / kBlock) * 144u * static_cast<size_t>(tw));
    if (with_sa) {
        L.s_a = off;
        off = align_ws(off + static_cast<size_t>(M) * 4);
    }
    L.total = off;
    return L;
}

// Prepared weights (a caller-owned buffer): weight records [ceil(N/128)][K/64], then the
// weight scales [ceil(N/128)][K/64][128].
struct WLayout {
    size_t sc = 0, total = 0;
    int64_t tiles = 0;
};

inline WLayout w_layout(int64_t N, int64_t K) {
    WLayout L;
    L.tiles = (N + kTileW - 1) / kTileW;
    const size_t recs = static_cast<size_t>(L.tiles) * static_cast<size_t>(K / kBlock);
    L.sc = align_ws(recs * kWRec);
    L.total = align_ws(L.sc + recs * kTileW * 4);
    return L;
}

// ---------------------------------------------------------------- pre-pass / pack
struct PrepArgs {
    // row job, quantize mode (x != nullptr) or pack mode (a_q_in != nullptr)
    const float* x = nullptr;
    const int8_t* a_q_in = nullptr;
    const int32_t* rs_in = nullptr;  // pack mode: row sums [M][K/64] (may be null: rx left unwritten)
    int64_t M = 0, K = 0;
    int64_t row0 = 0;                // first source row (debug window); outputs start at row 0
    // API-layout outputs (quant_pack)
    int8_t* a_q_out = nullptr;
    float* s_a_out = nullptr;
    int32_t* rs_out = nullptr;
    // GEMM-layout output: token records of width tw
    uint8_t* trec = nullptr;
    int tw = 128;
    // weight job (skipped when wrec == nullptr): rows n_first .. n_first + N - 1 of wq into
    // weight records; the zero-point rows and the scales (sc) only when s_w != nullptr
    const uint8_t* wq = nullptr;
    int64_t n_first = 0;
    const uint16_t* s_w = nullptr;
    const uint16_t* z_w = nullptr;
    int64_t N = 0;
    uint8_t* wrec = nullptr;
    float* sc = nullptr;
};

cudaError_t launch_quant(const PrepArgs& a, cudaStream_t s);  // x -> codes (+ weight job)
cudaError_t launch_pack(const PrepArgs& a, cudaStream_t s);   // a_q -> token records (+ weight job)

// ---------------------------------------------------------------- GEMM
struct GemmArgs {
    int64_t M = 0, N = 0, K = 0;       // output rows / columns (row stride N) and depth
    const uint8_t* trec = nullptr;      // token records [ceil(M/tw)][K/64]
    int tw = 128;                       // token tile (record width): 128 or 256
    int ksplit = 1;                     // 128-token tiles: CTAs (a cluster) sharing one tile's K range
    const uint8_t* wrec = nullptr;      // weight records [ceil(N/128)][K/64]
    const float* sc = nullptr;          // weight scales [ceil(N/128)][K/64][128]
    // packed-weight form (128-token tiles): the caller's wq [N][K/2], s_w and z_w [N][K/64],
    // read by the contraction itself (wmap: a tiled TMA map over wq, filled by the launcher)
    const uint8_t* wq = nullptr;
    const uint16_t* s_w = nullptr;
    const uint16_t* z_w = nullptr;
    int early = 0;                      // the previous kernel in the stream writes none of wq / s_w / z_w
    const float* s_a = nullptr;
    const float* bias = nullptr;
    OutSpec out;                        // y [M][N]
    int32_t* acc = nullptr;             // debug: [M][N][K/64]
    uint32_t* status = nullptr;
    uint64_t wait_limit_ns = 1000000000ull;
    CUtensorMap wmap{};
};

// Persistent launch over ceil(M/tw) x ceil(N/128) output tiles on at most `num_sms` CTAs, from
// weight records (wrec, sc).  With ksplit = 2 (128-token tiles) every tile is shared by a
// cluster of two CTAs, each contracting half of K; the second hands its partial sums to the
// first through distributed shared memory.
cudaError_t launch_gemm(const GemmArgs& a, bool debug, int num_sms, cudaStream_t s);
// The K split for a record contraction of this shape: 2 when its 128-token tiles would leave
// more than half of the SMs idle and K is an even number of at least 32 64-blocks, else 1.
// A function of the uncut call's shape, so every entry point (and every row chunk of the
// host-buffer call, which is told the uncut call's split) sums each output the same way.
int gemm_ksplit(int64_t M, int64_t N, int64_t K, int tw, int num_sms);
// The same contraction with 128-token tiles straight from the packed weights (wq, s_w, z_w): the
// u4 codes are staged by TMA and expanded to the tensor-core operand in shared memory.  With
// `early` set the weights are staged before the previous kernel in the stream has finished.
cudaError_t launch_gemm_packed(const GemmArgs& a, bool debug, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- few-token (decode) form
// Up to kGemvMaxM tokens (and a K whose staged activations fit on chip): the packed weights
// streamed once, integer dot products on the CUDA cores (gemv.cu), activations in the API
// layout (a_q [M][K], s_a [M], rs [M][K/64]).
constexpr int64_t kGemvMaxM = 8;

struct GemvArgs {
    const float* x = nullptr;           // fp32 [M][K]: quantize in the kernel (gemv_quantizes), or
    const int8_t* a_q = nullptr;        // the pre-pass outputs a_q / s_a / rs
    const float* s_a = nullptr;
    const int32_t* rs = nullptr;
    const uint8_t* wq = nullptr;        // [N][K/2]
    const uint16_t* s_w = nullptr;      // fp16 bits [N][K/64]
    const uint16_t* z_w = nullptr;
    const float* bias = nullptr;
    OutSpec out;                        // y [M][N]
    int64_t M = 0, N = 0, K = 0;
    int early = 0;                      // the previous kernel in the stream writes none of wq / s_w / z_w
};

// Scratch of the fused few-token call: the pre-pass outputs in the API layout.
struct DecodeLayout {
    size_t a_q = 0, s_a = 0, rs = 0, total = 0;
};

inline DecodeLayout decode_layout(int64_t M, int64_t K) {
    DecodeLayout L;
    L.s_a = align_ws(static_cast<size_t>(M) * static_cast<size_t>(K));
    L.rs = align_ws(L.s_a + static_cast<size_t>(M) * 4);
    L.total = align_ws(L.rs + static_cast<size_t>(M) * static_cast<size_t>(K / kBlock) * 4);
    return L;
}

// Whether M tokens of depth K fit the weight-streaming kernel (its staged activations and
// at least two weight stages must fit in one CTA's shared memory), and whether it can also
// quantize them itself (every CTA re-reads x from L2, so only for small M * K).
constexpr int64_t kGemvFuseElems = 16384;
bool gemv_supported(int64_t M, int64_t K);
bool gemv_quantizes(int64_t M, int64_t K);

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, uint32_t* status, cudaStream_t s);

// Up to kGemvMaxLinears independent linears of one M in one launch of the weight-streaming
// kernel: every CTA stages (or quantizes) all of their activations, then the CTAs walk the row
// tiles of all of them as one stream.  `early` is taken from the first entry.
constexpr int kGemvMaxLinears = 8;
bool gemv_batch_fits(const GemvArgs* a, int count);
int gemv_tile_rows(const GemvArgs& a, int num_sms);  // the tile height a launch of `a` alone uses (0: none)
cudaError_t launch_gemv_batch(const GemvArgs* a, int count, int num_sms, uint32_t* status, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace w4a8
