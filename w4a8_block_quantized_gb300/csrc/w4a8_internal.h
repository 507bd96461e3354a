// w4a8_internal.h -- declarations shared by the CUDA translation units of the library
// (host side: workspace layout, kernel argument blocks, launchers).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4a8 {

// Bits of the per-device status word (a kernel ORs them in; the host reads and clears).
constexpr uint32_t kStatusTimeout = 1u;

constexpr int kBlock = 64;     // weights per (s_w, z_w) pair along K
constexpr int kTileW = 128;    // GEMM tile weight rows (output columns n) = TMEM lanes
constexpr int kPadM = 256;     // token padding of the transposed row sums (largest token tile)
constexpr int kPadN = 256;     // weight-row padding of the re-laid-out weight scales

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Layout of the prepared activations (a caller-owned buffer):
//   apk : tensor-core activation operand, uint8 [M][2K]; per row and 64-block,
//         64 bytes of e4m3(16 * (a >> 4)) then 64 bytes of e4m3(a & 15)
//   s_a : fp32 [M]                           (omitted when the caller passes s_a)
//   rx  : [K/64][M_pad] x 16 bytes: the block row sum rs = 64*rh + rl (rh = rs >> 6,
//         rl = rs & 63) as the fp16 pair {rh / 8, rl / 512} followed by 12 zero bytes, the
//         K-major operand of the zero-point MMA (exact: |rh| <= 127, 0 <= rl <= 63)
// Layout of the prepared weight scales:
//   wsc : [K/64] x { fp32 [N_pad] 512 s_w[n,b], weight row n at 4*(n % 8) + (n % 32) / 8
//         within its group of 32 rows (an epilogue thread's rows n, n+8, n+16, n+24 in one
//         16-byte vector); fp16x2 [N_pad] {-z_w[n,b], -z_w[n,b]} in row order }, zero past N
inline size_t align_ws(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct ActLayout {
    size_t apk = 0, s_a = 0, rx = 0, total = 0;
    int64_t M_pad = 0;
};

inline ActLayout act_layout(int64_t M, int64_t K, bool with_sa, bool with_rows) {
    ActLayout L;
    const int64_t nb = K / kBlock;
    L.M_pad = round_up(M, kPadM);
    size_t off = 0;
    off = align_ws(off + static_cast<size_t>(M) * static_cast<size_t>(2 * K));
    if (with_sa) {
        L.s_a = off;
        off = align_ws(off + static_cast<size_t>(M) * 4);
    }
    if (with_rows) {
        L.rx = off;
        off = align_ws(off + static_cast<size_t>(nb) * static_cast<size_t>(L.M_pad) * 16);
    }
    L.total = off;
    return L;
}

inline int64_t n_pad(int64_t N) { return round_up(N, kPadN); }

inline size_t wsc_bytes(int64_t N, int64_t K) {
    return align_ws(static_cast<size_t>(K / kBlock) * static_cast<size_t>(n_pad(N)) * 8);
}

// ---------------------------------------------------------------- pre-pass / pack
struct PrepArgs {
    // row job, quantize mode (x != nullptr) or pack mode (a_q_in != nullptr)
    const float* x = nullptr;
    const int8_t* a_q_in = nullptr;
    const int32_t* rs_in = nullptr;  // pack mode: row sums [M][K/64] to re-lay out (may be null)
    int64_t M = 0, K = 0;
    int64_t row0 = 0;                // first source row (debug window); outputs start at row 0
    // API-layout outputs (quant_pack)
    int8_t* a_q_out = nullptr;
    float* s_a_out = nullptr;
    int32_t* rs_out = nullptr;
    // GEMM-layout outputs
    uint8_t* apk = nullptr;
    uint4* rx = nullptr;
    int64_t M_pad = 0;
    // weight-scale job (skipped when sz == nullptr)
    const uint16_t* s_w = nullptr;
    const uint16_t* z_w = nullptr;
    int64_t N = 0, N_pad = 0;
    float* wsc = nullptr;
};

cudaError_t launch_quant(const PrepArgs& a, cudaStream_t s);  // x -> codes (+ scales job)
cudaError_t launch_pack(const PrepArgs& a, cudaStream_t s);   // a_q -> apk (+ rx, scales)

// ---------------------------------------------------------------- GEMM
struct GemmArgs {
    int64_t M = 0, N = 0, K = 0;       // full problem (N, K) and rows in the operand map
    int64_t m_cnt = 0, n0 = 0, n_cnt = 0;  // rows [0, m_cnt) of apk, columns [n0, n0 + n_cnt)
    int64_t M_pad = 0, N_pad = 0;
    const float* wsc = nullptr;
    const uint4* rx = nullptr;
    const float* s_a = nullptr;
    const float* bias = nullptr;
    float* y = nullptr;                 // [M][N], row stride N
    int32_t* acc = nullptr;             // debug: [m_cnt][n_cnt][K/64]
    uint32_t* status = nullptr;
    uint64_t wait_limit_ns = 1000000000ull;
};

struct GemmMaps {
    CUtensorMap a;  // apk (tokens), uint8 [rows][2K], box 128 x TN, 128-byte swizzle
    CUtensorMap b;  // wq (weights), uint8 [N][K/2], box 32 x 128, no swizzle
};

// Token-tile width TN (the MMA's N) for a problem: 256, 128 or 64.
int pick_token_tile(int64_t m_cnt, int64_t n_cnt, int num_sms);
cudaError_t launch_gemm(const GemmMaps& maps, const GemmArgs& a, int tn, bool debug, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace w4a8
