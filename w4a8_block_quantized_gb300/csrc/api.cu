// api.cu -- the C ABI declared in include/w4a8.h: argument validation, workspace
// carving, routing by shape and kernel launches.  Nothing here allocates memory; the
// host-buffer call keeps a few streams and events per device, created on first use.
#include "../../include/w4a8.h"
#include "w4a8_internal.h"

#include <algorithm>
#include <cstring>
#include <mutex>

namespace w4a8 {
namespace {

__device__ uint32_t g_status;  // per-device status word (kernels OR kStatus* bits in)

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool checked = false;
    bool ok = false;
    int num_sms = 0;
    uint32_t* status = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

// Validates the current device once (sm_103) and resolves the status word's address.
int current_device(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4A8_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.checked) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return W4A8_ERR_CUDA;
        d.ok = (major == 10 && minor == 3);
        if (d.ok) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return W4A8_ERR_CUDA;
            d.status = static_cast<uint32_t*>(p);
        }
        d.checked = true;
    }
    if (!d.ok) return W4A8_ERR_DEVICE;
    *out = &d;
    return W4A8_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxDim = 2147483647LL;

int check_shape(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0) return W4A8_ERR_ARG;
    if (K <= 0 || K % kBlock != 0) return W4A8_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return W4A8_ERR_SHAPE;
    // the kernels' 32-bit row offsets (K/2 bytes per packed weight row) and row counts stay in range
    if (2 * K > kMaxDim || N > (int64_t(1) << 31)) return W4A8_ERR_SHAPE;
    // the GEMM counts its 64-blocks (output tiles x K/64) in 32 bits
    const int64_t tiles = ((M + kTileT - 1) / kTileT) * ((N + kTileW - 1) / kTileW);
    if (tiles > kMaxDim / (K / kBlock)) return W4A8_ERR_SHAPE;
    return W4A8_OK;
}

// Whether w4a8_linear_act contracts from the packed weights themselves (128-token tiles: the
// GEMM stages the u4 codes and expands them in shared memory, no workspace) or from weight
// records written into its workspace first (256-token tiles).
bool packed_form(int64_t M) { return token_tile(M) == kTileT; }

// Workspace of the one-call entry points: prepared activations, then prepared weights.
struct CallLayout {
    ActLayout act;
    WLayout w;
    size_t w_off = 0, total = 0;
};

CallLayout call_layout(int64_t M, int64_t N, int64_t K, bool with_sa, int tw) {
    CallLayout c;
    c.act = act_layout(M, K, with_sa, tw);
    c.w = w_layout(N, K);
    c.w_off = c.act.total;
    c.total = c.w_off + c.w.total;
    return c;
}

// The token-record width (and so the contraction kernel) of the one-call entry points
// (w4a8_prefill_linear, also as a one-chunk host-buffer call; w4a8_linear; the debug call) for
// a problem of this shape: 256 from 4096 tokens on; below that, 256 where 128-token tiles would take more waves of
// the SMs and run without the K split.  Per token the 256-token kernel takes about 4/5 of the
// 128-token kernel's time (measured at 8192 tokens), so a wave of it counts as 1.6 of a
// 128-token wave.  Measured on 512 tokens, K 2048 -> N 6144 (192 tiles of 128 tokens, 96 of
// 256): the contraction alone 34.1 -> 26.6 us.  Without the K split both kernels sum every
// output in the same order, so the width changes no output: the prepared-operand entry points,
// which keep token_tile(M), give the same results bit for bit.
int call_tile(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (token_tile(M) != kTileT) return token_tile(M);
    if (num_sms < 1 || gemm_ksplit(M, N, K, kTileT, num_sms) > 1) return kTileT;
    const int64_t tn = (N + kTileW - 1) / kTileW;
    const int64_t w128 = ((M + 127) / 128 * tn + num_sms - 1) / num_sms;
    const int64_t w256 = ((M + 255) / 256 * tn + num_sms - 1) / num_sms;
    return w256 * 256 * 4 < w128 * 128 * 5 ? 256 : kTileT;
}

// GEMM + epilogue from prepared activations (token records `tw` tokens wide) and prepared
// weights.  Each output depends only on its own row, the kernel the width selects and the K
// split (`ksplit`, by default the one of this shape: gemm_ksplit), so rows cut into whole tiles
// of one width and run with the uncut call's split give the uncut call's outputs.
int run_linear(const uint8_t* trec, const float* s_a, const uint8_t* pw, const float* bias, const OutSpec& out,
               int64_t M, int64_t N, int64_t K, int tw, const DeviceInfo& d, cudaStream_t st, int ksplit = 0) {
    const WLayout W = w_layout(N, K);
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.trec = trec;
    g.tw = tw;
    g.wrec = pw;
    g.sc = reinterpret_cast<const float*>(pw + W.sc);
    g.s_a = s_a;
    g.bias = bias;
    g.out = out;
    g.status = d.status;
    g.ksplit = ksplit > 0 ? ksplit : gemm_ksplit(M, N, K, tw, d.num_sms);
    return launch_gemm(g, false, d.num_sms, st) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

// GEMM + epilogue from prepared activations (128-token records) and the caller's packed
// weights, expanded inside the contraction.  `early`: the previous kernel in the stream is the
// call's own pre-pass, which writes none of the weights, so the GEMM may stage them before it
// has finished.  Each output equals run_linear's from weights prepared from the same arrays.
int run_linear_packed(const uint8_t* trec, const float* s_a, const uint8_t* wq, const uint16_t* w_scale,
                      const uint16_t* w_zero, const float* bias, const OutSpec& out, int64_t M, int64_t N, int64_t K,
                      bool early, const DeviceInfo& d, cudaStream_t st) {
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.trec = trec;
    g.tw = kTileT;
    g.wq = wq;
    g.s_w = w_scale;
    g.z_w = w_zero;
    g.early = early ? 1 : 0;
    g.s_a = s_a;
    g.bias = bias;
    g.out = out;
    g.status = d.status;
    g.ksplit = gemm_ksplit(M, N, K, kTileT, d.num_sms);  // as the record form of this shape
    return launch_gemm_packed(g, false, d.num_sms, st) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

// Weight job arguments: all N rows of wq into the weight records at `wrec`.
void set_weight_job(PrepArgs* p, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero, int64_t N,
                    int64_t K, uint8_t* wrec) {
    p->K = K;
    p->wq = wq;
    p->n_first = 0;
    p->s_w = w_scale;
    p->z_w = w_zero;
    p->N = N;
    p->wrec = wrec;
    p->sc = reinterpret_cast<float*>(wrec + w_layout(N, K).sc);
}

// Scratch bytes of the two workspace-taking entry points.  The few-token form needs none
// for w4a8_linear, and for the fused call none when the kernel quantizes the rows itself,
// else the pre-pass outputs; the tensor-core form needs the re-encoded activations and the
// prepared weights.
bool few_tokens(int64_t M, int64_t K) { return M <= kGemvMaxM && gemv_supported(M, K); }
// (The tensor-core form's size covers either token-record width, so it does not depend on the
// device.)
size_t call_ws(int64_t M, int64_t N, int64_t K, bool with_sa) {
    return std::max(call_layout(M, N, K, with_sa, kTileT).total, call_layout(M, N, K, with_sa, 256).total);
}
size_t linear_ws(int64_t M, int64_t N, int64_t K) { return few_tokens(M, K) ? 0 : call_ws(M, N, K, false); }
size_t prefill_ws(int64_t M, int64_t N, int64_t K) {
    if (few_tokens(M, K)) return gemv_quantizes(M, K) ? 0 : decode_layout(M, K).total;
    return call_ws(M, N, K, true);
}

// The few-token kernel from x (it quantizes) or from the pre-pass outputs.
int run_gemv(const float* x, const int8_t* a_q, const float* s_a, const int32_t* rs, const uint8_t* wq,
             const uint16_t* w_scale, const uint16_t* w_zero, const float* bias, const OutSpec& out, int64_t M,
             int64_t N, int64_t K, const DeviceInfo& d, cudaStream_t st, bool early = false) {
    GemvArgs g;
    g.early = early ? 1 : 0;
    g.x = x;
    g.a_q = a_q;
    g.s_a = s_a;
    g.rs = rs;
    g.wq = wq;
    g.s_w = w_scale;
    g.z_w = w_zero;
    g.bias = bias;
    g.out = out;
    g.M = M;
    g.N = N;
    g.K = K;
    return launch_gemv(g, d.num_sms, d.status, st) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

OutSpec f32_out(float* y) {
    OutSpec o;
    o.y = y;
    return o;
}

// The output spec of the *_ex entry points: a known dtype and lo <= hi (no NaN).
int make_out(void* y, int out_dtype, float lo, float hi, OutSpec* o) {
    if (out_dtype != W4A8_OUT_F32 && out_dtype != W4A8_OUT_BF16) return W4A8_ERR_ARG;
    if (!(lo <= hi)) return W4A8_ERR_ARG;
    o->y = y;
    o->bf16 = out_dtype == W4A8_OUT_BF16;
    o->lo = lo;
    o->hi = hi;
    return W4A8_OK;
}

int linear_impl(const int8_t* a_q, const float* a_scale, const int32_t* rowsum, const uint8_t* wq,
                const uint16_t* w_scale, const uint16_t* w_zero, const float* bias, const OutSpec& out, int64_t M,
                int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream);
int prefill_impl(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                 const float* bias, const OutSpec& out, int64_t M, int64_t N, int64_t K, void* workspace,
                 size_t workspace_bytes, void* stream, bool after_own = false);
int prefill_check(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                  const float* bias, const void* y, int64_t M, int64_t N, int64_t K, const void* workspace,
                  size_t workspace_bytes);
int linear_prepared_impl(const void* act, const void* pw, const float* bias, const OutSpec& out, int64_t M,
                         int64_t N, int64_t K, void* stream);

}  // namespace
}  // namespace w4a8

using namespace w4a8;

extern "C" {

int w4a8_abi_version(void) { return 204; }

const char* w4a8_status_string(int status) {
    switch (status) {
        case W4A8_OK: return "ok";
        case W4A8_ERR_ARG: return "invalid argument (null pointer or negative size)";
        case W4A8_ERR_ALIGN: return "pointer misaligned";
        case W4A8_ERR_SHAPE: return "unsupported shape (K must be a positive multiple of 64)";
        case W4A8_ERR_CUDA: return "CUDA error";
        case W4A8_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
        case W4A8_ERR_WORKSPACE: return "workspace missing or too small";
        case W4A8_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case W4A8_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the static no-alloc buffer holds";
        default: return "unknown status";
    }
}

size_t w4a8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (check_shape(M, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0 || N == 0) return 0;
    return linear_ws(M, N, K);
}

size_t w4a8_prefill_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (check_shape(M, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0 || N == 0) return 0;
    return prefill_ws(M, N, K);
}

// Sized for the wider token records, which never take less room than the 128-token ones, so
// one size serves the window whatever the full problem's M selects.
size_t w4a8_debug_workspace_bytes(int64_t m_cnt, int64_t n_cnt, int64_t K) {
    if (check_shape(m_cnt, n_cnt, K) != W4A8_OK || m_cnt == 0 || n_cnt == 0) return static_cast<size_t>(-1);
    return act_layout(m_cnt, K, false, 256).total + w_layout(n_cnt, K).total;
}

size_t w4a8_prepared_activations_bytes(int64_t M, int64_t K) {
    if (check_shape(M, 1, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0) return 0;
    return act_layout(M, K, true, token_tile(M)).total;
}

size_t w4a8_prepared_weights_bytes(int64_t N, int64_t K) {
    if (check_shape(1, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (N == 0) return 0;
    return w_layout(N, K).total;
}

int w4a8_quant_pack(const float* x, int64_t M, int64_t K, int8_t* a_q, float* a_scale, int32_t* rowsum,
                    void* stream) {
    int rc = check_shape(M, 1, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0) return W4A8_OK;
    if (!x || !a_q || !a_scale || !rowsum) return W4A8_ERR_ARG;
    if (!aligned(x, 16) || !aligned(a_q, 16) || !aligned(a_scale, 4) || !aligned(rowsum, 4)) return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    PrepArgs p;
    p.x = x;
    p.M = M;
    p.K = K;
    p.a_q_out = a_q;
    p.s_a_out = a_scale;
    p.rs_out = rowsum;
    return launch_quant(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int w4a8_linear(const int8_t* a_q, const float* a_scale, const int32_t* rowsum, const uint8_t* wq,
                const uint16_t* w_scale, const uint16_t* w_zero, const float* bias, float* y, int64_t M, int64_t N,
                int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    return linear_impl(a_q, a_scale, rowsum, wq, w_scale, w_zero, bias, f32_out(y), M, N, K, workspace,
                       workspace_bytes, stream);
}

int w4a8_linear_ex(const int8_t* a_q, const float* a_scale, const int32_t* rowsum, const uint8_t* wq,
                   const uint16_t* w_scale, const uint16_t* w_zero, const float* bias, void* y, int out_dtype,
                   float clamp_lo, float clamp_hi, int64_t M, int64_t N, int64_t K, void* workspace,
                   size_t workspace_bytes, void* stream) {
    OutSpec o;
    const int rc = make_out(y, out_dtype, clamp_lo, clamp_hi, &o);
    if (rc != W4A8_OK) return rc;
    return linear_impl(a_q, a_scale, rowsum, wq, w_scale, w_zero, bias, o, M, N, K, workspace, workspace_bytes,
                       stream);
}

}  // extern "C"

namespace w4a8 {
namespace {

int linear_impl(const int8_t* a_q, const float* a_scale, const int32_t* rowsum, const uint8_t* wq,
                const uint16_t* w_scale, const uint16_t* w_zero, const float* bias, const OutSpec& out, int64_t M,
                int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!a_q || !a_scale || !rowsum || !wq || !w_scale || !w_zero || !out.y) return W4A8_ERR_ARG;
    if (!aligned(a_q, 16) || !aligned(wq, 16) || !aligned(out.y, 16) || !aligned(a_scale, 4) || !aligned(rowsum, 4) ||
        !aligned(w_scale, 2) || !aligned(w_zero, 2) || (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (few_tokens(M, K)) {
        // few-token form: no scratch, the workspace is not touched
        if ((rc = current_device(&d)) != W4A8_OK) return rc;
        return run_gemv(nullptr, a_q, a_scale, rowsum, wq, w_scale, w_zero, bias, out, M, N, K, *d, st);
    }
    if (!workspace || workspace_bytes < linear_ws(M, N, K)) return W4A8_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    const CallLayout L = call_layout(M, N, K, false, call_tile(M, N, K, d->num_sms));
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    PrepArgs p;
    p.a_q_in = a_q;
    p.rs_in = rowsum;
    p.M = M;
    p.K = K;
    p.trec = ws + L.act.rec;
    p.tw = L.act.tw;
    set_weight_job(&p, wq, w_scale, w_zero, N, K, ws + L.w_off);
    if (launch_pack(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    return run_linear(ws + L.act.rec, a_scale, ws + L.w_off, bias, out, M, N, K, L.act.tw, *d, st);
}

// Argument checks of the fused call (everything but the device).
int prefill_check(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                  const float* bias, const void* y, int64_t M, int64_t N, int64_t K, const void* workspace,
                  size_t workspace_bytes) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!x || !wq || !w_scale || !w_zero || !y) return W4A8_ERR_ARG;
    if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(w_scale, 2) || !aligned(w_zero, 2) ||
        (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    const size_t need = prefill_ws(M, N, K);
    if (need > 0 && (!workspace || workspace_bytes < need)) return W4A8_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    return W4A8_OK;
}

// `after_own`: the previous kernel in the stream is one of this library's, which never writes
// the caller's weights, so a few-token kernel may start streaming them before it has finished.
int prefill_impl(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                 const float* bias, const OutSpec& out, int64_t M, int64_t N, int64_t K, void* workspace,
                 size_t workspace_bytes, void* stream, bool after_own) {
    int rc = prefill_check(x, wq, w_scale, w_zero, bias, out.y, M, N, K, workspace, workspace_bytes);
    if (rc != W4A8_OK || M == 0 || N == 0) return rc;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (few_tokens(M, K) && gemv_quantizes(M, K)) {
        // few-token form, one launch: the weight-streaming kernel quantizes x itself
        return run_gemv(x, nullptr, nullptr, nullptr, wq, w_scale, w_zero, bias, out, M, N, K, *d, st, after_own);
    }
    if (few_tokens(M, K)) {
        // few-token form: the pre-pass in the API layout, then the weight-streaming kernel
        const DecodeLayout D = decode_layout(M, K);
        PrepArgs p;
        p.x = x;
        p.M = M;
        p.K = K;
        p.a_q_out = reinterpret_cast<int8_t*>(ws + D.a_q);
        p.s_a_out = reinterpret_cast<float*>(ws + D.s_a);
        p.rs_out = reinterpret_cast<int32_t*>(ws + D.rs);
        if (launch_quant(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
        // the previous kernel is the pre-pass: the weights may stream while it runs
        return run_gemv(nullptr, p.a_q_out, p.s_a_out, p.rs_out, wq, w_scale, w_zero, bias, out, M, N, K, *d, st,
                        true);
    }
    const CallLayout L = call_layout(M, N, K, true, call_tile(M, N, K, d->num_sms));
    float* s_a = reinterpret_cast<float*>(ws + L.act.s_a);
    PrepArgs p;
    p.x = x;
    p.M = M;
    p.K = K;
    p.s_a_out = s_a;
    p.trec = ws + L.act.rec;
    p.tw = L.act.tw;
    set_weight_job(&p, wq, w_scale, w_zero, N, K, ws + L.w_off);
    if (launch_quant(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    return run_linear(ws + L.act.rec, s_a, ws + L.w_off, bias, out, M, N, K, L.act.tw, *d, st);
}

int linear_prepared_impl(const void* act, const void* pw, const float* bias, const OutSpec& out, int64_t M,
                         int64_t N, int64_t K, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!act || !pw || !out.y) return W4A8_ERR_ARG;
    if (!aligned(act, 16) || !aligned(pw, 16) || !aligned(out.y, 16) || (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    const ActLayout A = act_layout(M, K, true, token_tile(M));
    const uint8_t* a = static_cast<const uint8_t*>(act);
    return run_linear(a + A.rec, reinterpret_cast<const float*>(a + A.s_a), static_cast<const uint8_t*>(pw), bias,
                      out, M, N, K, A.tw, *d, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace w4a8

extern "C" {

int w4a8_prefill_linear(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                        const float* bias, float* y, int64_t M, int64_t N, int64_t K, void* workspace,
                        size_t workspace_bytes, void* stream) {
    return prefill_impl(x, wq, w_scale, w_zero, bias, f32_out(y), M, N, K, workspace, workspace_bytes, stream);
}

int w4a8_prefill_linear_ex(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                           const float* bias, void* y, int out_dtype, float clamp_lo, float clamp_hi, int64_t M,
                           int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    OutSpec o;
    const int rc = make_out(y, out_dtype, clamp_lo, clamp_hi, &o);
    if (rc != W4A8_OK) return rc;
    return prefill_impl(x, wq, w_scale, w_zero, bias, o, M, N, K, workspace, workspace_bytes, stream);
}

int w4a8_prefill_linear_batch(const w4a8_linear_ref* linears, int64_t count, int64_t M, void* stream) {
    if (count < 0 || (count > 0 && !linears)) return W4A8_ERR_ARG;
    // every entry is checked before anything is launched
    for (int64_t i = 0; i < count; ++i) {
        const w4a8_linear_ref& l = linears[i];
        const int rc = prefill_check(l.x, l.wq, l.w_scale, l.w_zero, l.bias, l.y, M, l.N, l.K, l.workspace,
                                     l.workspace_bytes);
        if (rc != W4A8_OK) return rc;
    }
    // Few tokens, every entry quantized by the weight-streaming kernel itself: one launch for
    // all of them when their activations fit one CTA and each entry's own launch would give
    // every output row one warp (then the sums run in the same order, and the outputs are those
    // of separate calls bit for bit).  The start-up cost of a launch is then paid once.
    // In one launch every CTA reads every entry's x before it writes any y, but CTAs run at
    // different times: so no y may overlap an x or another y (an entry that reads an earlier
    // entry's output takes the launch-per-entry path, where each kernel waits for the last).
    auto overlap = [](const void* a, size_t an, const void* b, size_t bn) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
        return a0 < b0 + bn && b0 < a0 + an;
    };
    bool disjoint = true;
    for (int64_t i = 0; i < count && disjoint; ++i) {
        const w4a8_linear_ref& yi = linears[i];
        const size_t ybytes = static_cast<size_t>(M) * static_cast<size_t>(yi.N) * 4u;
        for (int64_t j = 0; j < count && disjoint; ++j) {
            const w4a8_linear_ref& lj = linears[j];
            const size_t xbytes = static_cast<size_t>(M) * static_cast<size_t>(lj.K) * 4u;
            const size_t yjb = static_cast<size_t>(M) * static_cast<size_t>(lj.N) * 4u;
            disjoint = !overlap(yi.y, ybytes, lj.x, xbytes) && (i == j || !overlap(yi.y, ybytes, lj.y, yjb));
        }
    }
    if (disjoint && M >= 1 && M <= kGemvMaxM && count >= 1 && count <= kGemvMaxLinears) {
        GemvArgs g[kGemvMaxLinears];
        int n = 0;
        bool one = true;
        int64_t wbytes = 0;  // packed weights of all entries
        DeviceInfo* d = nullptr;
        int rc = current_device(&d);
        if (rc != W4A8_OK) return rc;
        for (int64_t i = 0; i < count && one; ++i) {
            const w4a8_linear_ref& l = linears[i];
            if (l.N == 0) continue;
            one = few_tokens(M, l.K) && gemv_quantizes(M, l.K);
            GemvArgs& a = g[n++];
            a.x = l.x;
            a.wq = l.wq;
            a.s_w = l.w_scale;
            a.z_w = l.w_zero;
            a.bias = l.bias;
            a.out = f32_out(l.y);
            a.M = M;
            a.N = l.N;
            a.K = l.K;
            wbytes += l.N * (l.K / 2);
            one = one && gemv_tile_rows(a, d->num_sms) >= 8;
        }
        // Measured (one token unless noted), a launch per entry -> one launch: a decoder layer's
        // seven linears 35 -> 21 us; pairs of 3 MB of weights (1024-deep) 14.3 -> 10.2, of
        // 12.6 MB (2048/6144-deep) 18.4 -> 14.3, two 2048-deep linears at four tokens
        // 20.5 -> 14.3; but the 7B-class pair (58.7 MB) 27.2 -> 28.8 on one box, where each of
        // two launches has every SM and the second streams its weights during the first's tail.
        // So one launch from three entries on, or for a pair of at most 24 MiB of weights.
        if (one && (n >= 3 || (n == 2 && wbytes <= (int64_t(24) << 20))) && gemv_batch_fits(g, n))
            return launch_gemv_batch(g, n, d->num_sms, d->status, static_cast<cudaStream_t>(stream)) == cudaSuccess
                       ? W4A8_OK
                       : W4A8_ERR_CUDA;
    }
    bool launched = false;  // a kernel of this call is the previous one in the stream
    for (int64_t i = 0; i < count; ++i) {
        const w4a8_linear_ref& l = linears[i];
        if (M == 0 || l.N == 0) continue;
        const int rc = prefill_impl(l.x, l.wq, l.w_scale, l.w_zero, l.bias, f32_out(l.y), M, l.N, l.K, l.workspace,
                                    l.workspace_bytes, stream, launched);
        if (rc != W4A8_OK) return rc;
        launched = true;
    }
    return W4A8_OK;
}

int w4a8_prepare_activations(const float* x, int64_t M, int64_t K, void* act, size_t act_bytes, void* stream) {
    int rc = check_shape(M, 1, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0) return W4A8_OK;
    if (!x || !act) return W4A8_ERR_ARG;
    if (!aligned(x, 16) || !aligned(act, 16)) return W4A8_ERR_ALIGN;
    const ActLayout A = act_layout(M, K, true, token_tile(M));
    if (act_bytes < A.total) return W4A8_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    uint8_t* a = static_cast<uint8_t*>(act);
    PrepArgs p;
    p.x = x;
    p.M = M;
    p.K = K;
    p.s_a_out = reinterpret_cast<float*>(a + A.s_a);
    p.trec = a + A.rec;
    p.tw = A.tw;
    return launch_quant(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int w4a8_prepare_weights(const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero, int64_t N, int64_t K,
                         void* pw, size_t pw_bytes, void* stream) {
    int rc = check_shape(1, N, K);
    if (rc != W4A8_OK) return rc;
    if (N == 0) return W4A8_OK;
    if (!wq || !w_scale || !w_zero || !pw) return W4A8_ERR_ARG;
    if (!aligned(wq, 16) || !aligned(w_scale, 2) || !aligned(w_zero, 2) || !aligned(pw, 16)) return W4A8_ERR_ALIGN;
    const WLayout W = w_layout(N, K);
    if (pw_bytes < W.total) return W4A8_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    PrepArgs p;
    p.M = 0;
    set_weight_job(&p, wq, w_scale, w_zero, N, K, static_cast<uint8_t*>(pw));
    return launch_pack(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int w4a8_linear_prepared(const void* act, const void* pw, const float* bias, float* y, int64_t M, int64_t N,
                         int64_t K, void* stream) {
    return linear_prepared_impl(act, pw, bias, f32_out(y), M, N, K, stream);
}

size_t w4a8_linear_act_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (check_shape(M, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0 || N == 0 || packed_form(M)) return 0;
    return w_layout(N, K).total;
}

int w4a8_linear_act(const void* act, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                    const float* bias, float* y, int64_t M, int64_t N, int64_t K, void* workspace,
                    size_t workspace_bytes, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!act || !wq || !w_scale || !w_zero || !y) return W4A8_ERR_ARG;
    if (!aligned(act, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(w_scale, 2) || !aligned(w_zero, 2) ||
        (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    const size_t need = w4a8_linear_act_workspace_bytes(M, N, K);
    if (need > 0 && (!workspace || workspace_bytes < need)) return W4A8_ERR_WORKSPACE;
    if (need > 0 && !aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ActLayout A = act_layout(M, K, true, token_tile(M));
    const uint8_t* a = static_cast<const uint8_t*>(act);
    const float* s_a = reinterpret_cast<const float*>(a + A.s_a);
    if (packed_form(M)) {
        // the previous kernel in the stream may have written the weights: no early staging
        return run_linear_packed(a + A.rec, s_a, wq, w_scale, w_zero, bias, f32_out(y), M, N, K, false, *d, st);
    }
    uint8_t* wrec = static_cast<uint8_t*>(workspace);
    PrepArgs p;
    p.M = 0;
    set_weight_job(&p, wq, w_scale, w_zero, N, K, wrec);
    if (launch_pack(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    return run_linear(a + A.rec, s_a, wrec, bias, f32_out(y), M, N, K, A.tw, *d, st);
}

int w4a8_linear_prepared_ex(const void* act, const void* pw, const float* bias, void* y, int out_dtype,
                            float clamp_lo, float clamp_hi, int64_t M, int64_t N, int64_t K, void* stream) {
    OutSpec o;
    const int rc = make_out(y, out_dtype, clamp_lo, clamp_hi, &o);
    if (rc != W4A8_OK) return rc;
    return linear_prepared_impl(act, pw, bias, o, M, N, K, stream);
}

int w4a8_debug_block_acc(const int8_t* a_q, const uint8_t* wq, int64_t M, int64_t N, int64_t K, int64_t m0,
                         int64_t m_cnt, int64_t n0, int64_t n_cnt, int32_t* acc, void* workspace,
                         size_t workspace_bytes, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (!a_q || !wq || !acc) return W4A8_ERR_ARG;
    if (m0 < 0 || n0 < 0 || m_cnt <= 0 || n_cnt <= 0 || m0 + m_cnt > M || n0 + n_cnt > N) return W4A8_ERR_SHAPE;
    if (!aligned(a_q, 16) || !aligned(wq, 16) || !aligned(acc, 4)) return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    // the token-record width (and so the contraction kernel) that w4a8_linear runs for this problem
    const ActLayout L = act_layout(m_cnt, K, false, call_tile(M, N, K, d->num_sms));
    const WLayout W = w_layout(n_cnt, K);
    if (!workspace || workspace_bytes < w4a8_debug_workspace_bytes(m_cnt, n_cnt, K)) return W4A8_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t* wrec = ws + L.total;
    // the window's token rows re-encoded, its weight rows expanded (no scales or zeros)
    PrepArgs p;
    p.a_q_in = a_q;
    p.M = m_cnt;
    p.K = K;
    p.row0 = m0;
    p.trec = ws + L.rec;
    p.tw = L.tw;
    p.wq = wq;
    p.n_first = n0;
    p.N = n_cnt;
    p.wrec = wrec;
    if (launch_pack(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    GemmArgs g;
    g.M = m_cnt;
    g.N = n_cnt;
    g.K = K;
    g.trec = ws + L.rec;
    g.tw = L.tw;
    g.wrec = wrec;
    g.acc = acc;
    g.status = d->status;
    return launch_gemm(g, true, d->num_sms, st) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int w4a8_sync_status(void* stream) {
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != W4A8_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return W4A8_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return W4A8_ERR_CUDA;
    if (v != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return W4A8_ERR_CUDA;
    }
    return (v & kStatusTimeout) ? W4A8_ERR_TIMEOUT : W4A8_OK;
}

int w4a8_selftest_wait_timeout(int64_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return W4A8_ERR_ARG;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != W4A8_OK) return rc;
    return launch_wait_selftest(d->status, static_cast<uint64_t>(limit_us) * 1000ull,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free variant
// Scratch of w4a8_prefill_linear_noalloc: reserved statically on every device the library
// is loaded on.  Host code must not use the array's name as an address (on the host it is
// only a stand-in for the device symbol); the device address comes from
// cudaGetSymbolAddress, resolved once per device with that device current.
namespace w4a8 {
namespace {
static __device__ __align__(256) uint8_t g_noalloc_scratch[W4A8_NOALLOC_SCRATCH_BYTES];
uint8_t* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

int noalloc_scratch(uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4A8_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return W4A8_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return W4A8_OK;
}
}  // namespace
}  // namespace w4a8

extern "C" {

int w4a8_prefill_linear_noalloc(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                                const float* bias, float* y, int64_t M, int64_t N, int64_t K, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (prefill_ws(M, N, K) > W4A8_NOALLOC_SCRATCH_BYTES) return W4A8_ERR_SCRATCH_LIMIT;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    uint8_t* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != W4A8_OK) return rc;
    return w4a8_prefill_linear(x, wq, w_scale, w_zero, bias, y, M, N, K, scratch, W4A8_NOALLOC_SCRATCH_BYTES,
                               stream);
}

}  // extern "C"

// ---------------------------------------------------------------- host-buffer call
// w4a8_prefill_linear_host: x and y in page-locked host memory.  The rows are cut into chunks
// so that the copy of chunk c+1 to the device, the linear on chunk c and the copy of chunk
// c-1 back run at the same time: one stream carries the host-to-device copies in row order,
// one the device-to-host copies, and the chunks' pre-passes and contractions rotate over
// kHostStreams streams of their own (a chunk's GEMM covers a part of the SMs; concurrent
// chunks fill the rest).  The weights are prepared once, on the caller's stream, while the
// first chunk is copied in.  Chunks are whole token tiles of the width the uncut call would
// use, and the GEMM is told that width, so chunking changes no output (the prepared form
// gives the fused call's results bit for bit).  A chunk moves at least kHostChunkBytes of x
// and y: below that the fixed cost of a copy and a launch outweighs the overlap, and a call
// too small for two chunks works on mapped host buffers in place instead.
namespace w4a8 {
namespace {

constexpr int kHostChunks = 16;
constexpr int kHostStreams = 4;
constexpr int64_t kHostChunkBytes = int64_t(8) << 20;

struct HostPlan {
    int chunks = 1;
    int tw = 128;          // token-record width of the uncut call
    int64_t M = 0;
    int64_t base = 0;      // token tiles of a chunk; the first `extra` chunks take one more
    int64_t extra = 0;
    size_t y_off = 0, ws_off = 0, act_stride = 0, total = 0;  // x at offset 0

    // first row and row count of chunk c (whole tiles; the last chunk ends at M)
    void chunk(int c, int64_t* r0, int64_t* rows) const {
        const int64_t t0 = c * base + std::min<int64_t>(c, extra);
        const int64_t tiles = base + (c < extra ? 1 : 0);
        *r0 = t0 * tw;
        *rows = std::min<int64_t>(tiles * tw, M - *r0);
    }
};

HostPlan host_plan(int64_t M, int64_t N, int64_t K, int tw) {
    HostPlan h;
    h.tw = tw;
    h.M = M;
    if (!few_tokens(M, K)) {
        const int64_t by_rows = M / h.tw;
        const int64_t by_bytes = M * (K + N) * 4 / kHostChunkBytes;
        h.chunks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({kHostChunks, by_rows, by_bytes})));
    }
    // the token tiles spread evenly: chunks differ by at most one tile
    const int64_t tiles = (M + h.tw - 1) / h.tw;
    h.base = tiles / h.chunks;
    h.extra = tiles % h.chunks;
    h.y_off = align_ws(static_cast<size_t>(M) * static_cast<size_t>(K) * 4u);
    h.ws_off = align_ws(h.y_off + static_cast<size_t>(M) * static_cast<size_t>(N) * 4u);
    if (h.chunks == 1) {
        h.total = h.ws_off + prefill_ws(M, N, K);
        return h;
    }
    // prepared weights, then one prepared-activation buffer per compute stream, sized for the
    // largest chunk (the first one); a stream's chunks run in order, so they can share one
    int64_t r0, largest;
    h.chunk(0, &r0, &largest);
    h.act_stride = act_layout(largest, K, true, h.tw).total;
    h.total = h.ws_off + w_layout(N, K).total + static_cast<size_t>(std::min(h.chunks, kHostStreams)) * h.act_stride;
    return h;
}

// Streams and events of the host-buffer call, created on a device's first chunked call and
// kept for the life of the process.  The mutex keeps concurrent callers from interleaving
// their event records.
struct HostRes {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr, comp[kHostStreams] = {};
    cudaEvent_t start = nullptr, weights = nullptr, done = nullptr, in[kHostChunks] = {}, out[kHostChunks] = {};
    std::mutex mu;
};

HostRes g_host[kMaxDevices];
std::mutex g_host_init_mu;

int host_resources(HostRes** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4A8_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_host_init_mu);
    HostRes& r = g_host[dev];
    if (!r.ready) {
        const unsigned sf = cudaStreamNonBlocking;
        const unsigned ef = cudaEventDisableTiming;
        // each handle is created once: a failed attempt keeps what it made for the next one
        auto stream = [&](cudaStream_t* h) { return *h || cudaStreamCreateWithFlags(h, sf) == cudaSuccess; };
        auto event = [&](cudaEvent_t* h) { return *h || cudaEventCreateWithFlags(h, ef) == cudaSuccess; };
        bool ok = stream(&r.h2d) && stream(&r.d2h) && event(&r.start) && event(&r.weights) && event(&r.done);
        for (int i = 0; ok && i < kHostStreams; ++i) ok = stream(&r.comp[i]);
        for (int c = 0; ok && c < kHostChunks; ++c) ok = event(&r.in[c]) && event(&r.out[c]);
        if (!ok) return W4A8_ERR_CUDA;
        r.ready = true;
    }
    *out = &r;
    return W4A8_OK;
}

// A page-locked host buffer and, when the driver maps it into the device's address space
// (always for cudaHostAlloc memory under unified addressing), the address kernels use.
struct HostBuf {
    bool locked = false;
    void* dev = nullptr;
};

HostBuf host_buffer(const void* p) {
    HostBuf h;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is an answer here, not a sticky error
        return h;
    }
    h.locked = a.type == cudaMemoryTypeHost;
    if (h.locked && a.devicePointer && aligned(a.devicePointer, 16)) h.dev = a.devicePointer;
    return h;
}

}  // namespace
}  // namespace w4a8

extern "C" {

size_t w4a8_prefill_host_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (check_shape(M, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0 || N == 0) return 0;
    return host_plan(M, N, K, token_tile(M)).total;
}

int w4a8_prefill_linear_host(const float* x_host, const uint8_t* wq, const uint16_t* w_scale,
                             const uint16_t* w_zero, const float* bias, float* y_host, int64_t M, int64_t N,
                             int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!x_host || !y_host || !wq || !w_scale || !w_zero || !workspace) return W4A8_ERR_ARG;
    if (!aligned(wq, 16) || !aligned(w_scale, 2) || !aligned(w_zero, 2) || (bias && !aligned(bias, 4)) ||
        !aligned(workspace, 16))
        return W4A8_ERR_ALIGN;
    // Row chunks keep the 128-token width below 4096 rows: a chunk has a fraction of the call's
    // tiles, so it would not fill the SMs with 256-token ones (measured: two chunks of 256 rows,
    // K 2048 -> N 6144, lost 8% end to end).  A one-chunk call is the fused call, which picks
    // its own width; either way the outputs are the same (call_tile).
    const HostPlan h = host_plan(M, N, K, token_tile(M));
    if (workspace_bytes < h.total) return W4A8_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    const HostBuf xb = host_buffer(x_host), yb = host_buffer(y_host);
    if (!xb.locked || !yb.locked) return W4A8_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* x_dev = reinterpret_cast<float*>(ws);
    float* y_dev = reinterpret_cast<float*>(ws + h.y_off);
    const size_t x_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * 4u;
    const size_t y_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * 4u;

    if (h.chunks == 1) {
        // Too little to cut into chunks.  Where the host buffers are mapped, the kernels work
        // on them in place over the host link, so the transfers overlap the computation
        // without a copy's fixed cost: the pre-pass reads x with plain loads, and every
        // epilogue writes y with plain stores.  The few-token kernel fetches x with bulk
        // copies, so its x goes through the device copy.  Unmapped buffers are copied.
        const bool x_direct = xb.dev && !few_tokens(M, K);
        const float* x_in = x_direct ? static_cast<const float*>(xb.dev) : x_dev;
        float* y_out = yb.dev ? static_cast<float*>(yb.dev) : y_dev;
        if (!x_direct && cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return W4A8_ERR_CUDA;
        rc = prefill_impl(x_in, wq, w_scale, w_zero, bias, f32_out(y_out), M, N, K, ws + h.ws_off,
                          workspace_bytes - h.ws_off, stream);
        if (rc != W4A8_OK || yb.dev) return rc;
        return cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess ? W4A8_OK
                                                                                                : W4A8_ERR_CUDA;
    }

    HostRes* r = nullptr;
    if ((rc = host_resources(&r)) != W4A8_OK) return rc;
    std::lock_guard<std::mutex> lk(r->mu);
    uint8_t* pw = ws + h.ws_off;
    uint8_t* act0 = pw + w_layout(N, K).total;
    bool ok = cudaEventRecord(r->start, st) == cudaSuccess && cudaStreamWaitEvent(r->h2d, r->start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(r->d2h, r->start, 0) == cudaSuccess;
    // the weight records, once, on the caller's stream
    if (ok) {
        PrepArgs p;
        p.M = 0;
        set_weight_job(&p, wq, w_scale, w_zero, N, K, pw);
        ok = launch_pack(p, st) == cudaSuccess && cudaEventRecord(r->weights, st) == cudaSuccess;
    }
    for (int c = 0; ok && c < h.chunks; ++c) {
        int64_t r0, rows;
        h.chunk(c, &r0, &rows);
        const size_t xo = static_cast<size_t>(r0) * static_cast<size_t>(K);
        const size_t yo = static_cast<size_t>(r0) * static_cast<size_t>(N);
        const int si = c % kHostStreams;
        cudaStream_t cs = r->comp[si];
        ok = cudaMemcpyAsync(x_dev + xo, x_host + xo, static_cast<size_t>(rows) * static_cast<size_t>(K) * 4u,
                             cudaMemcpyHostToDevice, r->h2d) == cudaSuccess &&
             cudaEventRecord(r->in[c], r->h2d) == cudaSuccess && cudaStreamWaitEvent(cs, r->in[c], 0) == cudaSuccess &&
             cudaStreamWaitEvent(cs, r->weights, 0) == cudaSuccess;
        if (ok) {
            uint8_t* act = act0 + static_cast<size_t>(si) * h.act_stride;
            const ActLayout A = act_layout(rows, K, true, h.tw);
            PrepArgs p;
            p.x = x_dev + xo;
            p.M = rows;
            p.K = K;
            p.s_a_out = reinterpret_cast<float*>(act + A.s_a);
            p.trec = act + A.rec;
            p.tw = A.tw;
            ok = launch_quant(p, cs) == cudaSuccess &&
                 run_linear(act + A.rec, p.s_a_out, pw, bias, f32_out(y_dev + yo), rows, N, K, h.tw, *d, cs,
                            gemm_ksplit(M, N, K, h.tw, d->num_sms)) ==
                     W4A8_OK &&
                 cudaEventRecord(r->out[c], cs) == cudaSuccess;
        }
        ok = ok && cudaStreamWaitEvent(r->d2h, r->out[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(y_host + yo, y_dev + yo, static_cast<size_t>(rows) * static_cast<size_t>(N) * 4u,
                             cudaMemcpyDeviceToHost, r->d2h) == cudaSuccess;
    }
    // The caller's stream resumes once the last copy back has landed.  It waits on every side
    // stream's final event, not only the last one's, so that a capture into a tape joins each
    // forked stream back to the capturing stream directly.
    ok = ok && cudaEventRecord(r->done, r->d2h) == cudaSuccess && cudaStreamWaitEvent(st, r->done, 0) == cudaSuccess &&
         cudaStreamWaitEvent(st, r->in[h.chunks - 1], 0) == cudaSuccess;
    for (int c = std::max(0, h.chunks - kHostStreams); ok && c < h.chunks; ++c)
        ok = cudaStreamWaitEvent(st, r->out[c], 0) == cudaSuccess;
    return ok ? W4A8_OK : W4A8_ERR_CUDA;
}

}  // extern "C"
