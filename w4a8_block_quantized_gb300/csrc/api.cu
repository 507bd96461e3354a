// api.cu -- the C ABI declared in include/w4a8.h: argument validation, workspace
// carving, tensor-map encoding and kernel launches.  Nothing here allocates memory.
#include "../../include/w4a8.h"
#include "w4a8_internal.h"

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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D uint8 tensor map: `rows` rows of `inner` bytes at `stride` bytes; box inner x rows.
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride,
                 uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxDim = 2147483647LL;

int check_shape(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0) return W4A8_ERR_ARG;
    if (K <= 0 || K % kBlock != 0) return W4A8_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return W4A8_ERR_SHAPE;
    // tensor-map coordinates and the weight-row byte stride stay within 32 bits
    if (2 * K > kMaxDim || N > (int64_t(1) << 31)) return W4A8_ERR_SHAPE;
    return W4A8_OK;
}

// Workspace of the one-call entry points: prepared activations, then prepared scales.
struct CallLayout {
    ActLayout act;
    size_t wsc = 0, total = 0;
};

CallLayout call_layout(int64_t M, int64_t N, int64_t K, bool with_sa) {
    CallLayout c;
    c.act = act_layout(M, K, with_sa, true);
    c.wsc = c.act.total;
    c.total = c.wsc + wsc_bytes(N, K);
    return c;
}

// GEMM + epilogue from prepared activations (apk, rx at act offsets) and prepared scales.
int run_linear(const uint8_t* act, const ActLayout& A, const float* s_a, const float* wsc, const uint8_t* wq,
               const float* bias, float* y, int64_t M, int64_t N, int64_t K, const DeviceInfo& d, cudaStream_t st) {
    GemmMaps maps;
    const int tn = pick_token_tile(M, N, d.num_sms);
    if (!make_map_u8(&maps.a, act + A.apk, 2 * K, M, 2 * K, 128, tn, CU_TENSOR_MAP_SWIZZLE_128B))
        return W4A8_ERR_CUDA;
    if (!make_map_u8(&maps.b, wq, K / 2, N, K / 2, 32, kTileW, CU_TENSOR_MAP_SWIZZLE_NONE)) return W4A8_ERR_CUDA;
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.m_cnt = M;
    g.n0 = 0;
    g.n_cnt = N;
    g.M_pad = A.M_pad;
    g.N_pad = n_pad(N);
    g.wsc = wsc;
    g.rx = reinterpret_cast<const uint4*>(act + A.rx);
    g.s_a = s_a;
    g.bias = bias;
    g.y = y;
    g.status = d.status;
    return launch_gemm(maps, g, tn, false, st) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

}  // namespace
}  // namespace w4a8

using namespace w4a8;

extern "C" {

int w4a8_abi_version(void) { return 100; }

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
    return call_layout(M, N, K, false).total;
}

size_t w4a8_prefill_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (check_shape(M, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0 || N == 0) return 0;
    return call_layout(M, N, K, true).total;
}

size_t w4a8_debug_workspace_bytes(int64_t m_cnt, int64_t K) {
    if (check_shape(m_cnt, 1, K) != W4A8_OK || m_cnt == 0) return static_cast<size_t>(-1);
    return act_layout(m_cnt, K, false, false).total;
}

size_t w4a8_prepared_activations_bytes(int64_t M, int64_t K) {
    if (check_shape(M, 1, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (M == 0) return 0;
    return act_layout(M, K, true, true).total;
}

size_t w4a8_prepared_weights_bytes(int64_t N, int64_t K) {
    if (check_shape(1, N, K) != W4A8_OK) return static_cast<size_t>(-1);
    if (N == 0) return 0;
    return wsc_bytes(N, K);
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
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!a_q || !a_scale || !rowsum || !wq || !w_scale || !w_zero || !y) return W4A8_ERR_ARG;
    if (!aligned(a_q, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(a_scale, 4) || !aligned(rowsum, 4) ||
        !aligned(w_scale, 2) || !aligned(w_zero, 2) || (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    const CallLayout L = call_layout(M, N, K, false);
    if (!workspace || workspace_bytes < L.total) return W4A8_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    PrepArgs p;
    p.a_q_in = a_q;
    p.rs_in = rowsum;
    p.M = M;
    p.K = K;
    p.apk = ws + L.act.apk;
    p.rx = reinterpret_cast<uint4*>(ws + L.act.rx);
    p.M_pad = L.act.M_pad;
    p.s_w = w_scale;
    p.z_w = w_zero;
    p.N = N;
    p.N_pad = n_pad(N);
    p.wsc = reinterpret_cast<float*>(ws + L.wsc);
    if (launch_pack(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    return run_linear(ws, L.act, a_scale, reinterpret_cast<const float*>(ws + L.wsc), wq, bias, y, M, N, K, *d, st);
}

int w4a8_prefill_linear(const float* x, const uint8_t* wq, const uint16_t* w_scale, const uint16_t* w_zero,
                        const float* bias, float* y, int64_t M, int64_t N, int64_t K, void* workspace,
                        size_t workspace_bytes, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!x || !wq || !w_scale || !w_zero || !y) return W4A8_ERR_ARG;
    if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(w_scale, 2) || !aligned(w_zero, 2) ||
        (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    const CallLayout L = call_layout(M, N, K, true);
    if (!workspace || workspace_bytes < L.total) return W4A8_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* s_a = reinterpret_cast<float*>(ws + L.act.s_a);
    PrepArgs p;
    p.x = x;
    p.M = M;
    p.K = K;
    p.s_a_out = s_a;
    p.apk = ws + L.act.apk;
    p.rx = reinterpret_cast<uint4*>(ws + L.act.rx);
    p.M_pad = L.act.M_pad;
    p.s_w = w_scale;
    p.z_w = w_zero;
    p.N = N;
    p.N_pad = n_pad(N);
    p.wsc = reinterpret_cast<float*>(ws + L.wsc);
    if (launch_quant(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    return run_linear(ws, L.act, s_a, reinterpret_cast<const float*>(ws + L.wsc), wq, bias, y, M, N, K, *d, st);
}

int w4a8_prepare_activations(const float* x, int64_t M, int64_t K, void* act, size_t act_bytes, void* stream) {
    int rc = check_shape(M, 1, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0) return W4A8_OK;
    if (!x || !act) return W4A8_ERR_ARG;
    if (!aligned(x, 16) || !aligned(act, 16)) return W4A8_ERR_ALIGN;
    const ActLayout A = act_layout(M, K, true, true);
    if (act_bytes < A.total) return W4A8_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    uint8_t* a = static_cast<uint8_t*>(act);
    PrepArgs p;
    p.x = x;
    p.M = M;
    p.K = K;
    p.s_a_out = reinterpret_cast<float*>(a + A.s_a);
    p.apk = a + A.apk;
    p.rx = reinterpret_cast<uint4*>(a + A.rx);
    p.M_pad = A.M_pad;
    return launch_quant(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int w4a8_prepare_weights(const uint16_t* w_scale, const uint16_t* w_zero, int64_t N, int64_t K, void* wsc,
                         size_t wsc_size, void* stream) {
    int rc = check_shape(1, N, K);
    if (rc != W4A8_OK) return rc;
    if (N == 0) return W4A8_OK;
    if (!w_scale || !w_zero || !wsc) return W4A8_ERR_ARG;
    if (!aligned(w_scale, 2) || !aligned(w_zero, 2) || !aligned(wsc, 16)) return W4A8_ERR_ALIGN;
    if (wsc_size < wsc_bytes(N, K)) return W4A8_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    PrepArgs p;
    p.M = 0;
    p.K = K;
    p.s_w = w_scale;
    p.z_w = w_zero;
    p.N = N;
    p.N_pad = n_pad(N);
    p.wsc = static_cast<float*>(wsc);
    return launch_pack(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int w4a8_linear_prepared(const void* act, const uint8_t* wq, const void* wsc, const float* bias, float* y,
                         int64_t M, int64_t N, int64_t K, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (M == 0 || N == 0) return W4A8_OK;
    if (!act || !wq || !wsc || !y) return W4A8_ERR_ARG;
    if (!aligned(act, 16) || !aligned(wq, 16) || !aligned(wsc, 16) || !aligned(y, 16) || (bias && !aligned(bias, 4)))
        return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    const ActLayout A = act_layout(M, K, true, true);
    const uint8_t* a = static_cast<const uint8_t*>(act);
    return run_linear(a, A, reinterpret_cast<const float*>(a + A.s_a), static_cast<const float*>(wsc), wq, bias, y,
                      M, N, K, *d, static_cast<cudaStream_t>(stream));
}

int w4a8_debug_block_acc(const int8_t* a_q, const uint8_t* wq, int64_t M, int64_t N, int64_t K, int64_t m0,
                         int64_t m_cnt, int64_t n0, int64_t n_cnt, int32_t* acc, void* workspace,
                         size_t workspace_bytes, void* stream) {
    int rc = check_shape(M, N, K);
    if (rc != W4A8_OK) return rc;
    if (!a_q || !wq || !acc) return W4A8_ERR_ARG;
    if (m0 < 0 || n0 < 0 || m_cnt <= 0 || n_cnt <= 0 || m0 + m_cnt > M || n0 + n_cnt > N) return W4A8_ERR_SHAPE;
    if (!aligned(a_q, 16) || !aligned(wq, 16) || !aligned(acc, 4)) return W4A8_ERR_ALIGN;
    const ActLayout L = act_layout(m_cnt, K, false, false);
    if (!workspace || workspace_bytes < L.total) return W4A8_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return W4A8_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    PrepArgs p;
    p.a_q_in = a_q;
    p.M = m_cnt;
    p.K = K;
    p.row0 = m0;
    p.apk = ws + L.apk;
    if (launch_pack(p, st) != cudaSuccess) return W4A8_ERR_CUDA;
    GemmMaps maps;
    const int tn = pick_token_tile(m_cnt, n_cnt, d->num_sms);
    if (!make_map_u8(&maps.a, ws + L.apk, 2 * K, m_cnt, 2 * K, 128, tn, CU_TENSOR_MAP_SWIZZLE_128B))
        return W4A8_ERR_CUDA;
    if (!make_map_u8(&maps.b, wq, K / 2, N, K / 2, 32, kTileW, CU_TENSOR_MAP_SWIZZLE_NONE)) return W4A8_ERR_CUDA;
    GemmArgs g;
    g.M = m_cnt;
    g.N = N;
    g.K = K;
    g.m_cnt = m_cnt;
    g.n0 = n0;
    g.n_cnt = n_cnt;
    g.acc = acc;
    g.status = d->status;
    return launch_gemm(maps, g, tn, true, st) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
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
    const size_t need = call_layout(M, N, K, true).total;
    if (need > W4A8_NOALLOC_SCRATCH_BYTES) return W4A8_ERR_SCRATCH_LIMIT;
    DeviceInfo* d = nullptr;
    if ((rc = current_device(&d)) != W4A8_OK) return rc;
    uint8_t* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != W4A8_OK) return rc;
    return w4a8_prefill_linear(x, wq, w_scale, w_zero, bias, y, M, N, K, scratch, W4A8_NOALLOC_SCRATCH_BYTES,
                               stream);
}

}  // extern "C"
