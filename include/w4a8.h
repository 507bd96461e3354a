/*
 * w4a8.h -- C ABI of the GB300 (sm_103a) W4A8 block-64 quantized prefill linear.
 *
 * The operation ("MNN LLM inference on the SpacemiT K3", section 3 eqs. (1)-(3),
 * section 4 steps 1-3):
 *
 *   weights   w[n,k] ~= s_w[n,b] * (q[n,k] - z_w[n,b]),   b = k / 64            (eq. 1)
 *   act.      s_a[m] = max_k |x[m,k]| / 127 (fp32), a_q[m,k] = clamp(round_half_away(x[m,k] / s_a[m]), +-127)
 *   row sums  rs[m,b] = sum_{k in block b} a_q[m,k]            ("srcKernelSum", section 4)
 *   output    y[m,n] = s_a[m] * sum_b s_w[n,b] * (acc[m,n,b] - z_w[n,b] * rs[m,b]) + bias[n]   (eq. 2)
 *             acc[m,n,b] = sum_{k in block b} a_q[m,k] * q[n,k]   (exact int32)
 *
 * Layouts (all row-major, no padding):
 *   x       fp32  [M][K]            activations
 *   a_q     int8  [M][K]            INT8 codes
 *   a_scale fp32  [M]               s_a
 *   rowsum  int32 [M][K/64]         rs
 *   wq      uint8 [N][K/2]          u4 codes, k even in the low nibble, k odd in the high nibble
 *   w_scale fp16  [N][K/64]         s_w, passed as raw IEEE binary16 bit patterns (uint16_t)
 *   w_zero  fp16  [N][K/64]         z_w, same encoding; a real value, not necessarily an integer
 *   bias    fp32  [N] or NULL
 *   y       fp32  [M][N]
 *
 * Conventions for every call below:
 *   - Every array pointer is a DEVICE pointer owned by the caller (w4a8_prefill_linear_host,
 *     below, takes x and y in host memory); the library never allocates, frees or retains
 *     memory (command tapes, and the streams and events the host-buffer call keeps, below,
 *     are the exceptions).  Scratch comes from the caller's `workspace`.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: W4A8_OK means the work was validated and enqueued.
 *   - Shapes: K must be a positive multiple of 64; M >= 0 and N >= 0 (M == 0 or
 *     N == 0 is an empty problem: nothing is launched and W4A8_OK is returned);
 *     M, N, K <= 2^31 - 1.
 *   - Alignment: x, a_q, wq, y and workspace must be 16-byte aligned; the other arrays
 *     naturally aligned for their element type.
 *   - A violated precondition returns a negative status and launches nothing.
 *   - Inputs are assumed finite; non-finite activations give unspecified codes.
 *   - Every wait inside the kernels is bounded.  A kernel that gives up records
 *     W4A8_ERR_TIMEOUT in a per-device status word and returns early; read it with
 *     w4a8_sync_status().
 *   - The current CUDA device must be an sm_103 GPU; the library holds no state besides
 *     that status word and the one-time device check.
 */
#ifndef W4A8_H_
#define W4A8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A8_OK = 0,
    W4A8_ERR_ARG = -1,        /* NULL pointer or negative size */
    W4A8_ERR_ALIGN = -2,      /* pointer misaligned */
    W4A8_ERR_SHAPE = -3,      /* K not a positive multiple of 64, size too large, bad window */
    W4A8_ERR_CUDA = -4,       /* a CUDA runtime call or a launch failed */
    W4A8_ERR_TIMEOUT = -5,    /* a kernel gave up on a bounded wait (read by w4a8_sync_status) */
    W4A8_ERR_WORKSPACE = -6,  /* workspace NULL or smaller than the *_workspace_bytes value */
    W4A8_ERR_DEVICE = -7,     /* current device is not an sm_103 GPU */
    W4A8_ERR_SCRATCH_LIMIT = -8 /* problem needs more scratch than w4a8_prefill_linear_noalloc holds */
} w4a8_status;

/* Activation pre-pass (section 4 step 1: absmax -> scale -> INT8 codes + srcKernelSum),
 * one read of x.  Outputs a_q [M][K], a_scale [M], rowsum [M][K/64]. */
int w4a8_quant_pack(const float *x, int64_t M, int64_t K,
                    int8_t *a_q, float *a_scale, int32_t *rowsum, void *stream);

/* Few-token (decode) form.  For M <= W4A8_DECODE_MAX_M, w4a8_linear and
 * w4a8_prefill_linear stream the packed weights once (wq, w_scale and w_zero as given:
 * 4.5 bits per weight) and form each block's exact integer product on the CUDA cores
 * (section 4's decode discussion: a decode step costs one read of the weights).  This
 * needs the tokens' staged codes to fit one CTA's shared memory next to two weight stages
 * (M * K up to about 180 000); deeper rows take the tensor-core form.  The result obeys the
 * same definition and tolerance as the tensor-core form; the fp32 sums are taken in a
 * different order, so the two forms need not agree bit for bit.  The *_workspace_bytes
 * calls give the size each call needs, 0 where the few-token form needs none. */
#define W4A8_DECODE_MAX_M 8

/* Quantized linear from pre-quantized activations (section 3 eq. (2), section 4
 * steps 2-3): block-64 integer contraction on the tensor cores, then the scale /
 * zero-point / bias epilogue writing fp32 y [M][N] directly.  Each output sums its blocks'
 * scaled products in an order that depends only on the shape (M, N, K) and the GPU's SM
 * count: in block order, or,
 * for linears with few 128-token output tiles and K of at least 2048, as the sum of the two
 * halves of K (two CTAs share the tile).  Every tensor-core entry point takes the same order
 * for the same shape.  The contraction runs tiles of 256 tokens from M = 4096 on, and below
 * that where tiles of 128 would take more waves of the SMs and no K split; both kernels sum
 * in block order, so the tile width changes no output.
 * workspace: at least w4a8_linear_workspace_bytes(M, N, K) bytes (the activation
 * operand re-encoded for the tensor cores).  In the few-token form that size is 0 and
 * `workspace` may be NULL. */
int w4a8_linear(const int8_t *a_q, const float *a_scale, const int32_t *rowsum,
                const uint8_t *wq, const uint16_t *w_scale, const uint16_t *w_zero,
                const float *bias, float *y, int64_t M, int64_t N, int64_t K,
                void *workspace, size_t workspace_bytes, void *stream);

/* Fused prefill linear: the pre-pass writes the tensor-core operand, the activation
 * scales and the row sums straight into the workspace (no int8 a_q array), then
 * the linear runs.  Same result, bit for bit, as w4a8_quant_pack + w4a8_linear.
 * For M <= W4A8_DECODE_MAX_M the few-token form runs: with M * K <= 16384 in one launch
 * that quantizes the rows itself (workspace size 0, `workspace` may be NULL), otherwise
 * after the pre-pass, whose outputs (a_q, a_scale, rowsum in the API layout) the workspace
 * holds.
 * workspace: at least w4a8_prefill_workspace_bytes(M, N, K) bytes. */
int w4a8_prefill_linear(const float *x, const uint8_t *wq, const uint16_t *w_scale,
                        const uint16_t *w_zero, const float *bias, float *y,
                        int64_t M, int64_t N, int64_t K,
                        void *workspace, size_t workspace_bytes, void *stream);

/* A sequence of fused calls (section 4: a decoder layer's linears) in one library call: the
 * same as w4a8_prefill_linear on each entry in order, on `stream`, bit for bit, with one M
 * for all.  Two ways the library uses what it then knows:
 *   - Few tokens (M <= W4A8_DECODE_MAX_M), 3 to 8 entries (or 2 whose packed weights total at
 *     most 24 MiB) whose rows the weight-streaming kernel quantizes itself (M * K <= 16384)
 *     and whose activations fit one CTA together,
 *     with no entry's y overlapping any x or another y: ONE launch walks the row tiles of all
 *     entries as a single weight stream, so the kernel's start-up cost is paid once.  (Used
 *     when each entry's own launch would give every output row one warp, so the sums run in
 *     the same order and the outputs equal separate calls bit for bit.)
 *   - Otherwise one launch per entry, in order; from the second entry on the previous kernel
 *     is the library's own, which never writes the caller's weights, so a few-token kernel
 *     starts streaming its weights before that kernel has finished (a programmatic dependent
 *     launch).  An entry's x may be an earlier entry's y: activations are read only after the
 *     previous kernel has finished.
 * Either way no entry's y may overlap any entry's wq, w_scale or w_zero.  Every entry is
 * checked before anything is launched; the first failing check's status is returned. */
typedef struct w4a8_linear_ref {
    const float *x;            /* fp32 [M][K] */
    const uint8_t *wq;         /* [N][K/2] */
    const uint16_t *w_scale;   /* fp16 bits [N][K/64] */
    const uint16_t *w_zero;    /* fp16 bits [N][K/64] */
    const float *bias;         /* fp32 [N] or NULL */
    float *y;                  /* fp32 [M][N] */
    int64_t N, K;
    void *workspace;           /* at least w4a8_prefill_workspace_bytes(M, N, K) bytes */
    size_t workspace_bytes;
} w4a8_linear_ref;
int w4a8_prefill_linear_batch(const w4a8_linear_ref *linears, int64_t count, int64_t M, void *stream);

/* Split form of w4a8_prefill_linear, for callers that reuse one side across calls
 * (one activation pre-pass shared by several linears that read the same input, or
 * weights prepared once at load time):
 *   w4a8_prepare_activations  section 4 step 1 into `act` (tensor-core operand planes,
 *                             s_a, transposed row sums); act: >= w4a8_prepared_activations_bytes(M, K)
 *   w4a8_prepare_weights      the weight operand of the tensor cores (the u4 codes of wq
 *                             expanded to one byte each) and s_w / z_w laid out for the
 *                             epilogue and the zero-point term, into `pw`;
 *                             pw: >= w4a8_prepared_weights_bytes(N, K)
 *   w4a8_linear_prepared      the contraction + epilogue from both (section 4 steps 2-3)
 * The buffers are opaque; their contents are only valid for the same M / N / K.  wq, the
 * scales and the zeros are not read again after w4a8_prepare_weights.
 * prepare_activations + prepare_weights + linear_prepared equals w4a8_prefill_linear
 * bit for bit for M > W4A8_DECODE_MAX_M; for fewer tokens linear_prepared still runs the
 * tensor-core form (the prepared weights hold no packed copy to stream). */
int w4a8_prepare_activations(const float *x, int64_t M, int64_t K, void *act, size_t act_bytes,
                             void *stream);
int w4a8_prepare_weights(const uint8_t *wq, const uint16_t *w_scale, const uint16_t *w_zero,
                         int64_t N, int64_t K, void *pw, size_t pw_bytes, void *stream);
int w4a8_linear_prepared(const void *act, const void *pw, const float *bias, float *y,
                         int64_t M, int64_t N, int64_t K, void *stream);
size_t w4a8_prepared_activations_bytes(int64_t M, int64_t K);
size_t w4a8_prepared_weights_bytes(int64_t N, int64_t K);

/* Contraction + epilogue (section 4 steps 2-3) from prepared activations (`act`, written by
 * w4a8_prepare_activations for the same M and K) and the weights as given: wq, w_scale and
 * w_zero in the layouts above.  One pre-pass can then serve several linears that read the
 * same input, with no prepared copy of their weights and no workspace.  Below 4096 tokens
 * the contraction stages the packed u4 codes itself (TMA) and expands them in shared memory
 * (section 4 step 2: each task reuses one staged weight tile), so no expanded weights are
 * written to or read from device memory, and `workspace` may be NULL (size 0).  The
 * expansion shares the SM with the tensor cores and costs more per 64-block than reading
 * expanded weights (w4a8_prepare_weights + w4a8_linear_prepared, or the fused call, whose
 * pre-pass launch expands them): this call trades that time for the memory.  From 4096
 * tokens on the weights are first expanded into the workspace, at least
 * w4a8_linear_act_workspace_bytes(M, N, K) bytes.  The result equals w4a8_prefill_linear on
 * the input `act` was prepared from, bit for bit, for M > W4A8_DECODE_MAX_M. */
size_t w4a8_linear_act_workspace_bytes(int64_t M, int64_t N, int64_t K);
int w4a8_linear_act(const void *act, const uint8_t *wq, const uint16_t *w_scale, const uint16_t *w_zero,
                    const float *bias, float *y, int64_t M, int64_t N, int64_t K,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Epilogue variants ("MNN LLM inference on the SpacemiT K3", section 4 step 3: the direct
 * epilogue adds the bias and may clamp).  The *_ex calls equal their plain counterparts
 * except for the store of y:
 *   y[m,n] = clamp(s_a[m] * sum_b (...) + bias[n], clamp_lo, clamp_hi)
 * stored as fp32 (out_dtype W4A8_OUT_F32) or as bf16, round to nearest even
 * (W4A8_OUT_BF16; y then holds M*N 16-bit values, still 16-byte aligned).  clamp_lo =
 * -INFINITY and clamp_hi = +INFINITY store the value unchanged, so the plain calls are the
 * *_ex calls with W4A8_OUT_F32 and those bounds, bit for bit.  An unknown out_dtype or
 * clamp_lo > clamp_hi (or either NaN) returns W4A8_ERR_ARG and launches nothing. */
#define W4A8_OUT_F32 0
#define W4A8_OUT_BF16 1
int w4a8_prefill_linear_ex(const float *x, const uint8_t *wq, const uint16_t *w_scale,
                           const uint16_t *w_zero, const float *bias, void *y, int out_dtype,
                           float clamp_lo, float clamp_hi, int64_t M, int64_t N, int64_t K,
                           void *workspace, size_t workspace_bytes, void *stream);
int w4a8_linear_ex(const int8_t *a_q, const float *a_scale, const int32_t *rowsum,
                   const uint8_t *wq, const uint16_t *w_scale, const uint16_t *w_zero,
                   const float *bias, void *y, int out_dtype, float clamp_lo, float clamp_hi,
                   int64_t M, int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                   void *stream);
int w4a8_linear_prepared_ex(const void *act, const void *pw, const float *bias, void *y,
                            int out_dtype, float clamp_lo, float clamp_hi, int64_t M, int64_t N,
                            int64_t K, void *stream);

/* w4a8_prefill_linear for callers that cannot allocate device memory (no counterpart in
 * the paper; it exists for integration only).  Some callers have no way to hand the
 * library a workspace: code that runs where cudaMalloc is not allowed or not wanted (an
 * allocator-free runtime, a region that must not synchronize the device, a host with no
 * spare memory budget for per-call buffers).  This entry point takes the same inputs
 * and output as w4a8_prefill_linear but keeps its scratch in one fixed array that the
 * library reserves statically on every GPU it is loaded on (W4A8_NOALLOC_SCRATCH_BYTES,
 * held until the process exits), so it allocates and frees nothing.
 *   - Problems whose w4a8_prefill_workspace_bytes(M, N, K) exceeds the array are rejected
 *     with W4A8_ERR_SCRATCH_LIMIT before anything is launched.
 *   - The first call on a device looks up the array's device address (a one-time
 *     runtime query per device); make that first call before any stream capture.
 *   - All calls on a device share the one array and it keeps the previous call's
 *     contents: calls that can overlap on the GPU (other streams, other threads) race on
 *     it and must be serialized by the caller.  Nothing in it needs clearing between
 *     calls: every scratch byte that feeds a stored output is rewritten by each call.
 *   - Results are bit-identical to w4a8_prefill_linear on the same inputs. */
#define W4A8_NOALLOC_SCRATCH_BYTES (16u << 20)
int w4a8_prefill_linear_noalloc(const float *x, const uint8_t *wq, const uint16_t *w_scale,
                                const uint16_t *w_zero, const float *bias, float *y,
                                int64_t M, int64_t N, int64_t K, void *stream);

/* w4a8_prefill_linear with x and y in HOST memory (no counterpart in the paper; it carries
 * the copies an application makes around the fused call, section 3 eq. (1)-(2), and hides
 * them behind the computation).  x_host: fp32 [M][K], y_host: fp32 [M][N], both page-locked
 * (cudaHostAlloc / cudaHostRegister; any other pointer gives W4A8_ERR_ARG); the weights,
 * bias and workspace are device memory as elsewhere.  workspace: at least
 * w4a8_prefill_host_workspace_bytes(M, N, K) bytes, 16-byte aligned (it holds the device
 * copies of x and y and the pre-pass scratch).
 *   - Large calls are cut into up to sixteen row chunks, each a whole number of token tiles
 *     and at least 8 MiB of x and y.  Chunk c+1's copy to the device, chunk c's linear and
 *     chunk c-1's copy back overlap, on six streams the library creates on a device's first
 *     chunked call and keeps until the process exits.
 *   - Smaller calls are one chunk.  When the driver maps the host buffers into the device's
 *     address space (cudaHostAlloc memory under unified addressing), the kernels then read
 *     x and write y in place over the host link, so the transfers overlap the computation;
 *     otherwise x and y are copied through the workspace.  The few-token form always copies
 *     x.
 *   - Stream-ordered like every call: the work starts after what was enqueued on `stream`
 *     before it, and what is enqueued after it sees y_host complete.  The host buffers must
 *     stay valid and x_host unchanged until then.  Calls sharing a workspace must be
 *     ordered (one stream).  It may be recorded into a tape (make one call of the shape
 *     first).  A chunked call joins the library's side streams to the capture until
 *     w4a8_tape_end, so meanwhile no other thread may make a host-buffer call on that
 *     device.
 *   - Results are bit-identical to w4a8_prefill_linear on the same inputs. */
size_t w4a8_prefill_host_workspace_bytes(int64_t M, int64_t N, int64_t K);
int w4a8_prefill_linear_host(const float *x_host, const uint8_t *wq, const uint16_t *w_scale,
                             const uint16_t *w_zero, const float *bias, float *y_host,
                             int64_t M, int64_t N, int64_t K, void *workspace,
                             size_t workspace_bytes, void *stream);

/* Workspace sizes in bytes (0 for an empty problem; (size_t)-1 for invalid shapes). */
size_t w4a8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t w4a8_prefill_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t w4a8_debug_workspace_bytes(int64_t m_cnt, int64_t n_cnt, int64_t K);

/* Debug: the exact per-block int32 accumulators acc[m][n][b] (section 3 eq. (2), first
 * sum) for the window m0 <= m < m0 + m_cnt, n0 <= n < n0 + n_cnt, computed by the
 * tensor-core contraction that w4a8_linear runs for this problem (M, N, K) on the current
 * device: the 256-token kernel (token records 256 wide, N = 256 MMAs) where w4a8_linear takes
 * it (always from M = 4096 on), the 128-token kernel otherwise.  For M <= W4A8_DECODE_MAX_M w4a8_linear forms its block products on the CUDA
 * cores instead; this call still runs the 128-token tensor-core contraction there.
 * acc: int32 [m_cnt][n_cnt][K/64], indexed by the position inside the window.  The window
 * must lie inside [0, M) x [0, N) and be non-empty.  workspace: at least
 * w4a8_debug_workspace_bytes(m_cnt, n_cnt, K) bytes (one size for either kernel). */
int w4a8_debug_block_acc(const int8_t *a_q, const uint8_t *wq, int64_t M, int64_t N, int64_t K,
                         int64_t m0, int64_t m_cnt, int64_t n0, int64_t n_cnt, int32_t *acc,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Command tapes (the XNet-DNN GPU inference article, section 2.3 "RCI Command Tape": a
 * frame's kernel queue is recorded once and replayed).  Between w4a8_tape_begin(stream)
 * and w4a8_tape_end(stream, &tape), the w4a8_* calls enqueued on `stream` are recorded, not
 * run; w4a8_tape_replay(tape, s) then runs the whole sequence with one launch on any
 * stream of the same device.  A replay reads and writes the very buffers the recorded calls
 * named: their contents may change between replays, their addresses and sizes must stay
 * valid until w4a8_tape_free.  Recording goes through CUDA stream capture (thread-local
 * mode), so `stream` must be a non-default stream that is not already capturing
 * (W4A8_ERR_ARG otherwise), and everything else enqueued on it meanwhile -- by this thread --
 * is recorded as well.  The tape object (host memory plus the driver's executable graph) is
 * the one resource the library allocates; w4a8_tape_free releases it.  Make one ordinary
 * call of each shape before recording, so no one-time setup falls inside the capture. */
typedef struct w4a8_tape w4a8_tape;
int w4a8_tape_begin(void *stream);
int w4a8_tape_end(void *stream, w4a8_tape **tape);
int w4a8_tape_replay(const w4a8_tape *tape, void *stream);
void w4a8_tape_free(w4a8_tape *tape);
/* The number of kernel launches one replay of the tape makes (the kernel nodes of its graph;
 * copies, event records and waits are not counted); -1 for a NULL tape. */
int64_t w4a8_tape_kernels(const w4a8_tape *tape);

/* Synchronizes `stream`, then returns and clears the current device's status word:
 * W4A8_OK, W4A8_ERR_TIMEOUT if a kernel gave up on a wait since the last call, or
 * W4A8_ERR_CUDA if the synchronization itself failed. */
int w4a8_sync_status(void *stream);

/* Diagnostic: launches one CTA that waits on a barrier nothing will ever complete,
 * with a wait limit of `limit_us` microseconds (1..10^6), so that the bounded-wait
 * path can be tested.  The kernel records W4A8_ERR_TIMEOUT and returns. */
int w4a8_selftest_wait_timeout(int64_t limit_us, void *stream);

/* Human-readable name of a status code (static string). */
const char *w4a8_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int w4a8_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H_ */
