// tape.cu -- recorded call sequences ("command tapes") replayed with one launch.
//
// The XNet-DNN GPU inference article, section 2.3 "RCI Command Tape": the kernel queue of a
// frame is the same every frame, so it is recorded once and replayed, and the per-frame
// command building and submission cost disappears (the article shows it for decode).  On the
// GPU the tape is a CUDA graph: w4a8_tape_begin puts the caller's stream into capture mode,
// every w4a8_* call enqueued on it is recorded instead of run (launches made with a
// programmatic dependence become programmatic graph edges), and w4a8_tape_end instantiates
// the executable graph.  Replays run the same kernels on the same buffers; the buffers'
// contents may change between replays, their addresses and sizes may not.
#include "../../include/w4a8.h"
#include "w4a8_internal.h"

#include <new>

struct w4a8_tape {
    cudaGraphExec_t exec = nullptr;
    int64_t kernels = 0;  // kernel nodes of the recorded graph: launches per replay
};

extern "C" {

int w4a8_tape_begin(void* stream) {
    if (!stream) return W4A8_ERR_ARG;  // the legacy default stream cannot be captured
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &st) != cudaSuccess) return W4A8_ERR_CUDA;
    if (st != cudaStreamCaptureStatusNone) return W4A8_ERR_ARG;
    return cudaStreamBeginCapture(static_cast<cudaStream_t>(stream), cudaStreamCaptureModeThreadLocal) ==
                   cudaSuccess
               ? W4A8_OK
               : W4A8_ERR_CUDA;
}

int w4a8_tape_end(void* stream, w4a8_tape** out) {
    if (!stream || !out) return W4A8_ERR_ARG;
    *out = nullptr;
    cudaGraph_t graph = nullptr;
    if (cudaStreamEndCapture(static_cast<cudaStream_t>(stream), &graph) != cudaSuccess || !graph)
        return W4A8_ERR_CUDA;
    // count the kernel nodes (the other nodes are event records and waits of the side streams)
    int64_t kernels = 0;
    size_t n = 0;
    if (cudaGraphGetNodes(graph, nullptr, &n) != cudaSuccess) {
        cudaGraphDestroy(graph);
        return W4A8_ERR_CUDA;
    }
    if (n > 0) {
        cudaGraphNode_t* nodes = new (std::nothrow) cudaGraphNode_t[n];
        if (!nodes) {
            cudaGraphDestroy(graph);
            return W4A8_ERR_ARG;
        }
        bool ok = cudaGraphGetNodes(graph, nodes, &n) == cudaSuccess;
        for (size_t i = 0; ok && i < n; ++i) {
            cudaGraphNodeType t;
            ok = cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess;
            if (ok && t == cudaGraphNodeTypeKernel) ++kernels;
        }
        delete[] nodes;
        if (!ok) {
            cudaGraphDestroy(graph);
            return W4A8_ERR_CUDA;
        }
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return W4A8_ERR_CUDA;
    w4a8_tape* t = new (std::nothrow) w4a8_tape;
    if (!t) {
        cudaGraphExecDestroy(exec);
        return W4A8_ERR_ARG;
    }
    t->exec = exec;
    t->kernels = kernels;
    *out = t;
    return W4A8_OK;
}

int w4a8_tape_replay(const w4a8_tape* tape, void* stream) {
    if (!tape || !tape->exec) return W4A8_ERR_ARG;
    return cudaGraphLaunch(tape->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? W4A8_OK : W4A8_ERR_CUDA;
}

int64_t w4a8_tape_kernels(const w4a8_tape* tape) { return tape ? tape->kernels : -1; }

void w4a8_tape_free(w4a8_tape* tape) {
    if (!tape) return;
    if (tape->exec) cudaGraphExecDestroy(tape->exec);
    delete tape;
}

}  // extern "C"
