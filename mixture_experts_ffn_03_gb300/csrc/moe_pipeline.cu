// Serving loop from host buffers (moe_pipeline_*): the layer of moe_forward
// fed from, and returning into, host memory, with the host<->device copies of
// neighbouring steps overlapping the compute.
//
// A pipeline owns two device staging sets (hidden rows, router logits,
// output), one moe_forward workspace, an input copy stream and an output
// copy stream; compute runs on the caller's stream. Step i uses staging set
// i % 2:
//   input stream   wait until step i-2 no longer reads set i % 2; copy the
//                  step's hidden rows and logits in; mark them landed
//   compute stream wait for them (and for step i-2's output copy, which
//                  reads the same output buffer); moe_forward; mark done
//   output stream  wait for the compute; copy the output back; mark read
// The directions have streams of their own, so step i+1's input copy runs
// while step i computes instead of queueing behind step i's output copy.
// Copies are one cudaMemcpyAsync each; with pinned host memory they are
// asynchronous and overlap, with pageable memory CUDA stages them.
#include <cuda_runtime.h>

#include <new>

#include "moe.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

struct moe_pipeline {
    moe_dims d;
    const void* w_gate_up;
    const void* w_down;
    const void* ws_gate_up;
    const void* ws_down;
    const void* w_g;
    int device;
    cudaStream_t cs;     // the caller's compute stream
    cudaStream_t in_s;   // host -> device copies
    cudaStream_t out_s;  // device -> host copies
    void* hid[2];
    void* logit[2];
    void* out[2];
    void* ws;
    size_t ws_bytes;
    cudaEvent_t in_ready[2], done[2], out_read[2];
    long long n;  // steps submitted
};

namespace {

size_t hidden_bytes(const moe_dims& d) { return static_cast<size_t>(d.T) * d.H * 2; }
size_t logit_bytes(const moe_dims& d) { return static_cast<size_t>(d.T) * d.E * 4; }

// Frees whatever `p` holds (members not created yet are null) and `p`.
void release(moe_pipeline* p) {
    if (!p) return;
    if (p->in_s) cudaStreamSynchronize(p->in_s);
    if (p->out_s) cudaStreamSynchronize(p->out_s);
    if (p->n > 0) cudaStreamSynchronize(p->cs);
    for (int b = 0; b < 2; ++b) {
        if (p->in_ready[b]) cudaEventDestroy(p->in_ready[b]);
        if (p->done[b]) cudaEventDestroy(p->done[b]);
        if (p->out_read[b]) cudaEventDestroy(p->out_read[b]);
        cudaFree(p->hid[b]);
        cudaFree(p->logit[b]);
        cudaFree(p->out[b]);
    }
    cudaFree(p->ws);
    if (p->in_s) cudaStreamDestroy(p->in_s);
    if (p->out_s) cudaStreamDestroy(p->out_s);
    delete p;
}

// Runs the calls of one entry point on the pipeline's device and restores the
// caller's current device afterwards.
class OnDevice {
public:
    explicit OnDevice(int dev) {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess &&
              (prev_ == dev || cudaSetDevice(dev) == cudaSuccess);
    }
    ~OnDevice() {
        int cur = -1;
        if (cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

private:
    int prev_ = 0;
    bool ok_ = false;
};

}  // namespace

MOE_API moe_status moe_pipeline_create(const moe_dims* d, const void* w_gate_up,
                                       const void* w_down, const void* ws_gate_up,
                                       const void* ws_down, const void* w_g, void* cuda_stream,
                                       moe_pipeline** out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!d || !w_gate_up || !w_down || !ws_gate_up || !ws_down || !w_g) return MOE_ERR_INVALID_ARG;
    const size_t ws_bytes = moe_workspace_size(d);
    if (ws_bytes == 0 || d->T < 1) return MOE_ERR_INVALID_ARG;
    moe_pipeline* p = new (std::nothrow) moe_pipeline();
    if (!p) return MOE_ERR_CUDA;
    p->d = *d;
    p->w_gate_up = w_gate_up;
    p->w_down = w_down;
    p->ws_gate_up = ws_gate_up;
    p->ws_down = ws_down;
    p->w_g = w_g;
    p->cs = static_cast<cudaStream_t>(cuda_stream);
    p->ws_bytes = ws_bytes;
    bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->in_s, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->out_s, cudaStreamNonBlocking) == cudaSuccess &&
              cudaMalloc(&p->ws, ws_bytes) == cudaSuccess;
    for (int b = 0; ok && b < 2; ++b)
        ok = cudaMalloc(&p->hid[b], hidden_bytes(*d)) == cudaSuccess &&
             cudaMalloc(&p->logit[b], logit_bytes(*d)) == cudaSuccess &&
             cudaMalloc(&p->out[b], hidden_bytes(*d)) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->in_ready[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->done[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->out_read[b], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        release(p);
        return MOE_ERR_CUDA;
    }
    *out = p;
    return MOE_OK;
}

MOE_API moe_status moe_pipeline_submit(moe_pipeline* p, const void* hidden_host,
                                       const float* logits_host, void* out_host) {
    if (!p || !hidden_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
    OnDevice on(p->device);
    if (!on.ok()) return MOE_ERR_CUDA;
    const int b = static_cast<int>(p->n & 1);
    const bool reuse = p->n >= 2;  // set b was used by step n - 2
    if (reuse && cudaStreamWaitEvent(p->in_s, p->done[b], 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(p->hid[b], hidden_host, hidden_bytes(p->d), cudaMemcpyHostToDevice,
                        p->in_s) != cudaSuccess ||
        cudaMemcpyAsync(p->logit[b], logits_host, logit_bytes(p->d), cudaMemcpyHostToDevice,
                        p->in_s) != cudaSuccess ||
        cudaEventRecord(p->in_ready[b], p->in_s) != cudaSuccess ||
        cudaStreamWaitEvent(p->cs, p->in_ready[b], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (reuse && cudaStreamWaitEvent(p->cs, p->out_read[b], 0) != cudaSuccess) return MOE_ERR_CUDA;
    const moe_status st =
        moe_forward(&p->d, p->hid[b], static_cast<const float*>(p->logit[b]), p->w_gate_up,
                    p->w_down, p->ws_gate_up, p->ws_down, p->w_g, p->out[b], nullptr, nullptr,
                    nullptr, p->ws, p->ws_bytes, p->cs);
    if (st != MOE_OK) return st;
    if (cudaEventRecord(p->done[b], p->cs) != cudaSuccess ||
        cudaStreamWaitEvent(p->out_s, p->done[b], 0) != cudaSuccess ||
        cudaMemcpyAsync(out_host, p->out[b], hidden_bytes(p->d), cudaMemcpyDeviceToHost,
                        p->out_s) != cudaSuccess ||
        cudaEventRecord(p->out_read[b], p->out_s) != cudaSuccess)
        return MOE_ERR_CUDA;
    ++p->n;
    return MOE_OK;
}

MOE_API moe_status moe_pipeline_drain(moe_pipeline* p) {
    if (!p) return MOE_ERR_INVALID_ARG;
    OnDevice on(p->device);
    if (!on.ok()) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(p->in_s) != cudaSuccess ||
        cudaStreamSynchronize(p->cs) != cudaSuccess ||
        cudaStreamSynchronize(p->out_s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return p->n > 0 ? moe_device_status(p->ws, p->cs) : MOE_OK;
}

MOE_API moe_status moe_pipeline_streams(const moe_pipeline* p, void** in_stream,
                                        void** out_stream) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (in_stream) *in_stream = p->in_s;
    if (out_stream) *out_stream = p->out_s;
    return MOE_OK;
}

MOE_API void moe_pipeline_destroy(moe_pipeline* p) {
    if (!p) return;
    OnDevice on(p->device);
    release(p);
}
