// Host-buffer steps: one forward + backward of the layer whose inputs and
// results live in host memory, the copies overlapped with the GPU work of the
// neighbouring steps. Built on the public calls only (moe_forward,
// moe_backward, moe_saved_*): the pipeline adds the staging, the copies and
// their ordering, nothing of the layer's arithmetic.
//
// Ordering (two staging sets A/B, step n uses set n mod 2):
//   upload stream  : [wait computed(set) of its previous step] H2D inputs -> record uploaded(set)
//   compute stream : wait uploaded(set), wait downloaded(set) of its previous step,
//                    wait computed of step n-1 (main_grad accumulates in call order)
//                    forward, backward -> record computed(set)
//   download stream: wait computed(set) D2H results -> record downloaded(set)
// so step n+1's uploads run during step n's kernels and step n's downloads
// during step n+1's.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/moe.h"

namespace {

constexpr size_t kPipeAlign = 256;

size_t round_up(size_t v) { return (v + kPipeAlign - 1) / kPipeAlign * kPipeAlign; }

struct StagingSet {
    void* hidden;       // [T,H] bf16
    float* probs;       // [T,E] fp32
    uint8_t* map;       // [T,E] bytes
    void* grad_out;     // [T,H] bf16
    void* out;          // [T,H] bf16
    void* dhidden;      // [T,H] bf16
    float* dprobs;      // [T,E] fp32
};

// Lays out two staging sets and the saved state in `base` (nullptr: sizes only);
// returns the bytes used.
size_t carve(int64_t T, int64_t H, int64_t E, size_t saved_bytes, uint8_t* base, StagingSet sets[2], void** saved) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        void* p = base ? base + off : nullptr;
        off += round_up(bytes);
        return p;
    };
    const size_t row_bytes = size_t(T) * size_t(H) * 2;
    const size_t te = size_t(T) * size_t(E);
    for (int s = 0; s < 2; ++s) {
        sets[s].hidden = take(row_bytes);
        sets[s].probs = static_cast<float*>(take(te * 4));
        sets[s].map = static_cast<uint8_t*>(take(te));
        sets[s].grad_out = take(row_bytes);
        sets[s].out = take(row_bytes);
        sets[s].dhidden = take(row_bytes);
        sets[s].dprobs = static_cast<float*>(take(te * 4));
    }
    *saved = take(saved_bytes);
    return off;
}

}  // namespace

struct moe_host_pipe {
    moe_handle* h;
    int64_t T, H, E;
    StagingSet sets[2];
    moe_saved* saved;
    cudaStream_t up, down;
    cudaEvent_t uploaded[2], computed[2], downloaded[2];
    bool used[2];
    int64_t n;  // steps enqueued
};

namespace {

void release(moe_host_pipe* p) {
    if (p->saved) moe_saved_destroy(p->saved);
    for (int s = 0; s < 2; ++s) {
        if (p->uploaded[s]) cudaEventDestroy(p->uploaded[s]);
        if (p->computed[s]) cudaEventDestroy(p->computed[s]);
        if (p->downloaded[s]) cudaEventDestroy(p->downloaded[s]);
    }
    if (p->up) cudaStreamDestroy(p->up);
    if (p->down) cudaStreamDestroy(p->down);
    delete p;
}

bool config_sizes(const moe_config* cfg, int64_t T, size_t* total) {
    size_t saved_bytes = 0;
    if (moe_saved_size(cfg, &saved_bytes) != MOE_OK) return false;
    StagingSet sets[2];
    void* saved = nullptr;
    *total = carve(T, cfg->hidden, cfg->num_experts, saved_bytes, nullptr, sets, &saved);
    return true;
}

}  // namespace

extern "C" {

moe_status moe_host_pipe_size(const moe_config* cfg, int64_t T, size_t* bytes) {
    if (!cfg || !bytes || T < 1 || T > cfg->max_tokens) return MOE_ERR_INVALID_ARG;
    size_t ws = 0;
    const moe_status st = moe_workspace_size(cfg, &ws);  // validates the configuration
    if (st != MOE_OK) return st;
    return config_sizes(cfg, T, bytes) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

moe_status moe_host_pipe_create(moe_handle* h, int64_t T, void* memory, size_t bytes, moe_host_pipe** out) {
    moe_config c;
    if (!h || !out || moe_handle_config(h, &c) != MOE_OK || T < 1 || T > c.max_tokens) return MOE_ERR_INVALID_ARG;
    const moe_config* cfg = &c;
    *out = nullptr;
    size_t need = 0;
    if (!config_sizes(cfg, T, &need)) return MOE_ERR_INVALID_ARG;
    if (!memory || bytes < need || reinterpret_cast<uintptr_t>(memory) % kPipeAlign) return MOE_ERR_INVALID_ARG;
    size_t saved_bytes = 0;
    moe_saved_size(cfg, &saved_bytes);
    moe_host_pipe* p = new (std::nothrow) moe_host_pipe;
    if (!p) return MOE_ERR_INVALID_ARG;
    std::memset(p, 0, sizeof(*p));
    p->h = h;
    p->T = T;
    p->H = cfg->hidden;
    p->E = cfg->num_experts;
    void* saved_mem = nullptr;
    carve(T, p->H, p->E, saved_bytes, static_cast<uint8_t*>(memory), p->sets, &saved_mem);
    moe_status st = moe_saved_create(h, saved_mem, saved_bytes, &p->saved);
    if (st != MOE_OK) {
        release(p);
        return st;
    }
    bool ok = cudaStreamCreateWithFlags(&p->up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->down, cudaStreamNonBlocking) == cudaSuccess;
    for (int s = 0; ok && s < 2; ++s)
        ok = cudaEventCreateWithFlags(&p->uploaded[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->computed[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->downloaded[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        release(p);
        return MOE_ERR_CUDA;
    }
    *out = p;
    return MOE_OK;
}

#define PIPE_CU(x)                                   \
    do {                                             \
        if ((x) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

moe_status moe_host_step(moe_host_pipe* p, const void* hidden, const float* probs, const uint8_t* routing_map,
                         const void* grad_out, const moe_weights* w, const moe_main_grads* mg, void* out,
                         void* dhidden, float* dprobs, void* stream) {
    if (!p || !hidden || !probs || !routing_map || !grad_out || !w || !mg || !out || !dhidden || !dprobs)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int s = int(p->n & 1);
    const int prev = s ^ 1;
    const StagingSet& b = p->sets[s];
    const size_t row_bytes = size_t(p->T) * size_t(p->H) * 2;
    const size_t te = size_t(p->T) * size_t(p->E);

    // uploads: the set's previous step must have finished reading its inputs
    if (p->used[s]) PIPE_CU(cudaStreamWaitEvent(p->up, p->computed[s], 0));
    PIPE_CU(cudaMemcpyAsync(b.hidden, hidden, row_bytes, cudaMemcpyHostToDevice, p->up));
    PIPE_CU(cudaMemcpyAsync(b.probs, probs, te * 4, cudaMemcpyHostToDevice, p->up));
    PIPE_CU(cudaMemcpyAsync(b.map, routing_map, te, cudaMemcpyHostToDevice, p->up));
    PIPE_CU(cudaMemcpyAsync(b.grad_out, grad_out, row_bytes, cudaMemcpyHostToDevice, p->up));
    PIPE_CU(cudaEventRecord(p->uploaded[s], p->up));

    // compute: inputs present, the set's previous results gone, the previous step done
    PIPE_CU(cudaStreamWaitEvent(st, p->uploaded[s], 0));
    if (p->used[s]) PIPE_CU(cudaStreamWaitEvent(st, p->downloaded[s], 0));
    if (p->used[prev]) PIPE_CU(cudaStreamWaitEvent(st, p->computed[prev], 0));
    moe_status r = moe_forward(p->h, p->T, b.hidden, b.probs, b.map, w, b.out, p->saved, stream);
    if (r == MOE_OK) r = moe_backward(p->h, b.grad_out, p->saved, b.dhidden, b.dprobs, mg, stream);
    if (r != MOE_OK) {
        // the set's uploads, and whatever part of the step was enqueued, finish before
        // the next step may write the same staging set
        cudaStreamSynchronize(p->up);
        cudaStreamSynchronize(st);
        return r;
    }
    PIPE_CU(cudaEventRecord(p->computed[s], st));

    // downloads
    PIPE_CU(cudaStreamWaitEvent(p->down, p->computed[s], 0));
    PIPE_CU(cudaMemcpyAsync(out, b.out, row_bytes, cudaMemcpyDeviceToHost, p->down));
    PIPE_CU(cudaMemcpyAsync(dhidden, b.dhidden, row_bytes, cudaMemcpyDeviceToHost, p->down));
    PIPE_CU(cudaMemcpyAsync(dprobs, b.dprobs, te * 4, cudaMemcpyDeviceToHost, p->down));
    PIPE_CU(cudaEventRecord(p->downloaded[s], p->down));
    p->used[s] = true;
    ++p->n;
    return MOE_OK;
}

moe_status moe_host_pipe_sync(moe_host_pipe* p) {
    if (!p) return MOE_ERR_INVALID_ARG;
    for (int s = 0; s < 2; ++s)
        if (p->used[s]) PIPE_CU(cudaEventSynchronize(p->downloaded[s]));
    return MOE_OK;
}

void moe_host_pipe_destroy(moe_host_pipe* p) {
    if (!p) return;
    moe_host_pipe_sync(p);
    release(p);
}

}  // extern "C"
