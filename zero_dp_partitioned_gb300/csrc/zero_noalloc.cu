// zero_noalloc.cu -- zero_shard_step_noalloc: the partitioned step for
// callers that cannot allocate device memory.
//
// zero_shard_step needs device scratch from its caller: a small workspace
// (per-block partial sums, a completion counter, the step's statistics) and,
// when it takes the two-pass path, a 16-bit buffer per shard for the reduced
// gradient.  Some callers have no way to provide that: code that must not
// call cudaMalloc because the call can synchronise the whole device and stall
// other work in a latency-bound loop, callers living inside a host program
// whose own allocator owns all device memory and forbids allocations behind
// its back, plugins that only receive raw device pointers through a C
// interface and have no CUDA memory API of their own, and code that must not
// be able to fail with out-of-memory in the middle of a step.  For them this
// entry point keeps its scratch in one array compiled into the library.
//
// The array is a file-scope device variable of NOALLOC_BYTES bytes: every
// GPU that loads the library holds it until the process exits.  Its device
// address is looked up once per device (cudaGetSymbolAddress, on the first
// call made with that device current) and passed to the kernels.  Every call
// shares the array and finds in it whatever the last call left, so each call
// clears the part that must start at zero (the completion counter and the
// statistics) on its stream before its kernels run; two calls whose work
// overlaps on the GPU (different streams, or different host threads) race on
// the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "zero_internal.h"

namespace zdp {

// Reduced-gradient elements the two-pass path can hold (all shards of one
// call together, each shard's region rounded up to 128 elements).
constexpr int64_t NOALLOC_MAX_GRAD_ELEMS = int64_t(1) << 21;
constexpr size_t NOALLOC_BYTES = WS_BYTES + 2 * (size_t)NOALLOC_MAX_GRAD_ELEMS;
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.
static int noalloc_scratch(unsigned char** out) {
    static std::mutex mu;
    static unsigned char* addr[NOALLOC_MAX_DEVICES] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "zero_shard_step_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) {
        set_error("zero_shard_step_noalloc: device index above 63");
        return ZERO_EINVAL;
    }
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "zero_shard_step_noalloc: cudaGetSymbolAddress of the scratch array");
        addr[dev] = static_cast<unsigned char*>(p);
    }
    *out = addr[dev];
    return ZERO_OK;
}

}  // namespace zdp

using namespace zdp;

extern "C" int zero_shard_step_noalloc(const void* const* grad_slices, int n_slices, int grad_dtype,
                                       const zero_shard* shards, int n_shards, void* flat_param, int param_dtype,
                                       const zero_hyper* hyper, float loss_scale, double extra_sumsq,
                                       int extra_overflow, zero_result* result, void* stream) {
    if (n_shards < 0 || n_shards > ZERO_MAX_SHARDS || (n_shards > 0 && !shards) || !hyper) {
        set_error("zero_shard_step_noalloc: bad shards or hyper argument");
        return n_shards > ZERO_MAX_SHARDS ? ZERO_ELIMIT : ZERO_EINVAL;
    }
    unsigned char* scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc != ZERO_OK) return rc;

    // The same path choice as zero_shard_step: two passes when clipping or
    // when a shard updates its state in place; then the reduced gradients
    // live in the scratch array instead of caller buffers.
    bool two_pass = hyper->max_grad_norm > 0.0f;
    for (int i = 0; i < n_shards && !two_pass; ++i)
        if (shards[i].numel > 0 && (shards[i].master_out == shards[i].master_in ||
                                    shards[i].m_out == shards[i].m_in || shards[i].v_out == shards[i].v_in))
            two_pass = true;
    zero_shard local[ZERO_MAX_SHARDS];
    if (n_shards > 0) std::memcpy(local, shards, sizeof(zero_shard) * n_shards);
    if (two_pass) {
        int64_t used = 0;
        for (int i = 0; i < n_shards; ++i) {
            if (local[i].numel < 0) {
                set_error("zero_shard_step_noalloc: negative shard size");
                return ZERO_EINVAL;
            }
            local[i].grad_shard = scratch + WS_BYTES + 2 * (size_t)used;
            used += (local[i].numel + 127) / 128 * 128;
            if (used > NOALLOC_MAX_GRAD_ELEMS) {
                set_error("zero_shard_step_noalloc: the shards' reduced gradients need more than the built-in "
                          "scratch holds (2097152 elements in all, each shard rounded up to 128); use "
                          "zero_shard_step with caller-provided buffers");
                return ZERO_ELIMIT;
            }
        }
    }
    // The completion counter and the statistics must start at zero.
    cudaError_t e = cudaMemsetAsync(scratch, 0, WS_PARTIALS, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "zero_shard_step_noalloc: clearing the scratch counter");
    return zero_shard_step(grad_slices, n_slices, grad_dtype, local, n_shards, flat_param, param_dtype, hyper,
                           loss_scale, extra_sumsq, extra_overflow, scratch, WS_BYTES, result, stream);
}
