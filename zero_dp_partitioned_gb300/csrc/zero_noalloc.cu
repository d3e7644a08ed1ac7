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
// GPU that loads the library holds it until the process exits.  Host code
// only has a stand-in for its name, so each call looks up its device address
// on the current device (cudaGetSymbolAddress; the first lookup on a device
// loads the library's device code there) and passes that to the kernels.
// Looking it up on every call, rather than caching it, keeps the address
// right after a device reset.  Every call shares the array and finds in it
// whatever the last call left, so each call clears the part that must start
// at zero (the completion counter and the statistics) on its stream before
// its kernels run; two calls whose work overlaps on the GPU (different
// streams, or different host threads) race on the array and must be
// serialised by the caller.
//
// Order of a call: host-side checks, the address lookup, the planning of the
// step (every argument check of zero_shard_step), and only then the clearing
// and the kernels -- a call that fails with an argument error enqueues
// nothing and leaves the array as it was.
#include <cuda_runtime.h>

#include <cstring>
#include <string>

#include "zero_internal.h"

namespace zdp {

// Reduced-gradient elements the two-pass path can hold (all shards of one
// call together, each shard's region rounded up to 128 elements).
constexpr int64_t NOALLOC_MAX_GRAD_ELEMS = int64_t(1) << 21;
constexpr size_t NOALLOC_BYTES = WS_BYTES + 2 * (size_t)NOALLOC_MAX_GRAD_ELEMS;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

// Device address of g_noalloc_scratch on the current device.
static int noalloc_scratch(unsigned char** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "zero_shard_step_noalloc: cudaGetSymbolAddress of the scratch array");
    *out = static_cast<unsigned char*>(p);
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
    // The same path choice as zero_shard_step: two passes when clipping or
    // when a shard updates its state in place; then the reduced gradients
    // live in the scratch array instead of caller buffers.
    bool two_pass = hyper->max_grad_norm > 0.0f;
    for (int i = 0; i < n_shards && !two_pass; ++i)
        if (shards[i].numel > 0 && (shards[i].master_out == shards[i].master_in ||
                                    shards[i].m_out == shards[i].m_in || shards[i].v_out == shards[i].v_in))
            two_pass = true;
    int64_t grad_at[ZERO_MAX_SHARDS];          // each shard's first reduced-gradient element in the scratch
    if (two_pass) {
        int64_t used = 0;
        for (int i = 0; i < n_shards; ++i) {
            if (shards[i].numel < 0) {
                set_error("zero_shard_step_noalloc: negative shard size");
                return ZERO_EINVAL;
            }
            grad_at[i] = used;
            used += (shards[i].numel + 127) / 128 * 128;
            if (used > NOALLOC_MAX_GRAD_ELEMS) {
                set_error("zero_shard_step_noalloc: the shards' reduced gradients need more than the built-in "
                          "scratch holds (2097152 elements in all, each shard rounded up to 128); use "
                          "zero_shard_step with caller-provided buffers");
                return ZERO_ELIMIT;
            }
        }
    }
    unsigned char* scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc != ZERO_OK) return rc;
    zero_shard local[ZERO_MAX_SHARDS];
    if (n_shards > 0) std::memcpy(local, shards, sizeof(zero_shard) * n_shards);
    if (two_pass)
        for (int i = 0; i < n_shards; ++i) local[i].grad_shard = scratch + WS_BYTES + 2 * (size_t)grad_at[i];
    StepPlan sp;
    rc = plan_step(sp, grad_slices, n_slices, grad_dtype, local, n_shards, flat_param, param_dtype, hyper, loss_scale,
                   extra_sumsq, extra_overflow, scratch, WS_BYTES, result);
    if (rc != ZERO_OK) return rc;
    // The completion counter and the statistics must start at zero.
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = cudaMemsetAsync(scratch, 0, WS_PARTIALS, s);
    if (e != cudaSuccess) return cuda_fail(e, "zero_shard_step_noalloc: clearing the scratch counter");
    return run_step(sp, s);
}
