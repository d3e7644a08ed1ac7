// zero_host.cu -- zero_shard_step_host: the step with its gradients in
// page-locked host memory and its parameters returned there.  The host link
// is the bound (211 GB/s up on GB300, whether the copy engine or SM loads
// move the bytes), so the step is cut into chunks and every chunk's kernels
// run while later chunks are still crossing: one stream of the library's
// copies the slices' chunks up into a ring of device slots, the caller's
// stream reduces and updates each chunk as it lands, and a second stream of
// the library's copies each updated chunk's parameters down, beside the
// uploads (the link carries both directions at once).
#include <cstring>
#include <map>
#include <mutex>

#include "zero_internal.h"

namespace zdp {

constexpr int HOST_RING = 4;              // chunk slots in the caller's device ring
constexpr int64_t HOST_CHUNK_ALIGN = 64;  // elements: every slot starts on a 128-byte line

// The streams and events of the host-buffer step on one device, made on the
// first call there and kept for the life of the process.
struct HostLane {
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, up_done = nullptr, down_done = nullptr;
    cudaEvent_t landed[HOST_RING] = {}, read[HOST_RING] = {};
};

static std::mutex g_lane_mu;                       // held for a whole call: calls are serialised
static std::map<int, HostLane> g_lanes;

static void drop_lane(HostLane& l) {
    cudaEvent_t* evs[] = {&l.start, &l.up_done, &l.down_done};
    for (cudaEvent_t* ev : evs)
        if (*ev) cudaEventDestroy(*ev);
    for (int k = 0; k < HOST_RING; ++k) {
        if (l.landed[k]) cudaEventDestroy(l.landed[k]);
        if (l.read[k]) cudaEventDestroy(l.read[k]);
    }
    if (l.up) cudaStreamDestroy(l.up);
    if (l.down) cudaStreamDestroy(l.down);
    l = HostLane{};
}

static int make_lane(HostLane& l) {
    cudaError_t e = cudaStreamCreateWithFlags(&l.up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&l.down, cudaStreamNonBlocking);
    cudaEvent_t* evs[] = {&l.start, &l.up_done, &l.down_done};
    for (cudaEvent_t* ev : evs)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int k = 0; k < HOST_RING && e == cudaSuccess; ++k) {
        e = cudaEventCreateWithFlags(&l.landed[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&l.read[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) drop_lane(l);
    return cuda_fail(e, "zero_shard_step_host: creating its streams and events");
}

// Host memory the copy engines can move asynchronously (page-locked); its
// device address when the device can load and store it (else NULL).
static bool page_locked(const void* p, void** dev_addr) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (dev_addr) *dev_addr = at.devicePointer;
    return at.type == cudaMemoryTypeHost;
}

// The chunk's piece of shard s as a shard of its own, reading slot-relative
// gradients (grad_offset 0) and writing its own state and parameter range.
static zero_shard sub_shard(const zero_shard& z, int64_t lo, int64_t hi) {
    zero_shard c = z;
    c.numel = hi - lo;
    c.grad_offset = 0;
    c.param_offset = z.param_offset + lo;
    c.master_in = z.master_in + lo;
    c.m_in = z.m_in + lo;
    c.v_in = z.v_in + lo;
    c.master_out = z.master_out + lo;
    c.m_out = z.m_out + lo;
    c.v_out = z.v_out + lo;
    c.grad_shard = z.grad_shard ? static_cast<void*>(static_cast<uint16_t*>(z.grad_shard) + lo) : nullptr;
    return c;
}

// Everything the step enqueues, in order: the copies up on the lane's first
// stream, each chunk's pass on the caller's stream as the chunk lands, the
// copies down on the lane's second stream, then the decision (or the apply
// pass and the shards' copies down).  Returns at the first failed call.
static int enqueue_host_step(HostLane& lane, const StepArgs& base, const void* const* host_grad_slices, int n_slices,
                             int grad_dtype, const zero_shard* shards, int n_shards, void* flat_param,
                             int param_dtype, void* host_param, void* host_param_dev, void* staging, int64_t chunk,
                             bool fused, cudaStream_t s) {
    const size_t esz = 2;
    int rc;
#define HOST_TRY(call, what)                                                                \
    do {                                                                                    \
        if ((rc = cuda_fail((call), "zero_shard_step_host: " what)) != ZERO_OK) return rc; \
    } while (0)
    HOST_TRY(cudaEventRecord(lane.start, s), "event");
    HOST_TRY(cudaStreamWaitEvent(lane.up, lane.start, 0), "event");
    HOST_TRY(cudaStreamWaitEvent(lane.down, lane.start, 0), "event");
    if (!any_elements(base)) HOST_TRY(cudaMemsetAsync(base.stats, 0, sizeof(zero_stats), s), "clearing the statistics");

    int64_t j = 0;                        // chunks so far; chunk j uses slot j mod HOST_RING
    for (int si = 0; si < n_shards; ++si)
    for (int64_t lo = 0; lo < shards[si].numel; lo += chunk, ++j) {
        const int k = (int)(j % HOST_RING);
        const zero_shard& z = shards[si];
        const int64_t hi = lo + chunk < z.numel ? lo + chunk : z.numel;
        const int64_t n = hi - lo;
        // up: slot k once the pass that read it last is done
        const void* slot[ZERO_MAX_SLICES];
        HOST_TRY(cudaStreamWaitEvent(lane.up, lane.read[k], 0), "event");
        for (int r = 0; r < n_slices; ++r) {
            char* dst = static_cast<char*>(staging) + ((size_t)k * n_slices + r) * (size_t)chunk * esz;
            const char* src = static_cast<const char*>(host_grad_slices[r]) + (size_t)(z.grad_offset + lo) * esz;
            HOST_TRY(cudaMemcpyAsync(dst, src, (size_t)n * esz, cudaMemcpyHostToDevice, lane.up), "copy up");
            slot[r] = dst;
        }
        HOST_TRY(cudaEventRecord(lane.landed[k], lane.up), "event");
        // the chunk's pass, on the caller's stream
        HOST_TRY(cudaStreamWaitEvent(s, lane.landed[k], 0), "event");
        StepArgs a = base;
        const zero_shard part = sub_shard(z, lo, hi);
        pack_slices(a, slot, n_slices);
        pack_shards(a, &part, 1, fused ? 1 : 2);
        a.accumulate = j > 0 ? 1 : 0;
        if (fused) {
            const int vec = vec8_ok(a, 1) ? 8 : 1;
            number_tiles(a, vec, HEAD_GRADS);
            const int grid = grid_for(fused_fn(a, grad_dtype, param_dtype, vec), a.n_tiles,
                                      n_slices <= FEW_SLICES ? BPS_FUSED_FEW : BPS_FUSED_MANY);
            if ((rc = launch_fused(a, grad_dtype, param_dtype, vec, grid, s)) != ZERO_OK) return rc;
        } else {
            const int vec = vec8_ok(a, 2) ? 8 : 1;
            number_tiles(a, vec, HEAD_GRADS);
            if ((rc = launch_reduce(a, grad_dtype, vec, s, false)) != ZERO_OK) return rc;
        }
        HOST_TRY(cudaEventRecord(lane.read[k], s), "event");
        // down: the chunk's parameters (final unless the commit skips the step)
        if (fused && host_param) {
            HOST_TRY(cudaStreamWaitEvent(lane.down, lane.read[k], 0), "event");
            const size_t off = (size_t)(z.param_offset + lo) * esz;
            HOST_TRY(cudaMemcpyAsync(static_cast<char*>(host_param) + off, static_cast<const char*>(flat_param) + off,
                                     (size_t)n * esz, cudaMemcpyDeviceToHost, lane.down),
                     "copy down");
        }
    }
    HOST_TRY(cudaEventRecord(lane.up_done, lane.up), "event");
    HOST_TRY(cudaEventRecord(lane.down_done, lane.down), "event");
    HOST_TRY(cudaStreamWaitEvent(s, lane.up_done, 0), "event");
    HOST_TRY(cudaStreamWaitEvent(s, lane.down_done, 0), "event");

    if (fused) {
        // the decision; a skipped step's parameters restored on the device and,
        // after the copies down have landed, in host memory too
        StepArgs a = base;
        if ((rc = launch_commit(a, s)) != ZERO_OK) return rc;
        if ((rc = launch_recover(a, param_dtype, s)) != ZERO_OK) return rc;
        if (host_param) {
            a.flat_param = host_param_dev;
            if ((rc = launch_recover(a, param_dtype, s)) != ZERO_OK) return rc;
        }
        return ZERO_OK;
    }
    StepArgs a = base;
    pack_shards(a, shards, n_shards, 3);
    const int vec = vec8_ok(a, 3) ? 8 : 1;
    number_tiles(a, vec, HEAD_STATE);
    if ((rc = launch_apply(a, grad_dtype, param_dtype, vec, s)) != ZERO_OK) return rc;
    if (host_param)
        for (int i = 0; i < n_shards; ++i) {
            if (shards[i].numel == 0) continue;
            const size_t off = (size_t)shards[i].param_offset * esz;
            HOST_TRY(cudaMemcpyAsync(static_cast<char*>(host_param) + off, static_cast<const char*>(flat_param) + off,
                                     (size_t)shards[i].numel * esz, cudaMemcpyDeviceToHost, s),
                     "copy down");
        }
#undef HOST_TRY
    return ZERO_OK;
}

}  // namespace zdp

using namespace zdp;

extern "C" int zero_shard_step_host(const void* const* host_grad_slices, int n_slices, int grad_dtype,
                                    const zero_shard* shards, int n_shards, void* flat_param, int param_dtype,
                                    void* host_param, const zero_hyper* hyper, float loss_scale, double extra_sumsq,
                                    int extra_overflow, void* staging, size_t staging_bytes, void* workspace,
                                    size_t workspace_bytes, zero_result* result, void* stream) {
    // ---- every argument check first: an error enqueues nothing
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    int rc;
    if ((rc = check_hyper(hyper, loss_scale)) != ZERO_OK) return rc;
    if (!result || !aligned(result, 8)) return fail(ZERO_EINVAL, "result is NULL or not 8-byte aligned");
    StepArgs base;
    std::memset(&base, 0, sizeof base);
    if ((rc = pack_slices(base, host_grad_slices, n_slices)) != ZERO_OK) return rc;
    for (int r = 0; r < n_slices; ++r)
        if (!page_locked(host_grad_slices[r], nullptr))
            return fail(ZERO_EINVAL, "zero_shard_step_host: a gradient slice is not page-locked host memory");
    void* host_param_dev = nullptr;
    if (host_param) {
        if (!aligned(host_param, 2)) return fail(ZERO_EALIGN, "host_param not 2-byte aligned");
        if (!page_locked(host_param, &host_param_dev) || !host_param_dev)
            return fail(ZERO_EINVAL, "zero_shard_step_host: host_param is not page-locked host memory the device "
                                     "can address");
    }
    if (!staging || !aligned(staging, 16)) return fail(ZERO_EALIGN, "staging is NULL or not 16-byte aligned");
    const int64_t chunk =
        (int64_t)(staging_bytes / ((size_t)HOST_RING * (size_t)n_slices * 2)) / HOST_CHUNK_ALIGN * HOST_CHUNK_ALIGN;
    if (chunk < HOST_CHUNK_ALIGN)
        return fail(ZERO_EWORKSPACE, "zero_shard_step_host: staging holds fewer than 64 elements per chunk");
    if ((rc = check_workspace(base, workspace, workspace_bytes)) != ZERO_OK) return rc;
    const bool fused = hyper->max_grad_norm <= 0.0f && !state_in_place(shards, n_shards);
    if ((rc = pack_shards(base, shards, n_shards, fused ? 1 : 2)) != ZERO_OK) return rc;
    if (!fused && (rc = pack_shards(base, shards, n_shards, 3)) != ZERO_OK) return rc;
    if (any_elements(base) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");

    // the step's arguments shared by every chunk, the commit and the apply
    base.flat_param = flat_param;
    base.sc = adam_scalars(*hyper);
    base.loss_scale = (double)loss_scale;
    base.k = (float)(1.0 / (double)loss_scale);
    base.max_norm = (double)hyper->max_grad_norm;
    base.extra_sumsq = extra_sumsq;
    base.extra_overflow = extra_overflow ? 1 : 0;
    base.result = result;
    base.stats = reinterpret_cast<zero_stats*>(static_cast<char*>(workspace) + WS_STATS);

    // ---- the pipeline
    std::lock_guard<std::mutex> guard(g_lane_mu);
    int dev = 0;
    if ((rc = cuda_fail(cudaGetDevice(&dev), "zero_shard_step_host: device query")) != ZERO_OK) return rc;
    HostLane& lane = g_lanes[dev];
    if (!lane.up && (rc = make_lane(lane)) != ZERO_OK) {
        g_lanes.erase(dev);
        return rc;
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = enqueue_host_step(lane, base, host_grad_slices, n_slices, grad_dtype, shards, n_shards, flat_param,
                           param_dtype, host_param, host_param_dev, staging, chunk, fused, s);
    if (rc != ZERO_OK) {
        // an enqueue failed part way: the caller's stream still waits for what
        // the library's streams hold (best effort; the first error is reported)
        cudaEventRecord(lane.up_done, lane.up);
        cudaEventRecord(lane.down_done, lane.down);
        cudaStreamWaitEvent(s, lane.up_done, 0);
        cudaStreamWaitEvent(s, lane.down_done, 0);
    }
    return rc;
}
