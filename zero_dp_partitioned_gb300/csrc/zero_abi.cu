// zero_abi.cu -- the C entry points declared in include/zero.h: argument
// checks, choice of the single- or two-pass path, packing of the kernel
// arguments, and the host-only planner and memory model.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <utility>

#include "zero_internal.h"
#include "zero_tma.cuh"

namespace zdp {

static thread_local std::string g_err;

void set_error(const std::string& msg) { g_err = msg; }

int cuda_fail(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ZERO_OK;
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return ZERO_ECUDA;
}

int grid_for_smem(const void* func, int64_t n_tiles, size_t dynamic_smem, int max_per_sm) {
    // Occupancy and SM count are cached per (device, kernel, dynamic shared
    // memory): a process may see GPUs with different SM counts.
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, size_t>, int> per_sm;   // -> resident blocks per SM
    static std::map<int, int> sms;                                        // device -> SM count
    int dev = 0;
    cudaGetDevice(&dev);
    int nb = 0, n_sm = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        auto si = sms.find(dev);
        if (si == sms.end()) {
            if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1)
                n_sm = 1;
            sms[dev] = n_sm;
        } else {
            n_sm = si->second;
        }
        const auto key = std::make_tuple(dev, func, dynamic_smem);
        auto it = per_sm.find(key);
        if (it == per_sm.end()) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, func, TILE_THREADS, dynamic_smem) != cudaSuccess ||
                nb < 1)
                nb = 1;
            per_sm[key] = nb;
        } else {
            nb = it->second;
        }
    }
    if (max_per_sm > 0 && nb > max_per_sm) nb = max_per_sm;
    int64_t g = (int64_t)nb * n_sm;
    if (g > n_tiles) g = n_tiles;
    if (g > MAX_BLOCKS) g = MAX_BLOCKS;
    if (g < 1) g = 1;
    return (int)g;
}

int grid_for(const void* func, int64_t n_tiles, int max_per_sm) {
    return grid_for_smem(func, n_tiles, 0, max_per_sm);
}

size_t smem_capping(const void* func, int blocks) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int>, size_t> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> g(mu);
    const auto key = std::make_tuple(dev, func, blocks);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    size_t smem = 0;
    int occ = 0, per_sm = 0, reserved = 0, optin = 0;
    bool refused = false;
    if (blocks > 0) {
        refused = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, func, TILE_THREADS, 0) != cudaSuccess ||
                  cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
                  cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
                  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess;
        // the smallest multiple of 16 bytes beside which a (blocks + 1)-th block no longer fits
        const long want = ((long)per_sm / (blocks + 1) - reserved + 16 + 15) / 16 * 16;
        if (!refused && occ > blocks && want > 0 && want <= optin) {
            int got = 0;
            refused = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)want) != cudaSuccess ||
                      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&got, func, TILE_THREADS, (size_t)want) !=
                          cudaSuccess;
            if (!refused && got == blocks) smem = (size_t)want;
        }
    }
    if (refused) cudaGetLastError();   // a refusal costs only the cap: leave no error for a later launch check
    cache[key] = smem;
    return smem;
}

// Tries per bounded wait of the TMA gather, from the environment (tests force
// a limit of 0 to exercise the timeout path without hanging anything).
static unsigned spin_limit() {
    const char* e = std::getenv("ZERO_GB300_SPIN_LIMIT");
    if (!e) return SPIN_LIMIT;
    return (unsigned)std::strtoul(e, nullptr, 10);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool valid_dtype(int d) { return d == ZERO_F16 || d == ZERO_BF16; }

int fail(int code, const char* msg) {
    set_error(msg);
    return code;
}

// Host scalars of one AdamW step: each computed in fp64 from the fp32
// hyper-parameters and rounded once to fp32; the bias corrections are folded
// into ss = lr / (1 - b1^t) and rb2 = 1 / sqrt(1 - b2^t).
AdamScalars adam_scalars(const zero_hyper& h) {
    const double t = (double)h.step;
    const double bc1 = 1.0 - std::pow((double)h.beta1, t);
    const double bc2 = 1.0 - std::pow((double)h.beta2, t);
    AdamScalars c;
    c.b1 = h.beta1;
    c.b2 = h.beta2;
    c.omb1 = (float)(1.0 - (double)h.beta1);
    c.omb2 = (float)(1.0 - (double)h.beta2);
    c.eps = h.eps;
    c.wdf = (float)(1.0 - (double)h.lr * (double)h.weight_decay);
    c.ss = (float)((double)h.lr / bc1);
    c.rb2 = (float)(1.0 / std::sqrt(bc2));
    return c;
}

// Common checks of slices and shards; fills the shard part of a and the tile
// numbering for vector width vec.  need: 1 = fused (state in/out), 2 = reduce
// (grad_shard out), 3 = apply (grad_shard in, state in/out).
int pack_shards(StepArgs& a, const zero_shard* shards, int n_shards, int need) {
    if (n_shards < 0) return fail(ZERO_EINVAL, "n_shards < 0");
    if (n_shards > ZERO_MAX_SHARDS) return fail(ZERO_ELIMIT, "more than ZERO_MAX_SHARDS shards");
    if (n_shards > 0 && !shards) return fail(ZERO_EINVAL, "shards is NULL");
    a.n_shards = n_shards;
    for (int i = 0; i < n_shards; ++i) {
        const zero_shard& s = shards[i];
        if (s.numel < 0 || s.grad_offset < 0 || s.param_offset < 0)
            return fail(ZERO_EINVAL, "negative shard size or offset");
        if (s.numel > 0) {
            if (need != 2) {
                if (!s.master_in || !s.m_in || !s.v_in || !s.master_out || !s.m_out || !s.v_out)
                    return fail(ZERO_EINVAL, "shard state pointer is NULL");
                const void* ps[6] = {s.master_in, s.m_in, s.v_in, s.master_out, s.m_out, s.v_out};
                for (const void* p : ps)
                    if (!aligned(p, 4)) return fail(ZERO_EALIGN, "fp32 state pointer not 4-byte aligned");
            }
            if (need != 1) {
                if (!s.grad_shard) return fail(ZERO_EINVAL, "grad_shard is NULL (the two-pass path needs it)");
                if (!aligned(s.grad_shard, 2)) return fail(ZERO_EALIGN, "grad_shard not 2-byte aligned");
            }
        }
        ShardDev& d = a.shards[i];
        d.numel = s.numel;
        d.grad_off = s.grad_offset;
        d.param_off = s.param_offset;
        d.mi = s.master_in;
        d.mmi = s.m_in;
        d.vi = s.v_in;
        d.mo = s.master_out;
        d.mmo = s.m_out;
        d.vo = s.v_out;
        d.gshard = s.grad_shard;
    }
    return ZERO_OK;
}

// Elements done one by one at the start of a shard so that the vector loop
// starts where the dominant stream sits on a 128-byte boundary.  Shards start
// wherever the partition puts them (the pages pad only to 2 * world_size
// elements), and a misaligned 128-bit stream costs extra DRAM reads: the
// GPT-2 1.5B fused pass read 48.0 GB per launch against 43.6 GB of
// algorithmic bytes with its shards 48 bytes (bf16) / 96 bytes (fp32) past a
// 128-byte line, and exactly 43.6 GB, 7% faster, with aligned shards.  The
// head must be a multiple of 8 elements so every stream stays 16-byte
// aligned for the vector loop; otherwise no head is taken.
static int64_t shard_head(const StepArgs& a, const ShardDev& d, int kind) {
    if (kind == HEAD_NONE || d.numel == 0) return 0;
    int64_t h;
    if (kind == HEAD_GRADS) {
        const uintptr_t g = reinterpret_cast<uintptr_t>(static_cast<const uint16_t*>(a.slices[0]) + d.grad_off);
        h = (int64_t)((128u - (g & 127u)) & 127u) / 2;
    } else {
        const uintptr_t m = reinterpret_cast<uintptr_t>(d.mi);
        h = (int64_t)((128u - (m & 127u)) & 127u) / 4;
    }
    return (h % 8) ? 0 : h;
}

void number_tiles(StepArgs& a, int vec, int kind) {
    const int64_t tile = (int64_t)TILE_THREADS * vec;
    int64_t t = 0;
    for (int i = 0; i < a.n_shards; ++i) {
        ShardDev& d = a.shards[i];
        d.head = vec == 8 ? shard_head(a, d, kind) : 0;
        if (d.head > d.numel) d.head = d.numel;
        d.tile_begin = t;
        const int64_t rest = d.numel - d.head;
        t += d.numel == 0 ? 0 : (rest > 0 ? (rest + tile - 1) / tile : 1);
    }
    a.n_tiles = t;
}

int pack_slices(StepArgs& a, const void* const* slices, int n_slices) {
    if (!slices) return fail(ZERO_EINVAL, "grad_slices is NULL");
    if (n_slices < 1) return fail(ZERO_EINVAL, "n_slices < 1");
    if (n_slices > ZERO_MAX_SLICES) return fail(ZERO_ELIMIT, "more than ZERO_MAX_SLICES slices");
    a.n_slices = n_slices;
    for (int r = 0; r < n_slices; ++r) {
        if (!slices[r]) return fail(ZERO_EINVAL, "a gradient slice is NULL");
        if (!aligned(slices[r], 2)) return fail(ZERO_EALIGN, "gradient slice not 2-byte aligned");
        a.slices[r] = slices[r];
    }
    a.divisor = (float)n_slices;
    return ZERO_OK;
}

// 16-byte vectors are possible when every gradient address a shard starts at
// and every pointer the vector path loads from are 16-byte aligned.
// The apply pass's 256-bit state accesses: every shard's six state arrays
// 32-byte aligned (the vector loop's element index is a multiple of 8, and
// so is the head), and its gradient stream starting on a 128-byte line.
// Measured on GB300 (sources alternated in one call): the pass on one
// 2.0B-element shard, every stream on a line, 8.494 ms against 8.629 ms with
// 128-bit accesses; on eight 195M-element shards cut from one
// averaged-gradient buffer (gradient streams 16-112 bytes off a line), 7.08
// against 6.99 ms (with a per-vector choice), so those keep 128-bit accesses.
bool state_wide(const StepArgs& a) {
    for (int i = 0; i < a.n_shards; ++i) {
        const ShardDev& d = a.shards[i];
        if (d.numel == 0) continue;
        const uintptr_t st = reinterpret_cast<uintptr_t>(d.mi) | reinterpret_cast<uintptr_t>(d.mmi) |
                             reinterpret_cast<uintptr_t>(d.vi) | reinterpret_cast<uintptr_t>(d.mo) |
                             reinterpret_cast<uintptr_t>(d.mmo) | reinterpret_cast<uintptr_t>(d.vo);
        const uintptr_t g = reinterpret_cast<uintptr_t>(static_cast<const uint16_t*>(d.gshard) + d.head);
        if (!d.mi || !d.gshard || (st & 31u) != 0 || (g & 127u) != 0) return false;
    }
    return true;
}

// The fused pass's 256-bit state accesses: every shard's six state arrays
// 32-byte aligned.  Measured on GB300 (sources alternated in one call): the
// 8-slice GPT-2 pass 9.354 against 9.399 ms, the 4-slice ZeRO-3 partial pass
// 0.2977 against 0.2999 ms, the 64-slice pass unchanged (2.631 against 2.632
// ms).
bool fused_state_wide(const StepArgs& a) {
    for (int i = 0; i < a.n_shards; ++i) {
        const ShardDev& d = a.shards[i];
        if (d.numel == 0) continue;
        const uintptr_t st = reinterpret_cast<uintptr_t>(d.mi) | reinterpret_cast<uintptr_t>(d.mmi) |
                             reinterpret_cast<uintptr_t>(d.vi) | reinterpret_cast<uintptr_t>(d.mo) |
                             reinterpret_cast<uintptr_t>(d.mmo) | reinterpret_cast<uintptr_t>(d.vo);
        if (!d.mi || (st & 31u) != 0) return false;
    }
    return true;
}

bool vec8_ok(const StepArgs& a, int need) {
    for (int i = 0; i < a.n_shards; ++i) {
        const ShardDev& d = a.shards[i];
        if (d.numel == 0) continue;
        if (need != 3)
            for (int r = 0; r < a.n_slices; ++r)
                if (!aligned(static_cast<const uint16_t*>(a.slices[r]) + d.grad_off, 16)) return false;
        if (need != 2) {
            const void* ps[6] = {d.mi, d.mmi, d.vi, d.mo, d.mmo, d.vo};
            for (const void* p : ps)
                if (!aligned(p, 16)) return false;
        }
        if (need == 3 && !aligned(d.gshard, 16)) return false;
    }
    return true;
}

int check_workspace(StepArgs& a, void* ws, size_t ws_bytes) {
    if (!ws) return fail(ZERO_EWORKSPACE, "workspace is NULL");
    if (ws_bytes < WS_BYTES) return fail(ZERO_EWORKSPACE, "workspace smaller than zero_workspace_bytes()");
    if (!aligned(ws, 16)) return fail(ZERO_EALIGN, "workspace not 16-byte aligned");
    char* w = static_cast<char*>(ws);
    a.counter = reinterpret_cast<unsigned*>(w + WS_COUNTER);
    a.partials = reinterpret_cast<double*>(w + WS_PARTIALS);
    a.block_flags = reinterpret_cast<int*>(w + WS_FLAGS);
    return ZERO_OK;
}

int check_hyper(const zero_hyper* h, float loss_scale) {
    if (!h) return fail(ZERO_EINVAL, "hyper is NULL");
    if (h->step < 1) return fail(ZERO_EINVAL, "hyper->step must be >= 1");
    if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale)) return fail(ZERO_EINVAL, "loss_scale must be finite and > 0");
    return ZERO_OK;
}

bool any_elements(const StepArgs& a) {
    for (int i = 0; i < a.n_shards; ++i)
        if (a.shards[i].numel > 0) return true;
    return false;
}

bool state_in_place(const zero_shard* shards, int n_shards) {
    for (int i = 0; i < n_shards && shards; ++i)
        if (shards[i].numel > 0 && (shards[i].master_out == shards[i].master_in ||
                                    shards[i].m_out == shards[i].m_in || shards[i].v_out == shards[i].v_in))
            return true;
    return false;
}

// Every argument check of zero_shard_step, then the packed kernel arguments
// and the path: nothing is enqueued, so a failing call leaves the device and
// the workspace untouched.
int plan_step(StepPlan& sp, const void* const* grad_slices, int n_slices, int grad_dtype, const zero_shard* shards,
              int n_shards, void* flat_param, int param_dtype, const zero_hyper* hyper, float loss_scale,
              double extra_sumsq, int extra_overflow, void* workspace, size_t workspace_bytes, zero_result* result) {
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    int rc;
    if ((rc = check_hyper(hyper, loss_scale)) != ZERO_OK) return rc;
    if (!result || !aligned(result, 8)) return fail(ZERO_EINVAL, "result is NULL or not 8-byte aligned");
    StepArgs& a = sp.a;
    std::memset(&a, 0, sizeof a);
    if ((rc = pack_slices(a, grad_slices, n_slices)) != ZERO_OK) return rc;
    if ((rc = check_workspace(a, workspace, workspace_bytes)) != ZERO_OK) return rc;

    // One fused pass needs a second state set to write (the skip decision is
    // only known at its end) and no clipping (the norm is needed before the
    // first update); otherwise reduce, then apply.
    bool fused = hyper->max_grad_norm <= 0.0f;
    for (int i = 0; fused && i < n_shards && shards; ++i)
        if (shards[i].numel > 0 && (shards[i].master_out == shards[i].master_in ||
                                    shards[i].m_out == shards[i].m_in || shards[i].v_out == shards[i].v_in))
            fused = false;
    if ((rc = pack_shards(a, shards, n_shards, fused ? 1 : 2)) != ZERO_OK) return rc;
    if (!fused && (rc = pack_shards(a, shards, n_shards, 3)) != ZERO_OK) return rc;
    if (any_elements(a) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    a.flat_param = flat_param;
    a.sc = adam_scalars(*hyper);
    a.loss_scale = (double)loss_scale;
    a.max_norm = (double)hyper->max_grad_norm;
    a.extra_sumsq = extra_sumsq;
    a.extra_overflow = extra_overflow ? 1 : 0;
    a.result = result;
    if (fused) {
        a.k = (float)(1.0 / (double)loss_scale);
    } else {
        a.stats = reinterpret_cast<zero_stats*>(static_cast<char*>(workspace) + WS_STATS);
        a.accumulate = 0;
    }
    sp.fused = fused;
    sp.gdt = grad_dtype;
    sp.pdt = param_dtype;
    return ZERO_OK;
}

// The kernels of a planned step: the fused pass and the parameter restore
// check, or the reduce and apply passes.
int run_step(StepPlan& sp, cudaStream_t s) {
    StepArgs& a = sp.a;
    int rc;
    if (sp.fused) {
        const int vec = vec8_ok(a, 1) ? 8 : 1;
        number_tiles(a, vec, HEAD_GRADS);
        const int grid = grid_for(fused_fn(a, sp.gdt, sp.pdt, vec), a.n_tiles,
                                  a.n_slices <= FEW_SLICES ? BPS_FUSED_FEW : BPS_FUSED_MANY);
        if ((rc = launch_fused(a, sp.gdt, sp.pdt, vec, grid, s)) != ZERO_OK) return rc;
        return launch_recover(a, sp.pdt, s);
    }
    int vec = vec8_ok(a, 2) ? 8 : 1;
    number_tiles(a, vec, HEAD_GRADS);
    if ((rc = launch_reduce(a, sp.gdt, vec, s)) != ZERO_OK) return rc;
    vec = vec8_ok(a, 3) ? 8 : 1;
    number_tiles(a, vec, HEAD_STATE);
    return launch_apply(a, sp.gdt, sp.pdt, vec, s);
}

}  // namespace zdp

using namespace zdp;

extern "C" {

const char* zero_last_error(void) { return g_err.c_str(); }

size_t zero_workspace_bytes(void) { return WS_BYTES; }

int zero_plan(const int64_t* numels, int n_tensors, int world_size, int mode, int64_t* tensor_offsets,
              int64_t* rank_offsets, int64_t* rank_numels, int64_t* padded_total, int64_t* padding) {
    if (n_tensors < 0 || world_size < 1 || (mode != ZERO_PLAN_PADDED && mode != ZERO_PLAN_UNPADDED))
        return fail(ZERO_EINVAL, "zero_plan: bad n_tensors, world_size or mode");
    if ((n_tensors > 0 && (!numels || !tensor_offsets)) || !rank_offsets || !rank_numels || !padded_total || !padding)
        return fail(ZERO_EINVAL, "zero_plan: NULL argument");
    int64_t total = 0;
    for (int i = 0; i < n_tensors; ++i) {
        if (numels[i] < 0) return fail(ZERO_EINVAL, "zero_plan: negative numel");
        tensor_offsets[i] = total;
        total += numels[i];
    }
    int64_t flat = total;
    if (mode == ZERO_PLAN_PADDED) {
        const int64_t q = 2 * (int64_t)world_size;      // 16-bit elements: shard starts on 4-byte boundaries
        flat = (total + q - 1) / q * q;
    }
    const int64_t base = flat / world_size, rem = flat % world_size;
    int64_t off = 0;
    for (int r = 0; r < world_size; ++r) {
        rank_offsets[r] = off;
        rank_numels[r] = base + (r < rem ? 1 : 0);
        off += rank_numels[r];
    }
    *padded_total = flat;
    *padding = flat - total;
    return ZERO_OK;
}

int zero_plan_intersections(const int64_t* tensor_offsets, const int64_t* numels, int n_tensors,
                            int64_t rank_offset, int64_t rank_numel, int64_t* out) {
    if (n_tensors < 0 || rank_offset < 0 || rank_numel < 0 || (n_tensors > 0 && (!tensor_offsets || !numels || !out)))
        return fail(ZERO_EINVAL, "zero_plan_intersections: bad argument");
    int rows = 0;
    const int64_t lo = rank_offset, hi = rank_offset + rank_numel;
    for (int i = 0; i < n_tensors; ++i) {
        const int64_t a = tensor_offsets[i], b = a + numels[i];
        const int64_t s = a > lo ? a : lo, e = b < hi ? b : hi;
        if (e <= s) continue;
        out[4 * rows + 0] = i;
        out[4 * rows + 1] = s - a;
        out[4 * rows + 2] = s - lo;
        out[4 * rows + 3] = e - s;
        ++rows;
    }
    return rows;
}

int zero_mem_model(double psi, double K, int n_d, int stage, double* bytes_out) {
    if (!bytes_out || n_d < 1 || stage < 0 || stage > 3 || !(psi >= 0.0) || !(K >= 0.0))
        return fail(ZERO_EINVAL, "zero_mem_model: bad argument");
    const double N = (double)n_d;
    double b = 0.0;
    switch (stage) {
    case 0: b = (4.0 + K) * psi; break;                 // DP: every rank holds everything
    case 1: b = 4.0 * psi + K * psi / N; break;         // P_os
    case 2: b = 2.0 * psi + (K + 2.0) * psi / N; break; // P_os+g
    default: b = (4.0 + K) * psi / N; break;            // P_os+g+p
    }
    *bytes_out = b;
    return ZERO_OK;
}

int zero_mem_model_plan(int64_t flat_numel, int64_t shard_numel, double K, int stage, int state_sets,
                        int64_t fp32_temp_numel, int64_t b16_temp_numel, double* bytes_out) {
    if (!bytes_out || flat_numel < 0 || shard_numel < 0 || !(K >= 0.0) || stage < 0 || stage > 3 ||
        state_sets < 1 || fp32_temp_numel < 0 || b16_temp_numel < 0)
        return fail(ZERO_EINVAL, "zero_mem_model_plan: bad argument");
    const double F = (double)flat_numel, n = (double)shard_numel;
    // P_os partitions the optimizer states, P_os+g the gradients too, P_os+g+p the parameters too
    bytes_out[0] = 2.0 * (stage == 3 ? n : F);
    bytes_out[1] = 2.0 * (stage >= 2 ? n : F);
    bytes_out[2] = K * (double)state_sets * (stage == 0 ? F : n);
    bytes_out[3] = 4.0 * (double)fp32_temp_numel + 2.0 * (double)b16_temp_numel;
    bytes_out[4] = bytes_out[0] + bytes_out[1] + bytes_out[2] + bytes_out[3];
    return ZERO_OK;
}

int zero_comm_volume(double psi, int n_d, int stage, int ring, double* elements_out) {
    if (!elements_out || n_d < 1 || stage < 0 || stage > 3 || !(psi >= 0.0))
        return fail(ZERO_EINVAL, "zero_comm_volume: bad argument");
    // one reduce-scatter or all-gather of psi elements; a ring moves (n_d-1)/n_d of it
    const double phase = ring ? psi * (double)(n_d - 1) / (double)n_d : psi;
    const int phases = stage == 3 ? 3 : 2;   // ZeRO-3 gathers the parameters twice
    *elements_out = phases * phase;
    return ZERO_OK;
}

int zero_plan_round_robin(int n_tensors, int world_size, int64_t* order_out) {
    if (n_tensors < 0 || world_size < 1 || (n_tensors > 0 && !order_out))
        return fail(ZERO_EINVAL, "zero_plan_round_robin: bad argument");
    int k = 0;
    for (int g = 0; g < world_size; ++g)
        for (int i = g; i < n_tensors; i += world_size) order_out[k++] = i;
    return ZERO_OK;
}

int zero_shard_step(const void* const* grad_slices, int n_slices, int grad_dtype, const zero_shard* shards,
                    int n_shards, void* flat_param, int param_dtype, const zero_hyper* hyper, float loss_scale,
                    double extra_sumsq, int extra_overflow, void* workspace, size_t workspace_bytes,
                    zero_result* result, void* stream) {
    StepPlan sp;
    const int rc = plan_step(sp, grad_slices, n_slices, grad_dtype, shards, n_shards, flat_param, param_dtype, hyper,
                             loss_scale, extra_sumsq, extra_overflow, workspace, workspace_bytes, result);
    if (rc != ZERO_OK) return rc;
    return run_step(sp, static_cast<cudaStream_t>(stream));
}

int zero_shard_init(const zero_shard* shards, int n_shards, const void* flat_param, int param_dtype, void* stream) {
    if (!valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    int rc;
    if ((rc = pack_shards(a, shards, n_shards, 1)) != ZERO_OK) return rc;
    if (!any_elements(a)) return ZERO_OK;
    if (!flat_param || !aligned(flat_param, 2)) return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    a.flat_param = const_cast<void*>(flat_param);
    return launch_init(a, param_dtype, static_cast<cudaStream_t>(stream));
}

int zero_adam_scalar_table(const zero_hyper* hyper, int64_t t0, int64_t n, float* table_out) {
    if (!hyper || t0 < 1 || n < 0 || (n > 0 && !table_out)) return fail(ZERO_EINVAL, "zero_adam_scalar_table: bad argument");
    zero_hyper h = *hyper;
    for (int64_t i = 0; i < n; ++i) {
        h.step = t0 + i;
        const AdamScalars c = adam_scalars(h);
        table_out[2 * i] = c.ss;
        table_out[2 * i + 1] = c.rb2;
    }
    return ZERO_OK;
}

int zero_shard_step_chained(const void* const* grad_slices, int n_slices, int grad_dtype, const zero_shard* shards,
                            int n_shards, void* flat_param, int param_dtype, const zero_hyper* hyper,
                            const float* scalar_table, int64_t table_t0, int64_t n_table, zero_chain* chain,
                            double extra_sumsq, int extra_overflow, void* workspace, size_t workspace_bytes,
                            zero_result* result, void* stream) {
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    if (!hyper) return fail(ZERO_EINVAL, "hyper is NULL");
    if (!chain || !aligned(chain, 8)) return fail(ZERO_EINVAL, "chain is NULL or not 8-byte aligned");
    if (!scalar_table || !aligned(scalar_table, 4) || n_table < 1 || table_t0 < 1)
        return fail(ZERO_EINVAL, "scalar_table is NULL or misaligned, or n_table / table_t0 < 1");
    if (!result || !aligned(result, 8)) return fail(ZERO_EINVAL, "result is NULL or not 8-byte aligned");
    int rc;
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    if ((rc = pack_slices(a, grad_slices, n_slices)) != ZERO_OK) return rc;
    if ((rc = check_workspace(a, workspace, workspace_bytes)) != ZERO_OK) return rc;
    for (int i = 0; i < n_shards && shards; ++i)
        if (shards[i].numel > 0 && (shards[i].master_out == shards[i].master_in ||
                                    shards[i].m_out == shards[i].m_in || shards[i].v_out == shards[i].v_in))
            return fail(ZERO_EINVAL, "zero_shard_step_chained: a shard updates its state in place; give two sets");
    const bool fused = hyper->max_grad_norm <= 0.0f;
    if ((rc = pack_shards(a, shards, n_shards, fused ? 1 : 2)) != ZERO_OK) return rc;
    if (!fused && (rc = pack_shards(a, shards, n_shards, 3)) != ZERO_OK) return rc;
    if (any_elements(a) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    a.flat_param = flat_param;
    zero_hyper h1 = *hyper;
    h1.step = 1;
    a.sc = adam_scalars(h1);              // t-independent scalars; ss and rb2 come from the table
    a.max_norm = (double)hyper->max_grad_norm;
    a.extra_sumsq = extra_sumsq;
    a.extra_overflow = extra_overflow ? 1 : 0;
    a.result = result;
    a.chain = chain;
    a.sc_table = scalar_table;
    a.t0 = table_t0;
    a.n_table = n_table;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (fused) {
        // the fused pass derives k = fp32(1/S) from chain->loss_scale on the device
        const int vec = vec8_ok(a, 1) ? 8 : 1;
        number_tiles(a, vec, HEAD_GRADS);
        const int grid = grid_for(fused_fn(a, grad_dtype, param_dtype, vec), a.n_tiles,
                                  n_slices <= FEW_SLICES ? BPS_FUSED_FEW : BPS_FUSED_MANY);
        if ((rc = launch_fused(a, grad_dtype, param_dtype, vec, grid, s)) != ZERO_OK) return rc;
        if ((rc = launch_recover(a, param_dtype, s)) != ZERO_OK) return rc;
    } else {
        a.stats = reinterpret_cast<zero_stats*>(static_cast<char*>(workspace) + WS_STATS);
        a.accumulate = 0;
        int vec = vec8_ok(a, 2) ? 8 : 1;
        number_tiles(a, vec, HEAD_GRADS);
        if ((rc = launch_reduce(a, grad_dtype, vec, s)) != ZERO_OK) return rc;
        vec = vec8_ok(a, 3) ? 8 : 1;
        number_tiles(a, vec, HEAD_STATE);
        if ((rc = launch_apply(a, grad_dtype, param_dtype, vec, s)) != ZERO_OK) return rc;
    }
    return launch_chain_update(chain, result, s);
}

int zero_shard_reduce(const void* const* grad_slices, int n_slices, int grad_dtype, const zero_shard* shards,
                      int n_shards, int accumulate, zero_stats* stats, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (!valid_dtype(grad_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    if (!stats || !aligned(stats, 8)) return fail(ZERO_EINVAL, "stats is NULL or not 8-byte aligned");
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    int rc;
    if ((rc = pack_slices(a, grad_slices, n_slices)) != ZERO_OK) return rc;
    if ((rc = check_workspace(a, workspace, workspace_bytes)) != ZERO_OK) return rc;
    if ((rc = pack_shards(a, shards, n_shards, 2)) != ZERO_OK) return rc;
    a.stats = stats;
    a.accumulate = accumulate ? 1 : 0;
    const int vec = vec8_ok(a, 2) ? 8 : 1;
    number_tiles(a, vec, HEAD_GRADS);
    return launch_reduce(a, grad_dtype, vec, static_cast<cudaStream_t>(stream));
}

int zero_shard_apply(const zero_shard* shards, int n_shards, int grad_dtype, void* flat_param, int param_dtype,
                     const zero_hyper* hyper, float loss_scale, const zero_stats* stats, double extra_sumsq,
                     int extra_overflow, void* workspace, size_t workspace_bytes, zero_result* result,
                     void* stream) {
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    int rc;
    if ((rc = check_hyper(hyper, loss_scale)) != ZERO_OK) return rc;
    if (!stats || !aligned(stats, 8)) return fail(ZERO_EINVAL, "stats is NULL or not 8-byte aligned");
    if (!result || !aligned(result, 8)) return fail(ZERO_EINVAL, "result is NULL or not 8-byte aligned");
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    if ((rc = pack_shards(a, shards, n_shards, 3)) != ZERO_OK) return rc;
    if (any_elements(a) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    a.flat_param = flat_param;
    a.sc = adam_scalars(*hyper);
    a.loss_scale = (double)loss_scale;
    a.max_norm = (double)hyper->max_grad_norm;
    a.extra_sumsq = extra_sumsq;
    a.extra_overflow = extra_overflow ? 1 : 0;
    a.stats = const_cast<zero_stats*>(stats);
    a.result = result;
    if ((rc = check_workspace(a, workspace, workspace_bytes)) != ZERO_OK) return rc;
    const int vec = vec8_ok(a, 3) ? 8 : 1;
    number_tiles(a, vec, HEAD_STATE);
    return launch_apply(a, grad_dtype, param_dtype, vec, static_cast<cudaStream_t>(stream));
}

int zero_shard_apply_chained(const zero_shard* shards, int n_shards, int grad_dtype, void* flat_param,
                             int param_dtype, const zero_hyper* hyper, const float* scalar_table, int64_t table_t0,
                             int64_t n_table, zero_chain* chain, const zero_stats* stats, double extra_sumsq,
                             int extra_overflow, void* workspace, size_t workspace_bytes, zero_result* result,
                             void* stream) {
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    if (!hyper) return fail(ZERO_EINVAL, "hyper is NULL");
    if (!chain || !aligned(chain, 8)) return fail(ZERO_EINVAL, "chain is NULL or not 8-byte aligned");
    if (!scalar_table || !aligned(scalar_table, 4) || n_table < 1 || table_t0 < 1)
        return fail(ZERO_EINVAL, "scalar_table is NULL or misaligned, or n_table / table_t0 < 1");
    if (!stats || !aligned(stats, 8)) return fail(ZERO_EINVAL, "stats is NULL or not 8-byte aligned");
    if (!result || !aligned(result, 8)) return fail(ZERO_EINVAL, "result is NULL or not 8-byte aligned");
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    int rc;
    if ((rc = pack_shards(a, shards, n_shards, 3)) != ZERO_OK) return rc;
    if (any_elements(a) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    if ((rc = check_workspace(a, workspace, workspace_bytes)) != ZERO_OK) return rc;
    a.flat_param = flat_param;
    zero_hyper h1 = *hyper;
    h1.step = 1;
    a.sc = adam_scalars(h1);              // t-independent scalars; ss and rb2 come from the table
    a.max_norm = (double)hyper->max_grad_norm;
    a.extra_sumsq = extra_sumsq;
    a.extra_overflow = extra_overflow ? 1 : 0;
    a.stats = const_cast<zero_stats*>(stats);
    a.result = result;
    a.chain = chain;
    a.sc_table = scalar_table;
    a.t0 = table_t0;
    a.n_table = n_table;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int vec = vec8_ok(a, 3) ? 8 : 1;
    number_tiles(a, vec, HEAD_STATE);
    if ((rc = launch_apply(a, grad_dtype, param_dtype, vec, s)) != ZERO_OK) return rc;
    return launch_chain_update(chain, result, s);
}

// The step's scalars from the chain (t, S, the state set) when there is one,
// else from hyper->step and loss_scale; checks shared by the partial pass and
// the commit.
static int step_source(StepArgs& a, const zero_hyper* hyper, float loss_scale, const float* scalar_table,
                       int64_t table_t0, int64_t n_table, zero_chain* chain) {
    if (!hyper) return fail(ZERO_EINVAL, "hyper is NULL");
    if (chain) {
        if (!aligned(chain, 8)) return fail(ZERO_EINVAL, "chain is not 8-byte aligned");
        if (!scalar_table || !aligned(scalar_table, 4) || n_table < 1 || table_t0 < 1)
            return fail(ZERO_EINVAL, "scalar_table is NULL or misaligned, or n_table / table_t0 < 1");
        zero_hyper h1 = *hyper;
        h1.step = 1;
        a.sc = adam_scalars(h1);          // t-independent scalars; ss and rb2 come from the table
        a.chain = chain;
        a.sc_table = scalar_table;
        a.t0 = table_t0;
        a.n_table = n_table;
        return ZERO_OK;
    }
    int rc;
    if ((rc = check_hyper(hyper, loss_scale)) != ZERO_OK) return rc;
    a.sc = adam_scalars(*hyper);
    a.loss_scale = (double)loss_scale;
    a.k = (float)(1.0 / (double)loss_scale);
    return ZERO_OK;
}

int zero_shard_step_partial(const void* const* grad_slices, int n_slices, int grad_dtype, const zero_shard* shards,
                            int n_shards, void* flat_param, int param_dtype, const zero_hyper* hyper,
                            float loss_scale, const float* scalar_table, int64_t table_t0, int64_t n_table,
                            zero_chain* chain, int accumulate, zero_stats* stats, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    if (!stats || !aligned(stats, 8)) return fail(ZERO_EINVAL, "stats is NULL or not 8-byte aligned");
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    int rc;
    if ((rc = step_source(a, hyper, loss_scale, scalar_table, table_t0, n_table, chain)) != ZERO_OK) return rc;
    if (hyper->max_grad_norm > 0.0f)
        return fail(ZERO_EINVAL, "zero_shard_step_partial: clipping needs the global norm before any update; "
                                 "use zero_shard_reduce and zero_shard_apply");
    if (state_in_place(shards, n_shards))
        return fail(ZERO_EINVAL, "zero_shard_step_partial: a shard updates its state in place; give two sets");
    if ((rc = pack_slices(a, grad_slices, n_slices)) != ZERO_OK) return rc;
    if ((rc = check_workspace(a, workspace, workspace_bytes)) != ZERO_OK) return rc;
    if ((rc = pack_shards(a, shards, n_shards, 1)) != ZERO_OK) return rc;
    if (any_elements(a) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    a.flat_param = flat_param;
    a.stats = stats;
    a.accumulate = accumulate ? 1 : 0;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int vec = vec8_ok(a, 1) ? 8 : 1;
    number_tiles(a, vec, HEAD_GRADS);
    const void* f = fused_fn(a, grad_dtype, param_dtype, vec);
    const int bps = n_slices <= FEW_SLICES ? BPS_FUSED_FEW : BPS_FUSED_MANY;
    const size_t smem = smem_capping(f, bps);
    const int grid = grid_for_smem(f, a.n_tiles, smem, bps);
    return launch_fused_early(a, grad_dtype, param_dtype, vec, grid, smem, s);
}

int zero_shard_step_commit(const zero_shard* shards, int n_shards, void* flat_param, int param_dtype,
                           float loss_scale, int64_t table_t0, int64_t n_table, zero_chain* chain,
                           const zero_stats* stats, double extra_sumsq, int extra_overflow, zero_result* result,
                           void* stream) {
    if (!valid_dtype(param_dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    if (!stats || !aligned(stats, 8)) return fail(ZERO_EINVAL, "stats is NULL or not 8-byte aligned");
    if (!result || !aligned(result, 8)) return fail(ZERO_EINVAL, "result is NULL or not 8-byte aligned");
    if (chain && !aligned(chain, 8)) return fail(ZERO_EINVAL, "chain is not 8-byte aligned");
    if (chain && (n_table < 1 || table_t0 < 1)) return fail(ZERO_EINVAL, "n_table / table_t0 < 1");
    if (!chain && (!(loss_scale > 0.0f) || !std::isfinite(loss_scale)))
        return fail(ZERO_EINVAL, "loss_scale must be finite and > 0");
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    int rc;
    if ((rc = pack_shards(a, shards, n_shards, 1)) != ZERO_OK) return rc;
    if (any_elements(a) && (!flat_param || !aligned(flat_param, 2)))
        return fail(ZERO_EINVAL, "flat_param is NULL or not 2-byte aligned");
    a.flat_param = flat_param;
    a.stats = const_cast<zero_stats*>(stats);
    a.extra_sumsq = extra_sumsq;
    a.extra_overflow = extra_overflow ? 1 : 0;
    a.result = result;
    a.chain = chain;
    a.loss_scale = (double)loss_scale;
    a.k = chain ? 0.0f : (float)(1.0 / (double)loss_scale);
    // a chained step whose t lies outside the partial passes' scalar table was
    // skipped by them: the commit reports it (ZERO_ELIMIT) rather than apply it
    a.t0 = table_t0;
    a.n_table = n_table;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = launch_commit(a, s)) != ZERO_OK) return rc;
    if ((rc = launch_recover(a, param_dtype, s)) != ZERO_OK) return rc;
    return chain ? launch_chain_update(chain, result, s) : ZERO_OK;
}

// The register-staged gather's arguments for n pieces laid end to end in out
// (pointers and lengths already validated); returns the vector width.
static int gather_args(const void* const* src, const int64_t* len, int n, void* out, GatherArgs& g) {
    std::memset(&g, 0, sizeof g);
    g.n = n;
    g.out = out;
    int64_t off = 0;
    bool v8 = aligned(out, 16);
    for (int p = 0; p < n; ++p) {
        g.src[p] = src[p];
        g.len[p] = len[p];
        g.dst_off[p] = off;
        v8 = v8 && aligned(src[p], 16) && (off % 8 == 0);
        off += len[p];
    }
    const int vec = v8 ? 8 : 1;
    const int64_t tile = (int64_t)TILE_THREADS * vec * (vec == 8 ? GATHER_UNROLL : 2);
    int64_t t = 0;
    for (int p = 0; p < n; ++p) {
        g.tile_begin[p] = t;
        t += (g.len[p] + tile - 1) / tile;
    }
    g.tile_begin[n] = t;
    return vec;
}

// Checks shared by the gathers; returns ZERO_OK and the total length in *total.
static int check_pieces(const char* who, const void* const* src, const int64_t* len, int n, int dtype, void* out,
                        int64_t* total) {
    std::string w(who);
    if (!valid_dtype(dtype)) return fail(ZERO_EINVAL, (w + ": unknown dtype").c_str());
    if (n < 1) return fail(ZERO_EINVAL, (w + ": no segments").c_str());
    if (n > ZERO_MAX_SLICES) return fail(ZERO_ELIMIT, (w + ": more than ZERO_MAX_SLICES segments").c_str());
    if (!src || !len || !out) return fail(ZERO_EINVAL, (w + ": NULL pointer").c_str());
    if (!aligned(out, 2)) return fail(ZERO_EALIGN, (w + ": layer_out not 2-byte aligned").c_str());
    int64_t off = 0;
    for (int p = 0; p < n; ++p) {
        if (len[p] < 0) return fail(ZERO_EINVAL, (w + ": negative segment length").c_str());
        if (len[p] > 0 && !src[p]) return fail(ZERO_EINVAL, (w + ": a segment pointer is NULL").c_str());
        if (!aligned(src[p], 2)) return fail(ZERO_EALIGN, (w + ": segment pointer not 2-byte aligned").c_str());
        off += len[p];
    }
    *total = off;
    return ZERO_OK;
}

static int gather_segments(const void* const* src, const int64_t* len, int n, int dtype, void* out, void* stream) {
    int64_t total = 0;
    int rc = check_pieces("zero3_gather", src, len, n, dtype, out, &total);
    if (rc != ZERO_OK || total == 0) return rc;
    GatherArgs g;
    const int vec = gather_args(src, len, n, out, g);
    return launch_gather(g, vec, static_cast<cudaStream_t>(stream));
}

int zero3_gather_layer(const void* const* part_ptrs, int world_size, int64_t unit_numel, int dtype, void* layer_out,
                       void* stream) {
    if (!valid_dtype(dtype)) return fail(ZERO_EINVAL, "unknown dtype");
    if (world_size < 1) return fail(ZERO_EINVAL, "world_size < 1");
    if (world_size > ZERO_MAX_SLICES) return fail(ZERO_ELIMIT, "world_size above ZERO_MAX_SLICES");
    if (unit_numel < 0 || unit_numel % world_size != 0)
        return fail(ZERO_EINVAL, "unit_numel must be >= 0 and divisible by world_size");
    if (unit_numel == 0) return ZERO_OK;
    if (!part_ptrs || !layer_out) return fail(ZERO_EINVAL, "NULL pointer");
    int64_t len[ZERO_MAX_SLICES];
    for (int r = 0; r < world_size; ++r) len[r] = unit_numel / world_size;
    return gather_segments(part_ptrs, len, world_size, dtype, layer_out, stream);
}

int zero3_gather_segments(const void* const* segment_ptrs, const int64_t* segment_numels, int n_segments,
                          int dtype, void* layer_out, void* stream) {
    return gather_segments(segment_ptrs, segment_numels, n_segments, dtype, layer_out, stream);
}

int zero3_gather_bulk(const void* const* segment_ptrs, const int64_t* segment_numels, int n_segments, int dtype,
                      void* layer_out, int n_ctas, int32_t* status, void* stream) {
    if (!status) return fail(ZERO_EINVAL, "zero3_gather_bulk: NULL status");
    if (n_ctas < 0) return fail(ZERO_EINVAL, "zero3_gather_bulk: negative n_ctas");
    if (!aligned(status, 4)) return fail(ZERO_EINVAL, "zero3_gather_bulk: status not 4-byte aligned");
    int64_t total = 0;
    int rc = check_pieces("zero3_gather_bulk", segment_ptrs, segment_numels, n_segments, dtype, layer_out, &total);
    if (rc != ZERO_OK || total == 0) return rc;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "zero3_gather_bulk: device query");
    int ctas = n_ctas == 0 ? sms : n_ctas;

    BulkGatherArgs b;
    std::memset(&b, 0, sizeof b);
    b.n = n_segments;
    b.out = static_cast<uint8_t*>(layer_out);
    b.status = status;
    bool congruent = true;
    int64_t off = 0;
    for (int p = 0; p < n_segments; ++p) {
        const int64_t L = segment_numels[p];
        const uintptr_t sa = reinterpret_cast<uintptr_t>(segment_ptrs[p]);
        const uintptr_t da = reinterpret_cast<uintptr_t>(layer_out) + 2 * (uintptr_t)off;
        if (L > 0 && (sa - da) % 16 != 0) congruent = false;
        b.src[p] = static_cast<const uint8_t*>(segment_ptrs[p]);
        b.bytes[p] = 2 * L;
        b.dst_off[p] = 2 * off;
        const int64_t h = (int64_t)((16 - sa % 16) % 16);
        b.head[p] = h < b.bytes[p] ? h : b.bytes[p];
        b.mid[p] = (b.bytes[p] - b.head[p]) / 16 * 16;
        off += L;
    }
    if (!congruent) {
        // no bulk copies possible: the register-staged gather on at most `ctas` blocks
        GatherArgs g;
        const int vec = gather_args(segment_ptrs, segment_numels, n_segments, layer_out, g);
        return launch_gather(g, vec, static_cast<cudaStream_t>(stream), ctas);
    }
    // A CTA with an SM of its own gets the deeper pipeline; many CTAs share the
    // bandwidth with smaller ones.
    const bool few = 2 * (int64_t)ctas <= sms;
    b.chunk = few ? 32768 : 16384;
    b.stages = few ? 6 : 4;
    int64_t c = 0;
    for (int p = 0; p < n_segments; ++p) {
        b.chunk_begin[p] = c;
        c += (b.mid[p] + b.chunk - 1) / b.chunk;
    }
    b.chunk_begin[n_segments] = c;
    if (ctas > c) ctas = (int)(c > 0 ? c : 1);
    if (ctas > MAX_BLOCKS) ctas = MAX_BLOCKS;
    b.spin_limit = spin_limit();
    b.drain_limit = SPIN_LIMIT;
    return launch_gather_bulk(b, ctas, static_cast<cudaStream_t>(stream));
}

int zero3_reduce_bucket(const void* const* bucket_ptrs, int world_size, int owner, int64_t unit_numel, int grad_dtype,
                        void* grad_part, int accumulate, zero_stats* stats, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (world_size < 1 || owner < 0 || owner >= world_size) return fail(ZERO_EINVAL, "bad world_size or owner");
    if (unit_numel < 0 || unit_numel % world_size != 0)
        return fail(ZERO_EINVAL, "unit_numel must be >= 0 and divisible by world_size");
    zero_shard s;
    std::memset(&s, 0, sizeof s);
    s.numel = unit_numel / world_size;
    s.grad_offset = (int64_t)owner * s.numel;
    s.grad_shard = grad_part;
    return zero_shard_reduce(bucket_ptrs, world_size, grad_dtype, &s, 1, accumulate, stats, workspace,
                             workspace_bytes, stream);
}

}  // extern "C"
