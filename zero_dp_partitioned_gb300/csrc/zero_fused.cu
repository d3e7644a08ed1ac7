// zero_fused.cu -- instantiations and launchers of the fused single pass (K1a)
// and of the parameter restore that follows it (K1r).
#include "zero_internal.h"

namespace zdp {

template <int G, int P, int V, bool C, bool W>
static const void* fused_ptr(int ns) {
    if (ns == 4) return (const void*)k_step_fused<G, P, V, 4, C, W>;
    return ns == NS_FEW ? (const void*)k_step_fused<G, P, V, NS_FEW, C, W> : (const void*)k_step_fused<G, P, V, 0, C, W>;
}

template <int G, int P, bool C>
static const void* fused_ptr_v(int vec, int ns, bool wide) {
    if (vec != 8) return fused_ptr<G, P, 1, C, false>(ns);
    return wide ? fused_ptr<G, P, 8, C, true>(ns) : fused_ptr<G, P, 8, C, false>(ns);
}

template <bool C>
static const void* fused_pick(int gdt, int pdt, int vec, int ns, bool wide) {
    if (gdt == ZERO_BF16) return pdt == ZERO_BF16 ? fused_ptr_v<ZERO_BF16, ZERO_BF16, C>(vec, ns, wide)
                                                  : fused_ptr_v<ZERO_BF16, ZERO_F16, C>(vec, ns, wide);
    return pdt == ZERO_BF16 ? fused_ptr_v<ZERO_F16, ZERO_BF16, C>(vec, ns, wide) : fused_ptr_v<ZERO_F16, ZERO_F16, C>(vec, ns, wide);
}

const void* fused_kernel(int gdt, int pdt, int vec, int ns, bool wide) { return fused_pick<false>(gdt, pdt, vec, ns, wide); }

// Chained steps: the same passes, instantiated with the device-side
// bookkeeping (t, S and the state set read from the chain).
const void* fused_kernel_chain(int gdt, int pdt, int vec, int ns, bool wide) {
    return fused_pick<true>(gdt, pdt, vec, ns, wide);
}

// The fused pass's kernel for these arguments: chained or not, and with
// 256-bit state accesses when every shard's state arrays allow them.
const void* fused_fn(const StepArgs& a, int gdt, int pdt, int vec) {
    const int ns = fused_ns(a.n_slices);
    const bool wide = vec == 8 && fused_state_wide(a);
    return a.chain ? fused_kernel_chain(gdt, pdt, vec, ns, wide) : fused_kernel(gdt, pdt, vec, ns, wide);
}

int launch_fused(const StepArgs& a, int gdt, int pdt, int vec, int grid, cudaStream_t s) {
    const void* f = fused_fn(a, gdt, pdt, vec);
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, 0, s), "fused step launch");
}

int launch_recover(const StepArgs& a, int pdt, cudaStream_t s) {
    const void* f = pdt == ZERO_BF16 ? (const void*)k_recover<ZERO_BF16> : (const void*)k_recover<ZERO_F16>;
    int64_t n = 0;
    for (int i = 0; i < a.n_shards; ++i) n = a.shards[i].numel > n ? a.shards[i].numel : n;
    const int grid = grid_for(f, (n + TILE_THREADS - 1) / TILE_THREADS, BPS_RECOVER);
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, 0, s), "recover launch");
}

// ---------------------------------------------------------------- K0: state initialisation
// Every shard's *_in set: master = fp32(param) (the exact widening of the
// 16-bit value at the shard's parameter offset), m = v = 0.
template <int PDT>
__global__ void __launch_bounds__(TILE_THREADS) k_init(const __grid_constant__ StepArgs a) {
    const uint16_t* P = static_cast<const uint16_t*>(a.flat_param);
    for (int si = 0; si < a.n_shards; ++si) {
        const ShardDev& d = a.shards[si];
        float* M = const_cast<float*>(d.mi);
        float* Mm = const_cast<float*>(d.mmi);
        float* V = const_cast<float*>(d.vi);
        for (int64_t i = (int64_t)blockIdx.x * TILE_THREADS + threadIdx.x; i < d.numel;
             i += (int64_t)gridDim.x * TILE_THREADS) {
            M[i] = Half16<PDT>::widen(P[d.param_off + i]);
            Mm[i] = 0.0f;
            V[i] = 0.0f;
        }
    }
}

int launch_init(const StepArgs& a, int pdt, cudaStream_t s) {
    const void* f = pdt == ZERO_BF16 ? (const void*)k_init<ZERO_BF16> : (const void*)k_init<ZERO_F16>;
    int64_t n = 0;
    for (int i = 0; i < a.n_shards; ++i) n = a.shards[i].numel > n ? a.shards[i].numel : n;
    const int grid = grid_for(f, (n + TILE_THREADS - 1) / TILE_THREADS, 0);
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, 0, s), "init launch");
}

// ---------------------------------------------------------------- K1d: the decision after partial fused passes
// A step whose shards were updated by partial fused passes (each adding its
// statistics to *a.stats) is decided here, from every pass's statistics and
// the other ranks' share: skip on overflow (k_recover, launched next,
// restores the parameters), or commit (the caller or the chain keeps the
// written state set).  One thread.
__global__ void k_commit(const __grid_constant__ StepArgs a) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const zero_stats st = *a.stats;
    const double S = step_S(a);
    zero_result r;
    r.overflow = (st.overflow | a.extra_overflow) ? 1 : 0;
    r.status = (a.chain && step_bad(a)) ? ZERO_ELIMIT : 0;
    r.applied = (r.overflow || r.status) ? 0 : 1;
    r.path = 3;
    r.sumsq = st.sumsq + a.extra_sumsq;
    r.grad_norm = sqrt(r.sumsq) / S;
    r.clip_coef = 1.0;
    r.grad_mult = a.chain ? (float)(1.0 / S) : a.k;
    r.reserved = 0.0f;
    *a.result = r;
}

int launch_commit(const StepArgs& a, cudaStream_t s) {
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cuda_fail(cudaLaunchKernel((const void*)k_commit, dim3(1), dim3(32), args, 0, s), "commit launch");
}

int launch_fused_early(const StepArgs& a, int gdt, int pdt, int vec, int grid, size_t smem, cudaStream_t s) {
    const void* f = fused_fn(a, gdt, pdt, vec);
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cuda_fail(launch_after_previous(f, grid, TILE_THREADS, args, smem, s), "partial fused pass launch");
}

// ---------------------------------------------------------------- chained steps: the bookkeeping
// After a chained step's kernels: applied -> next t, the other state set;
// overflow -> half the loss scale, unless that would take it below the
// floor (then S stays and the step counts as failed: a chain stuck at its
// floor must not slide towards an S whose reciprocal overflows fp32);
// another failure -> counted only.
__global__ void k_chain_update(zero_chain* chain, const zero_result* result) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const zero_result r = *result;
    if (r.applied) {
        chain->step += 1;
        chain->cur ^= 1;
        chain->applied += 1;
    } else if (r.overflow && r.status == 0) {
        const double floor = chain->min_loss_scale > 0.0 ? chain->min_loss_scale : 0x1p-126;
        const double half = chain->loss_scale * 0.5;
        if (half >= floor) {
            chain->loss_scale = half;
            chain->skipped += 1;
        } else {
            chain->failed += 1;
        }
    } else {
        chain->failed += 1;
    }
}

int launch_chain_update(zero_chain* chain, const zero_result* result, cudaStream_t s) {
    k_chain_update<<<1, 32, 0, s>>>(chain, result);
    return cuda_fail(cudaGetLastError(), "chain update launch");
}

}  // namespace zdp
