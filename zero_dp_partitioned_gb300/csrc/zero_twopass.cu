// zero_twopass.cu -- instantiations and launchers of the reduce + statistics
// pass (K1b, also the ZeRO-3 bucket reduce K4), the apply pass (K1c) and the
// ZeRO-3 layer gather (K3).
#include "zero_internal.h"

namespace zdp {

template <int G, int V>
static const void* reduce_ptr(int ns) {
    if (V == 1) return (const void*)k_reduce<G, 1, 0>;
    switch (ns) {
    case 1: return (const void*)k_reduce<G, V, 1>;
    case 2: return (const void*)k_reduce<G, V, 2>;
    case 3: return (const void*)k_reduce<G, V, 3>;
    case 4: return (const void*)k_reduce<G, V, 4>;
    case 8: return (const void*)k_reduce<G, V, 8>;
    default: return (const void*)k_reduce<G, V, 0>;
    }
}

const void* reduce_kernel(int gdt, int vec, int ns) {
    if (gdt == ZERO_BF16) return vec == 8 ? reduce_ptr<ZERO_BF16, 8>(ns) : reduce_ptr<ZERO_BF16, 1>(ns);
    return vec == 8 ? reduce_ptr<ZERO_F16, 8>(ns) : reduce_ptr<ZERO_F16, 1>(ns);
}

template <int G, int P>
static const void* apply_ptr(int vec, bool wide) {
    if (vec != 8) return (const void*)k_apply<G, P, 1>;
    return wide ? (const void*)k_apply<G, P, 8, true> : (const void*)k_apply<G, P, 8>;
}

const void* apply_kernel(int gdt, int pdt, int vec, bool wide) {
    if (gdt == ZERO_BF16)
        return pdt == ZERO_BF16 ? apply_ptr<ZERO_BF16, ZERO_BF16>(vec, wide) : apply_ptr<ZERO_BF16, ZERO_F16>(vec, wide);
    return pdt == ZERO_BF16 ? apply_ptr<ZERO_F16, ZERO_BF16>(vec, wide) : apply_ptr<ZERO_F16, ZERO_F16>(vec, wide);
}

int launch_reduce(const StepArgs& a, int gdt, int vec, cudaStream_t s, bool early) {
    const void* f = reduce_kernel(gdt, vec, ns_variant(a.n_slices));
    const int grid = grid_for(f, a.n_tiles, BPS_REDUCE);
    void* args[] = {const_cast<StepArgs*>(&a)};
    if (!early) return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, 0, s), "reduce launch");
    return cuda_fail(launch_after_previous(f, grid, TILE_THREADS, args, 0, s), "reduce launch");
}

int launch_apply(const StepArgs& a, int gdt, int pdt, int vec, cudaStream_t s) {
    const void* f = apply_kernel(gdt, pdt, vec, vec == 8 && state_wide(a));
    const int grid = grid_for(f, a.n_tiles, BPS_APPLY);
    void* args[] = {const_cast<StepArgs*>(&a)};
    return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, 0, s), "apply launch");
}

int launch_gather(const GatherArgs& a, int vec, cudaStream_t s, int max_grid) {
    const void* f = vec == 8 ? (const void*)k_gather<8> : (const void*)k_gather<1>;
    int grid = grid_for(f, a.tile_begin[a.n], BPS_GATHER);
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    void* args[] = {const_cast<GatherArgs*>(&a)};
    return cuda_fail(launch_after_previous(f, grid, TILE_THREADS, args, 0, s), "gather launch");
}

}  // namespace zdp

namespace zdp {

// A launch allowed to begin while the previous kernel of the stream finishes
// (programmatic stream serialisation); the kernel waits for that kernel's
// completion before its first memory access.
cudaError_t launch_after_previous(const void* f, int grid, int block, void** args, size_t smem, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace zdp
