// zero_stream.cu -- instantiations and launcher of the shared-memory-staged
// (bulk asynchronous copy) fused and apply passes.
#include <mutex>
#include <unordered_map>

#include "zero_internal.h"
#include "zero_stream.cuh"

namespace zdp {

template <int G, int P>
static const void* stream_ptr(bool fused) {
    return fused ? (const void*)k_stream<G, P, true> : (const void*)k_stream<G, P, false>;
}

static const void* stream_kernel(int gdt, int pdt, bool fused) {
    if (gdt == ZERO_BF16) return pdt == ZERO_BF16 ? stream_ptr<ZERO_BF16, ZERO_BF16>(fused)
                                                  : stream_ptr<ZERO_BF16, ZERO_F16>(fused);
    return pdt == ZERO_BF16 ? stream_ptr<ZERO_F16, ZERO_BF16>(fused) : stream_ptr<ZERO_F16, ZERO_F16>(fused);
}

// Stages that fit 113 KB per block, so that two blocks share an SM's 228 KB
// (each block also reserves 1 KB).
int stream_stages(int n_grad_arrays) {
    const StreamLayout L1 = stream_layout(n_grad_arrays, 1);
    const size_t budget = 113 * 1024 - 64 - 2 * (size_t)L1.out_bytes;
    int s = (int)(budget / L1.in_bytes);
    return s < 2 ? 2 : (s > 8 ? 8 : s);
}

int launch_stream(const StreamArgs& sa, int gdt, int pdt, bool fused, cudaStream_t s) {
    const void* f = stream_kernel(gdt, pdt, fused);
    const StreamLayout L = stream_layout(fused ? sa.a.n_slices : 1, sa.stages);
    const size_t smem = stream_smem_bytes(L);
    static std::mutex mu;
    static std::unordered_map<const void*, size_t> configured[16];
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> g(mu);
        size_t& have = configured[dev & 15][f];
        if (have < smem) {
            int rc = cuda_fail(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                               "raising the shared-memory limit of the staged kernel");
            if (rc != ZERO_OK) return rc;
            have = smem;
        }
    }
    const int grid = grid_for_smem(f, sa.a.n_tiles, smem, 0);
    void* args[] = {const_cast<StreamArgs*>(&sa)};
    return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, smem, s), "staged kernel launch");
}

}  // namespace zdp
