// zero_internal.h -- host-side helpers shared by the library's translation
// units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <string>

#include "zero_kernels.cuh"

namespace zdp {

void set_error(const std::string& msg);
int cuda_fail(cudaError_t e, const char* what);

// Blocks of 256 threads to launch for `func` over n_tiles tiles: resident
// blocks per SM x SM count, capped by the tile count and MAX_BLOCKS.
int grid_for(const void* func, int64_t n_tiles);

// Launchers; each validates nothing (the entry points did) and returns
// ZERO_OK or ZERO_ECUDA.  vec is 8 or 1.
int launch_fused(const StepArgs& a, int gdt, int pdt, int vec, int grid, cudaStream_t s);
int launch_recover(const StepArgs& a, int pdt, cudaStream_t s);
int launch_reduce(const StepArgs& a, int gdt, int vec, cudaStream_t s);
int launch_apply(const StepArgs& a, int gdt, int pdt, int vec, cudaStream_t s);
int launch_gather(const GatherArgs& a, int vec, cudaStream_t s);

// Kernel addresses, for the occupancy query.
const void* fused_kernel(int gdt, int pdt, int vec, int ns);
const void* reduce_kernel(int gdt, int vec, int ns);
const void* apply_kernel(int gdt, int pdt, int vec);

// The slice-count specialisation used for n slices (0 = the generic loop).
inline int ns_variant(int n) { return (n >= 1 && n <= 4) ? n : (n == 8 ? 8 : 0); }

}  // namespace zdp
