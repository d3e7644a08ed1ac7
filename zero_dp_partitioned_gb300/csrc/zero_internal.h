// zero_internal.h -- host-side helpers shared by the library's translation
// units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <string>

#include "zero_kernels.cuh"

namespace zdp {

void set_error(const std::string& msg);
int cuda_fail(cudaError_t e, const char* what);

// Resident blocks per SM each pass is launched with (0 = as many as fit).
// Measured on GB300 over the full workloads: passes that write a third or
// more of their bytes (the fused pass with few slices, the apply pass) reach
// more of the HBM bandwidth with fewer concurrent warps -- 2 blocks of 256
// threads per SM: 10.8 ms vs 11.7 ms for the 8-slice fused GPT-2 step at 4
// blocks (with an earlier 64-register loop; the loop now used needs up to 128
// registers, so 2 blocks is also all that fits), 8.6 ms vs 9.5 ms at 3
// blocks for the Llama apply pass -- while read-dominated passes want every
// block they can get (the 64-slice
// fused pass: 2.63 ms at 4 blocks, 3.11 ms at 2; the reduce pass is best at
// 6: 2.98 ms, against 3.13 at 4 and 3.11 at the 8 its 32 registers allow);
// the gather (a copy) peaks at 4.
constexpr int BPS_FUSED_FEW = 2;        // fused pass with at most FEW_SLICES slices
constexpr int FEW_SLICES = 12;
constexpr int BPS_FUSED_MANY = 0;
constexpr int BPS_APPLY = 2;
constexpr int BPS_REDUCE = 6;
constexpr int BPS_GATHER = 4;
constexpr int BPS_RECOVER = 0;

// Blocks of 256 threads to launch for `func` over n_tiles tiles: resident
// blocks per SM (at most max_per_sm when that is > 0) x SM count, capped by
// the tile count and MAX_BLOCKS.
int grid_for(const void* func, int64_t n_tiles, int max_per_sm = 0);
int grid_for_smem(const void* func, int64_t n_tiles, size_t dynamic_smem, int max_per_sm = 0);

// Dynamic shared memory for `func` (256-thread blocks) that leaves room for
// at most `blocks` resident blocks per SM, the kernel's limit raised to it;
// 0 when its registers already allow no more or the device refuses.  A grid
// of `blocks` per SM launched early, while the previous pass still runs,
// would otherwise let the next pass's blocks take the free slots first and
// settle three to an SM on some SMs and one on others.
size_t smem_capping(const void* func, int blocks);

// Launch of a kernel that starts with pdl_wait() (the gathers and the
// reduce), allowed to begin while the previous kernel of the stream finishes.
cudaError_t launch_after_previous(const void* f, int grid, int block, void** args, size_t smem, cudaStream_t s);

// Launchers; each validates nothing (the entry points did) and returns
// ZERO_OK or ZERO_ECUDA.  vec is 8 or 1.
const void* fused_fn(const StepArgs& a, int gdt, int pdt, int vec);
int launch_fused(const StepArgs& a, int gdt, int pdt, int vec, int grid, cudaStream_t s);
int launch_recover(const StepArgs& a, int pdt, cudaStream_t s);
int launch_init(const StepArgs& a, int pdt, cudaStream_t s);
int launch_chain_update(zero_chain* chain, const zero_result* result, cudaStream_t s);
int launch_commit(const StepArgs& a, cudaStream_t s);
// The fused pass launched early (programmatic stream serialisation): for the
// partial passes, which run back to back, one per ZeRO-3 unit.
int launch_fused_early(const StepArgs& a, int gdt, int pdt, int vec, int grid, size_t smem, cudaStream_t s);
// early: launched with programmatic stream serialisation (back-to-back
// bucket reduces); plain otherwise.
int launch_reduce(const StepArgs& a, int gdt, int vec, cudaStream_t s, bool early = true);
int launch_apply(const StepArgs& a, int gdt, int pdt, int vec, cudaStream_t s);
int launch_gather(const GatherArgs& a, int vec, cudaStream_t s, int max_grid = 0);

// The TMA-moved gather (zero_gather_bulk.cu).  Offsets and sizes in bytes;
// piece p is head[p] unaligned bytes, mid[p] bytes moved in chunks (a
// multiple of 16, starting 16-byte aligned at both ends), then the rest.
struct BulkGatherArgs {
    const uint8_t* src[ZERO_MAX_SLICES];
    int64_t bytes[ZERO_MAX_SLICES];
    int64_t dst_off[ZERO_MAX_SLICES];
    int64_t head[ZERO_MAX_SLICES];
    int64_t mid[ZERO_MAX_SLICES];
    int64_t chunk_begin[ZERO_MAX_SLICES + 1];   // first chunk of each piece's middle; [n] = chunk count
    uint8_t* out;
    int32_t* status;                            // bit 0 set by a CTA whose wait ran out
    int n, chunk, stages;
    unsigned spin_limit, drain_limit;
};
size_t gather_bulk_smem(int chunk, int stages);
int launch_gather_bulk(const BulkGatherArgs& a, int grid, cudaStream_t s);

// Argument checks and kernel-argument packing shared by the entry points
// (zero_abi.cu); each check sets the thread's error message and returns its
// code, and none touches the device.
bool aligned(const void* p, size_t a);
bool valid_dtype(int d);
int fail(int code, const char* msg);
AdamScalars adam_scalars(const zero_hyper& h);
int check_hyper(const zero_hyper* h, float loss_scale);
// need: 1 = fused (state in/out), 2 = reduce (grad_shard out), 3 = apply
// (grad_shard in, state in/out)
int pack_shards(StepArgs& a, const zero_shard* shards, int n_shards, int need);
int pack_slices(StepArgs& a, const void* const* slices, int n_slices);
int check_workspace(StepArgs& a, void* ws, size_t ws_bytes);
bool vec8_ok(const StepArgs& a, int need);
bool state_wide(const StepArgs& a);          // the apply pass may take 256-bit state accesses
bool fused_state_wide(const StepArgs& a);    // the fused pass may take 256-bit state accesses
bool any_elements(const StepArgs& a);
bool state_in_place(const zero_shard* shards, int n_shards);
// Which stream a pass's vector loop aligns to 128 bytes: its dominant one.
enum HeadKind { HEAD_NONE = 0, HEAD_GRADS = 1, HEAD_STATE = 2 };
void number_tiles(StepArgs& a, int vec, int kind = HEAD_NONE);

// zero_shard_step in two phases: plan_step makes every argument check and
// packs the kernel arguments without touching the device (an argument error
// therefore enqueues nothing); run_step launches the planned kernels.
struct StepPlan {
    StepArgs a;
    bool fused;          // one fused pass (+ parameter restore check), else reduce + apply
    int gdt, pdt;
};
int plan_step(StepPlan& sp, const void* const* grad_slices, int n_slices, int grad_dtype, const zero_shard* shards,
              int n_shards, void* flat_param, int param_dtype, const zero_hyper* hyper, float loss_scale,
              double extra_sumsq, int extra_overflow, void* workspace, size_t workspace_bytes, zero_result* result);
int run_step(StepPlan& sp, cudaStream_t s);

// Kernel addresses, for the occupancy query.
const void* fused_kernel(int gdt, int pdt, int vec, int ns, bool wide = false);
const void* fused_kernel_chain(int gdt, int pdt, int vec, int ns, bool wide = false);
const void* reduce_kernel(int gdt, int vec, int ns);
const void* apply_kernel(int gdt, int pdt, int vec, bool wide = false);

// The slice-count specialisation of the reduce pass for n slices (0 = the
// generic loop).
inline int ns_variant(int n) { return (n >= 1 && n <= 4) ? n : (n == 8 ? 8 : 0); }

// The fused pass's slice loop: unrolled for exactly 4 slices (the ZeRO-3
// and rank-local steps at N_d = 4: a unit's partial pass took 0.3130 ms
// against 0.3200 ms with the generic loop), else generic, at 2 blocks per SM
// for at most FEW_SLICES slices (NS_FEW) or at 4 for more (0).
constexpr int NS_FEW = -1;
inline int fused_ns(int n) { return n == 4 ? 4 : (n <= FEW_SLICES ? NS_FEW : 0); }

}  // namespace zdp
