// zero_ws.cu -- the fused single pass with a producer warp feeding TMA-staged
// chunks to consumer warps.
//
// An alternative to the register-staged fused pass, selected by
// ZERO_GB300_PATH=ws.  Moving the pass's traffic mix by bulk asynchronous
// copies reached more of the HBM bandwidth than a 64-register pass could
// (6.8-7.1 TB/s against 6.7), and this pass measured 9.62-9.71 ms on the
// GPT-2 step against 10.01 ms for that register pass; the register pass that
// now keeps every load of a vector in flight (up to 128 registers) takes
// 9.50 ms, so this one is opt-in.  The staged pass with a block-wide cycle
// per chunk loses the copies' advantage to the cycle.  Here the roles are
// split (two blocks of 8 warps per SM):
//   warp 0, lane 0 (producer): for each chunk of this block, waits until the
//     stage it needs is free, then issues the bulk loads of the chunk's
//     gradient slices and fp32 state into it (one full mbarrier per stage,
//     completed by the copies' byte count);
//   warps 1-7 (consumers, WS_VEC elements per lane, so a chunk is 7 x 32 x WS_VEC):
//     wait for the chunk's stage, reduce the slices, update, store the state
//     and the 16-bit parameters straight to global memory, and release the
//     stage (one empty mbarrier per stage, one arrival per consumer warp).
// No block-wide barrier inside the loop: each consumer warp runs as far ahead
// as the loaded stages let it, and the producer keeps every free stage busy.
//
// Chunks are numbered shard after shard.  A shard's first d.head elements
// (fewer than 64) are done one by one, so that its chunks start where the
// gradient slices sit on a 128-byte boundary (a copy that starts mid-line
// fetches one line more); a chunk's bulk part is its length rounded down to
// 8 elements, and a shard's last (fewer than 8) elements are loaded and
// stored with plain accesses.  Every wait is bounded; a wait that
// runs out marks the block's flags and the step is reported as not applied.
// Before the block finishes, the producer waits (bounded again) for the last
// loads it issued, whether or not a consumer took them.
#include <mutex>
#include <unordered_map>

#include "zero_internal.h"
#include "zero_stream.cuh"

namespace zdp {

constexpr int WS_CONSUMER_WARPS = 7;
constexpr int WS_VEC = 8;                                 // elements per consumer lane and chunk
constexpr int WS_CHUNK = WS_CONSUMER_WARPS * 32 * WS_VEC;
constexpr int WS_MAX_STAGES = 8;
constexpr int WS_HEADER = 128;                           // 8 full + 8 empty mbarriers
// Two blocks per SM: 14 consumer warps with 8 elements each.  Measured on the
// GPT-2 step (N_d = 8): 9.83 ms, against 9.89 / 9.92 ms with 4 elements at 2 / 3
// blocks, 10.28 ms with 8 elements at one block (4 stages), 12.3 ms with 4
// elements at one block; the 64-register pass of the time took 10.01 ms.
constexpr int WS_BLOCKS_PER_SM = 2;

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Stage bytes for ng 16-bit arrays (the slices, or the reduced gradient) and
// the three fp32 state arrays.
__host__ __device__ inline uint32_t ws_stage_bytes(int ng) {
    return (uint32_t)(2 * ng + 12) * WS_CHUNK;
}

// Loads of elements [c0, c0 + len) of shard d into the stage at smem offset
// `stage`: the 16-bit arrays first (2 * WS_CHUNK bytes each: FUSED, every
// slice at the shard's gradient offset; otherwise the reduced gradient), then
// master, m, v.
template <bool FUSED>
__device__ __forceinline__ void ws_issue(const StepArgs& a, const ShardDev& d, bool sw, int64_t c0, int64_t len,
                                         uint32_t stage, uint32_t bar) {
    const int ng = FUSED ? a.n_slices : 1;
    const uint32_t blen = (uint32_t)(len & ~int64_t(7));
    mbar_expect_tx(bar, blen * (2u * ng + 12u));
    if (blen == 0) return;
    for (int r = 0; r < ng; ++r) {
        const uint16_t* src = FUSED ? static_cast<const uint16_t*>(a.slices[r]) + d.grad_off + c0
                                    : static_cast<const uint16_t*>(d.gshard) + c0;
        bulk_load(stage + (uint32_t)r * WS_CHUNK * 2, src, blen * 2u, bar);
    }
    const uint32_t so = (uint32_t)ng * WS_CHUNK * 2;
    const StatePtrs p = state_ptrs(d, sw);
    bulk_load(stage + so, p.mi + c0, blen * 4u, bar);
    bulk_load(stage + so + WS_CHUNK * 4, p.mmi + c0, blen * 4u, bar);
    bulk_load(stage + so + 2 * WS_CHUNK * 4, p.vi + c0, blen * 4u, bar);
}

// V 16-bit values from shared memory as V/2 words.
template <int V>
__device__ __forceinline__ void load_halves(const uint8_t* p, uint32_t (&u)[V / 2]) {
    if constexpr (V == 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        u[0] = w.x; u[1] = w.y; u[2] = w.z; u[3] = w.w;
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        u[0] = w.x; u[1] = w.y;
    }
}

// One element by plain loads and stores (a shard's head and last few elements).
template <int GDT, int PDT, bool FUSED>
__device__ __forceinline__ void ws_elem(const StepArgs& a, const ShardDev& d, int64_t i, float k, const Ctl& c,
                                        SumSq& sumsq, int& flags) {
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    uint32_t h;
    if (FUSED) {
        h = average16<GDT>(reduce1<GDT>(a, d.grad_off + i), a.divisor);
        if (Half16<GDT>::nonfinite(h)) flags |= FLAG_OVERFLOW;
    } else {
        h = static_cast<const uint16_t*>(d.gshard)[i];
    }
    const float af = Half16<GDT>::widen(h);
    if (FUSED) sumsq.add_fp64(af);
    const StatePtrs p = state_ptrs(d, c.sw);
    float th = p.mi[i], mm = p.mmi[i], vv = p.vi[i];
    adamw1(th, mm, vv, af, k, a.sc, c.ss, c.rb2);
    p.mo[i] = th;
    p.mmo[i] = mm;
    p.vo[i] = vv;
    P[d.param_off + i] = (uint16_t)Half16<PDT>::narrow(th);
}

// FUSED: reduce the slices, statistics, AdamW with multiplier a.k, and (last
// block) the result.  Otherwise the apply pass: AdamW from the reduced
// gradient with the decision every block derives from the statistics; on
// overflow nothing is loaded or written.  Either way every block publishes
// its flags and the last block to finish writes the result, so a timeout
// anywhere is reported.
template <int GDT, int PDT, bool FUSED>
__global__ void __launch_bounds__(TILE_THREADS, WS_BLOCKS_PER_SM) k_ws(const __grid_constant__ StreamArgs sa) {
    extern __shared__ __align__(128) uint8_t smem[];
    const StepArgs& a = sa.a;
    const int S = sa.stages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ng = FUSED ? a.n_slices : 1;
    const uint32_t full0 = smem_addr(smem), empty0 = full0 + 8 * WS_MAX_STAGES;
    const uint32_t stage0 = full0 + WS_HEADER;
    const uint32_t stage_bytes = ws_stage_bytes(ng);
    const int64_t G = gridDim.x;
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);

    const Ctl c = step_ctl(a);
    float k = c.k;
    int overflow_in = 0;
    double st_sumsq = 0.0, norm = 0.0, clip = 1.0;
    if (!FUSED) {
        const zero_stats st = *a.stats;
        overflow_in = (st.overflow | a.extra_overflow) ? 1 : 0;
        st_sumsq = st.sumsq + a.extra_sumsq;
        k = grad_multiplier(st_sumsq, step_S(a), a.max_norm, norm, clip);
    }
    const int64_t n_local = (!overflow_in && !c.bad && a.n_tiles > (int64_t)blockIdx.x)
                                ? (a.n_tiles - 1 - blockIdx.x) / G + 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, WS_CONSUMER_WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    SumSq sumsq;
    int flags = 0;
    if (warp == 0) {
        if (lane == 0 && n_local > 0) {
            int si = 0;
            int st = 0;
            uint32_t phase = 0;         // parity of the empty barrier's phase this use waits for
            int64_t j = 0;
            for (; j < n_local; ++j) {
                if (j >= S && !mbar_wait(empty0 + 8 * st, phase, sa.spin_limit)) {
                    flags |= FLAG_TIMEOUT;
                    break;
                }
                const int64_t chunk = blockIdx.x + j * G;
                while (si + 1 < a.n_shards && a.shards[si + 1].tile_begin <= chunk) ++si;
                const ShardDev& d = a.shards[si];
                const int64_t c0 = d.head + (chunk - d.tile_begin) * WS_CHUNK;
                const int64_t rem = d.numel - c0;
                ws_issue<FUSED>(a, d, c.sw, c0, rem < WS_CHUNK ? (rem > 0 ? rem : 0) : WS_CHUNK,
                                stage0 + (uint32_t)st * stage_bytes, full0 + 8 * st);
                if (++st == S) {        // the uses of round r >= 1 wait for the consumption of round r - 1
                    st = 0;
                    if (j >= S) phase ^= 1u;
                }
            }
            // Before the block moves on, the last S chunks issued (one per stage,
            // the latest use of each) must have landed, also when a consumer
            // gave up on them: a bounded wait for each (at once when complete).
            for (int64_t q = (j > S ? j - S : 0); q < j; ++q)
                mbar_wait(full0 + 8 * (int)(q % S), (uint32_t)((q / S) & 1), sa.drain_limit);
        }
    } else {
        constexpr int V = WS_VEC;
        const int e0 = V * ((warp - 1) * 32 + lane);
        int si = 0;
        int st = 0;
        uint32_t phase = 0;
        for (int64_t j = 0; j < n_local; ++j) {
            if (!mbar_wait(full0 + 8 * st, phase, sa.spin_limit)) {
                flags |= FLAG_TIMEOUT;
                break;
            }
            const int64_t chunk = blockIdx.x + j * G;
            while (si + 1 < a.n_shards && a.shards[si + 1].tile_begin <= chunk) ++si;
            const ShardDev& d = a.shards[si];
            const int64_t it = chunk - d.tile_begin;
            const int64_t c0 = d.head + it * WS_CHUNK;
            const int64_t rem = d.numel - c0;
            const int64_t len = rem < WS_CHUNK ? (rem > 0 ? rem : 0) : WS_CHUNK;
            const int64_t blen = len & ~int64_t(7);
            const uint8_t* in = smem + WS_HEADER + (size_t)st * stage_bytes;
            if (it == 0 && e0 / V < d.head) ws_elem<GDT, PDT, FUSED>(a, d, e0 / V, k, c, sumsq, flags);  // the head
            if (e0 + V <= blen) {
                uint32_t hg[V];                   // the averaged (FUSED) or reduced 16-bit gradient
                if (FUSED) {
                    float sv[V];
#pragma unroll
                    for (int e = 0; e < V; ++e) sv[e] = 0.0f;
                    for (int r = 0; r < ng; ++r) {
                        uint32_t u[V / 2];
                        load_halves<V>(in + (size_t)r * WS_CHUNK * 2 + e0 * 2, u);
#pragma unroll
                        for (int q = 0; q < V / 2; ++q) {
                            sv[2 * q] = __fadd_rn(sv[2 * q], Half16<GDT>::widen(u[q] & 0xFFFFu));
                            sv[2 * q + 1] = __fadd_rn(sv[2 * q + 1], Half16<GDT>::widen(u[q] >> 16));
                        }
                    }
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        hg[e] = average16<GDT>(sv[e], a.divisor);
                        if (Half16<GDT>::nonfinite(hg[e])) flags |= FLAG_OVERFLOW;
                    }
                } else {
                    uint32_t u[V / 2];
                    load_halves<V>(in + e0 * 2, u);
#pragma unroll
                    for (int q = 0; q < V / 2; ++q) {
                        hg[2 * q] = u[q] & 0xFFFFu;
                        hg[2 * q + 1] = u[q] >> 16;
                    }
                }
                const uint8_t* sin = in + (size_t)ng * WS_CHUNK * 2;
                float th[V], mm[V], vv[V];
#pragma unroll
                for (int q = 0; q < V / 4; ++q) {
                    const float4 t = *reinterpret_cast<const float4*>(sin + (e0 + 4 * q) * 4);
                    const float4 m = *reinterpret_cast<const float4*>(sin + WS_CHUNK * 4 + (e0 + 4 * q) * 4);
                    const float4 v = *reinterpret_cast<const float4*>(sin + 2 * WS_CHUNK * 4 + (e0 + 4 * q) * 4);
                    th[4 * q] = t.x; th[4 * q + 1] = t.y; th[4 * q + 2] = t.z; th[4 * q + 3] = t.w;
                    mm[4 * q] = m.x; mm[4 * q + 1] = m.y; mm[4 * q + 2] = m.z; mm[4 * q + 3] = m.w;
                    vv[4 * q] = v.x; vv[4 * q + 1] = v.y; vv[4 * q + 2] = v.z; vv[4 * q + 3] = v.w;
                }
                float af[V];
                uint32_t hp[V];
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    af[e] = Half16<GDT>::widen(hg[e]);
                    adamw1(th[e], mm[e], vv[e], af[e], k, a.sc, c.ss, c.rb2);
                }
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    const uint32_t w = Half16<PDT>::narrow2(th[e], th[e + 1]);
                    hp[e] = w & 0xFFFFu;
                    hp[e + 1] = w >> 16;
                }
                if (FUSED) {
                    if constexpr (V == 8) sumsq.add8(*reinterpret_cast<const float(*)[8]>(af));
                    else sumsq.add4(*reinterpret_cast<const float(*)[4]>(af));
                }
                const StatePtrs sp = state_ptrs(d, c.sw);
#pragma unroll
                for (int q = 0; q < V / 4; ++q) {
                    const int e = 4 * q;
                    st_stream4(sp.mo + c0 + e0 + e, make_float4(th[e], th[e + 1], th[e + 2], th[e + 3]));
                    st_stream4(sp.mmo + c0 + e0 + e, make_float4(mm[e], mm[e + 1], mm[e + 2], mm[e + 3]));
                    st_stream4(sp.vo + c0 + e0 + e, make_float4(vv[e], vv[e + 1], vv[e + 2], vv[e + 3]));
                }
                if constexpr (V == 8) store8(P, d.param_off + c0 + e0, *reinterpret_cast<const uint32_t(*)[8]>(hp));
                else store4(P, d.param_off + c0 + e0, *reinterpret_cast<const uint32_t(*)[4]>(hp));
            } else if (e0 < len) {
                // the shard's last (fewer than 8) elements: plain loads and stores
                const int64_t end = (e0 + V < len) ? e0 + V : len;
                for (int64_t e = (e0 > blen ? e0 : blen); e < end; ++e)
                    ws_elem<GDT, PDT, FUSED>(a, d, c0 + e, k, c, sumsq, flags);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            if (++st == S) {
                st = 0;
                phase ^= 1u;
            }
        }
    }

    double acc = FUSED ? sumsq.total() : 0.0;
    block_reduce(acc, flags);
    if (!publish_partial(a, acc, flags)) return;
    double sum;
    int flag;
    combine_partials(a, sum, flag);
    if (threadIdx.x == 0) {
        zero_result r;
        if (FUSED) {
            r.overflow = ((flag & FLAG_OVERFLOW) || a.extra_overflow) ? 1 : 0;
            r.sumsq = sum + a.extra_sumsq;
            r.grad_norm = sqrt(r.sumsq) / step_S(a);
            r.clip_coef = 1.0;
            r.grad_mult = (float)(1.0 / step_S(a));
        } else {
            r.overflow = overflow_in;
            r.sumsq = st_sumsq;
            r.grad_norm = norm;
            r.clip_coef = clip;
            r.grad_mult = k;
        }
        r.status = (flag & FLAG_TIMEOUT) ? ZERO_ETIMEOUT : (step_bad(a) ? ZERO_ELIMIT : 0);
        r.applied = (r.overflow || r.status) ? 0 : 1;
        r.path = FUSED ? 5 : 6;
        r.reserved = 0.0f;
        *a.result = r;
    }
}

template <int G, int P>
static const void* ws_ptr(bool fused) {
    return fused ? (const void*)k_ws<G, P, true> : (const void*)k_ws<G, P, false>;
}

static const void* ws_kernel(int gdt, int pdt, bool fused) {
    if (gdt == ZERO_BF16) return pdt == ZERO_BF16 ? ws_ptr<ZERO_BF16, ZERO_BF16>(fused)
                                                  : ws_ptr<ZERO_BF16, ZERO_F16>(fused);
    return pdt == ZERO_BF16 ? ws_ptr<ZERO_F16, ZERO_BF16>(fused) : ws_ptr<ZERO_F16, ZERO_F16>(fused);
}

int ws_chunk() { return WS_CHUNK; }

// Stages of a block for ng 16-bit arrays: as many as fit 110 KB (two blocks
// share an SM), at most 8.
int ws_stages(int ng) {
    const int s = (int)((110 * 1024 - WS_HEADER) / ws_stage_bytes(ng));
    return s > WS_MAX_STAGES ? WS_MAX_STAGES : s;
}

int launch_ws(const StreamArgs& sa, int gdt, int pdt, bool fused, cudaStream_t s) {
    const void* f = ws_kernel(gdt, pdt, fused);
    const size_t smem = WS_HEADER + (size_t)sa.stages * ws_stage_bytes(fused ? sa.a.n_slices : 1);
    static std::mutex mu;
    static std::unordered_map<const void*, size_t> configured[16];
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> g(mu);
        size_t& have = configured[dev & 15][f];
        if (have < smem) {
            int rc = cuda_fail(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                               "raising the shared-memory limit of the producer/consumer kernel");
            if (rc != ZERO_OK) return rc;
            have = smem;
        }
    }
    const int grid = grid_for_smem(f, sa.a.n_tiles, smem, WS_BLOCKS_PER_SM);
    void* args[] = {const_cast<StreamArgs*>(&sa)};
    return cuda_fail(cudaLaunchKernel(f, dim3(grid), dim3(TILE_THREADS), args, smem, s),
                     "producer/consumer kernel launch");
}

}  // namespace zdp
