// zero_kernels.cuh -- device code of the partitioned mixed-precision step for
// sm_103a (GB300).  Everything here is memory-bound streaming: per shard
// element the fused pass moves 2*N_d bytes of gradient slices, 12 bytes of
// fp32 state in and 12 out, and 2 bytes of parameter out.  No tensor cores:
// nothing on this path is a contraction.
//
// Design:
//  * Work unit = a tile of TILE_THREADS x VEC elements of one shard; tiles are
//    numbered shard after shard and a grid of (SM count x resident blocks)
//    strides over them.  VEC = 8 uses 128-bit loads of 8 16-bit gradients
//    per slice and two 128-bit loads per fp32 state array; VEC = 1 is the
//    path for pointers that are not 16-byte aligned.
//  * All loads of one vector (state first, then the slices in groups of 8)
//    are issued before their values are used, so each thread keeps ~100-250
//    bytes in flight; loads and stores use the streaming cache hints because
//    no byte is touched twice.
//  * Gradient statistics: squares of the 16-bit reduced values are exact in
//    fp32 (at most 22 significant bits).  Each vector's squares are summed on
//    the fp32 pipe with error-free TwoSum steps, the vector sum is added in
//    fp64 (one fp64 add per 8 elements: GB300's fp64 rate is far too low for
//    one per element) and the exact rounding errors are carried apart (see
//    SumSq).  A warp shuffle and a shared-memory pass give one fp64 partial
//    per block, stored in the workspace; the last block to finish (one atomic
//    per block) adds the partials in block order, so the result is
//    deterministic for a given grid.
//  * Every fp32 operation of the reduction and of AdamW is an explicitly
//    rounded intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn) so no
//    multiply-add is contracted: results are those of the plain IEEE sequence.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "zero.h"

namespace zdp {

constexpr int TILE_THREADS = 256;
constexpr int MAX_BLOCKS = 2048;

// ---------------------------------------------------------------- layout of the workspace
// [0, 64)              completion counter (unsigned) -- zero between calls
// [64, 80)             the step's internal zero_stats (two-pass path of zero_shard_step)
// [128, 128 + 8*MB)    per-block fp64 partial sums of squares
// [.., + 4*MB)         per-block overflow flags
constexpr size_t WS_COUNTER = 0;
constexpr size_t WS_STATS = 64;
constexpr size_t WS_PARTIALS = 128;
constexpr size_t WS_FLAGS = WS_PARTIALS + 8 * (size_t)MAX_BLOCKS;
constexpr size_t WS_BYTES = ((WS_FLAGS + 4 * (size_t)MAX_BLOCKS) + 4095) / 4096 * 4096;

// ---------------------------------------------------------------- kernel arguments
struct ShardDev {
    int64_t numel, grad_off, param_off;
    int64_t tile_begin;             // index of the shard's first tile
    int64_t head;                   // elements before the first 128-byte-aligned vector (done one by one)
    const float *mi, *mmi, *vi;     // master, m, v in
    float *mo, *mmo, *vo;           // master, m, v out
    void* gshard;                   // 16-bit reduced gradient shard
};

struct AdamScalars {                // fp32, each rounded once from fp64 on the host
    float b1, b2, omb1, omb2, eps, wdf, ss, rb2;
};

struct StepArgs {
    const void* slices[ZERO_MAX_SLICES];
    ShardDev shards[ZERO_MAX_SHARDS];
    int n_slices, n_shards;
    int64_t n_tiles;
    void* flat_param;
    float divisor;                  // N_d
    float k;                        // gradient multiplier (fused path: 1/S, exact for S a power of two)
    AdamScalars sc;
    double loss_scale, max_norm, extra_sumsq;
    int extra_overflow, accumulate;
    double* partials;
    int* block_flags;
    unsigned* counter;
    zero_stats* stats;
    zero_result* result;
    // chained steps (NULL chain otherwise): t, S and the state set in use come
    // from *chain; the step-dependent scalars from sc_table (2 per step, from t0)
    zero_chain* chain;
    const float* sc_table;
    int64_t t0, n_table;
};

// ---------------------------------------------------------------- 16-bit conversions
template <int DT> struct Half16;
template <> struct Half16<ZERO_BF16> {
    static __device__ __forceinline__ float widen(uint32_t h) { return __uint_as_float(h << 16); }
    static __device__ __forceinline__ uint32_t narrow(float x) {
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
    static __device__ __forceinline__ bool nonfinite(uint32_t h) { return (h & 0x7F80u) == 0x7F80u; }
    // two values, rounded as narrow() does, packed low | high << 16
    static __device__ __forceinline__ uint32_t narrow2(float lo, float hi) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&p);
    }
};
template <> struct Half16<ZERO_F16> {
    static __device__ __forceinline__ float widen(uint32_t h) {
        return __half2float(__ushort_as_half((unsigned short)h));
    }
    static __device__ __forceinline__ uint32_t narrow(float x) {
        return (uint32_t)__half_as_ushort(__float2half_rn(x));
    }
    static __device__ __forceinline__ bool nonfinite(uint32_t h) { return (h & 0x7C00u) == 0x7C00u; }
    static __device__ __forceinline__ uint32_t narrow2(float lo, float hi) {
        const __half2 p = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&p);
    }
};

// 8 packed 16-bit values (one uint4) -> fp32, added in order to s[0..7]
template <int DT>
__device__ __forceinline__ void add8(float (&s)[8], const uint4& w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        s[2 * q] = __fadd_rn(s[2 * q], Half16<DT>::widen(u[q] & 0xFFFFu));
        s[2 * q + 1] = __fadd_rn(s[2 * q + 1], Half16<DT>::widen(u[q] >> 16));
    }
}

// ---------------------------------------------------------------- streaming memory access
// Data that no thread writes while the kernel runs (gradient slices; the
// *_in state of the fused pass, whose outputs go to a distinct state set) is
// read through the non-coherent read-only path; data that may be written in
// place (the apply pass's state) with streaming loads.  Stores are streaming
// (evict-first): nothing is read back.
__device__ __forceinline__ uint4 ld_ro(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float4 ld_ro4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ uint4 ld_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float4 ld_stream4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream4(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

// A thread's 8 consecutive fp32 state values.  WIDE: one 256-bit access
// (sm_100 and later; the address 32-byte aligned), so that a warp's request
// covers 1 KB of one array with every 32-byte sector whole, where two 128-bit
// accesses each ask for half of every sector of the same 1 KB.  The host
// picks the instantiation for a whole launch (state_wide, fused_state_wide):
// a per-vector choice inside one kernel cost more than the wider accesses
// saved.  ld_state8: streaming loads (the apply pass, whose state may be
// updated in place); ld_state8_ro: the read-only path (the fused pass's *_in
// state, which no thread writes).
template <bool WIDE>
__device__ __forceinline__ void ld_state8(const float* p, float4& lo, float4& hi) {
    if (WIDE) {
        asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z), "=f"(hi.w)
                     : "l"(p));
    } else {
        lo = ld_stream4(p);
        hi = ld_stream4(p + 4);
    }
}

template <bool WIDE>
__device__ __forceinline__ void ld_state8_ro(const float* p, float4& lo, float4& hi) {
    if (WIDE) {
        asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z), "=f"(hi.w)
                     : "l"(p));
    } else {
        lo = ld_ro4(p);
        hi = ld_ro4(p + 4);
    }
}

template <bool WIDE>
__device__ __forceinline__ void st_state8(float* p, const float (&v)[8]) {
    if (WIDE) {
        asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :
                     : "l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                     : "memory");
    } else {
        st_stream4(p, make_float4(v[0], v[1], v[2], v[3]));
        st_stream4(p + 4, make_float4(v[4], v[5], v[6], v[7]));
    }
}

// ---------------------------------------------------------------- programmatic dependent launch
// The gather and reduce kernels run back to back many times per step (two
// gathers and one reduce per ZeRO-3 unit), 0.1 ms each, and a launch's
// ramp-up and tail cost them a few microseconds each.  They are launched with
// programmatic stream serialisation: a launch may begin while the previous
// kernel of the stream finishes.  Every thread first waits for the previous
// grid to complete and its memory to be visible (griddepcontrol.wait; at once
// if there is no such grid), so no access is reordered.  Each block then lets
// the next kernel of the stream launch (griddepcontrol.launch_dependents).
// That kernel launches only once every block of this grid has started, so its
// waiting blocks cannot keep any of this grid's blocks from running.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------- per-element arithmetic
// Reduce-scatter arithmetic for one element: s is the rank-ordered fp32 sum.
template <int GDT>
__device__ __forceinline__ uint32_t average16(float s, float divisor) {
    return Half16<GDT>::narrow(__fdiv_rn(s, divisor));
}

// The same with the slice count known at compile time: a power-of-two
// divisor is a multiplication by its exact reciprocal, which rounds the same
// exact value s / 2^k once -- the identical result, in one instruction.
template <int GDT, int NS>
__device__ __forceinline__ uint32_t average16n(float s, float divisor) {
    if (NS == 1 || NS == 2 || NS == 4 || NS == 8) return Half16<GDT>::narrow(__fmul_rn(s, 1.0f / (float)NS));
    return average16<GDT>(s, divisor);
}

// AdamW on one coordinate, the operations in the order of the update rule.
// ss and rb2 (the step-dependent scalars) come apart from the rest, so that
// the rest can stay in the kernel's parameter space.
__device__ __forceinline__ void adamw1(float& th, float& m, float& v, float a, float k, const AdamScalars& c,
                                       float ss, float rb2) {
    const float g = __fmul_rn(a, k);
    th = __fmul_rn(th, c.wdf);
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
    const float g2 = __fmul_rn(g, g);
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, g2));
    const float den = __fadd_rn(__fmul_rn(__fsqrt_rn(v), rb2), c.eps);
    th = __fsub_rn(th, __fmul_rn(ss, __fdiv_rn(m, den)));
}

__device__ __forceinline__ void adamw1(float& th, float& m, float& v, float a, float k, const AdamScalars& c) {
    adamw1(th, m, v, a, k, c, c.ss, c.rb2);
}

// Store 8 16-bit values at dst + q with the widest stores its address allows
// (16, 4 or 2 bytes; the choice is uniform across a shard's vectors).
__device__ __forceinline__ void store8(uint16_t* dst, int64_t q, const uint32_t (&h)[8]) {
    const int mis = (int)(reinterpret_cast<uintptr_t>(dst + q) & 15u);
    if (mis == 0) {
        uint4 w;
        w.x = h[0] | (h[1] << 16);
        w.y = h[2] | (h[3] << 16);
        w.z = h[4] | (h[5] << 16);
        w.w = h[6] | (h[7] << 16);
        __stcs(reinterpret_cast<uint4*>(dst + q), w);
    } else if ((mis & 3) == 0) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) __stcs(reinterpret_cast<unsigned*>(dst + q + e), h[e] | (h[e + 1] << 16));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) __stcs(reinterpret_cast<unsigned short*>(dst + q + e), (unsigned short)h[e]);
    }
}

// ---------------------------------------------------------------- reductions
// Sum of squares of 16-bit values.  A square of a 16-bit value is exact in
// fp32 (at most 22 significant bits).  The squares of one vector are added in
// fp32 with TwoSum (Knuth): t = s + q rounded, and e = (s - (t - z)) + (q - z)
// with z = t - s is exactly the rounding error s + q - t, whatever the
// operands' magnitudes.  Each vector's fp32 sum goes into an fp64 accumulator
// (one fp64 add per vector: a small share of GB300's fp64 rate) and its
// rounding errors into an fp32 one, added in at the end.  The result is then
// off the exact sum by a few fp64 roundings, far below fp32 resolution, so
// the multiplier fp32(c / S) derived from it almost never differs from the
// one an exactly rounded sum gives -- even for a thread that sums only one
// vector, where a Kahan-compensated fp32 sum loses its compensation (the
// correction falls below half an ulp of the next term; measured: 3e-9
// relative off the exact sum on a small clipped step).
struct SumSq {
    double acc = 0.0;   // sum of the vectors' fp32 sums (and of any squares taken in fp64)
    float err = 0.0f;   // sum of the exact TwoSum rounding errors

    // Add s + q to the running vector sum s, keeping the rounding error.
    __device__ __forceinline__ void two_sum(float& s, float q) {
        const float t = __fadd_rn(s, q);
        const float z = __fsub_rn(t, s);
        err = __fadd_rn(err, __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(q, z)));
        s = t;
    }
    // Add the squares of N fp32 values (exact products); vectors whose squares
    // leave the fp32 range go to fp64 directly.
    template <int N>
    __device__ __forceinline__ void addn(const float (&a)[N]) {
        float q[N];
        bool ok = true;
#pragma unroll
        for (int e = 0; e < N; ++e) {
            q[e] = __fmul_rn(a[e], a[e]);
            ok &= q[e] < 1e30f;          // false for inf, NaN and huge squares
        }
        if (ok) {
            float s = q[0];
#pragma unroll
            for (int e = 1; e < N; ++e) two_sum(s, q[e]);
            acc += (double)s;
        } else {
#pragma unroll
            for (int e = 0; e < N; ++e) acc += (double)a[e] * (double)a[e];
        }
    }
    __device__ __forceinline__ void add8(const float (&a)[8]) { addn<8>(a); }
    __device__ __forceinline__ void add_fp64(float a) { acc += (double)a * (double)a; }
    __device__ __forceinline__ double total() { return acc + (double)err; }
};

__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Block-wide sum (fixed order) of x and bitwise OR of f; valid in thread 0.
__device__ __forceinline__ void block_reduce(double& x, int& f) {
    __shared__ double sx[TILE_THREADS / 32];
    __shared__ int sf[TILE_THREADS / 32];
    x = warp_sum(x);
    f = (int)__reduce_or_sync(0xffffffffu, (unsigned)f);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { sx[w] = x; sf[w] = f; }
    __syncthreads();
    if (w == 0) {
        x = l < TILE_THREADS / 32 ? sx[l] : 0.0;
        f = l < TILE_THREADS / 32 ? sf[l] : 0;
        x = warp_sum(x);
        f = (int)__reduce_or_sync(0xffffffffu, (unsigned)f);
    }
}

// Publish this block's partial; returns true in thread 0 of the last block to
// finish, after which that block may read every partial.
__device__ __forceinline__ bool publish_partial(const StepArgs& a, double x, int f) {
    __shared__ bool last;
    if (threadIdx.x == 0) {
        a.partials[blockIdx.x] = x;
        a.block_flags[blockIdx.x] = f;
        __threadfence();
        const unsigned done = atomicAdd(a.counter, 1u);
        last = (done == gridDim.x - 1);
    }
    __syncthreads();
    return last;
}

// In the last block: the sum of all partials in block order and the OR of the
// flags (thread 0 gets the result); resets the counter for the next call.
__device__ __forceinline__ void combine_partials(const StepArgs& a, double& sum, int& flag) {
    __threadfence();
    // fixed order: thread t adds partials t, t + 256, ... ; then the block sum
    double x = 0.0;
    int f = 0;
    for (int b = threadIdx.x; b < (int)gridDim.x; b += TILE_THREADS) {
        x += __ldcg(a.partials + b);
        f |= __ldcg(a.block_flags + b);
    }
    block_reduce(x, f);
    sum = x;
    flag = f;
    if (threadIdx.x == 0) *a.counter = 0u;
}

// Clip decision from the statistics (fp64, the same on every block).
__device__ __forceinline__ float grad_multiplier(double sumsq, double S, double max_norm, double& norm,
                                                 double& clip) {
    norm = sqrt(sumsq) / S;
    clip = 1.0;
    if (max_norm > 0.0) {
        const double c = max_norm / (norm + 1e-6);
        if (c < 1.0) clip = c;
    }
    return (float)(clip / S);
}

// The shard that holds `tile`, searched upward from shard s: a block's tiles
// only increase, so a loop passes the previous answer and the search costs
// one comparison a tile instead of one per preceding shard.
__device__ __forceinline__ int find_shard(const StepArgs& a, int64_t tile, int s = 0) {
    while (s + 1 < a.n_shards && a.shards[s + 1].tile_begin <= tile) ++s;
    return s;
}

// ---------------------------------------------------------------- gradient reduction of one vector
// Sum of the n slices' 8 values at element offset off (rank order), with the
// loads of each group of 8 slices issued together.
template <int GDT, int NS>
__device__ __forceinline__ void reduce8(const StepArgs& a, int64_t off, float (&s)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = 0.0f;
    if (NS > 0) {
        uint4 w[NS > 0 ? NS : 1];
#pragma unroll
        for (int r = 0; r < NS; ++r) w[r] = ld_ro(static_cast<const uint16_t*>(a.slices[r]) + off);
#pragma unroll
        for (int r = 0; r < NS; ++r) add8<GDT>(s, w[r]);
    } else {
        const int n = a.n_slices;
        int r = 0;
        for (; r + 8 <= n; r += 8) {
            uint4 w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) w[q] = ld_ro(static_cast<const uint16_t*>(a.slices[r + q]) + off);
#pragma unroll
            for (int q = 0; q < 8; ++q) add8<GDT>(s, w[q]);
        }
        if (NS < 0) {
            // The few-slice loop (up to 128 registers): the last n - r < 8
            // slices too with every load issued before the first add.  One at
            // a time, a slice's load would wait for the previous slice's add:
            // with 4 slices (a ZeRO-3 unit pass) that is every slice.
            const int rem = n - r;
            if (rem > 0) {
                uint4 w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < rem) w[q] = ld_ro(static_cast<const uint16_t*>(a.slices[r + q]) + off);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < rem) add8<GDT>(s, w[q]);
            }
        } else {
            for (; r < n; ++r) add8<GDT>(s, ld_ro(static_cast<const uint16_t*>(a.slices[r]) + off));
        }
    }
}

template <int GDT>
__device__ __forceinline__ float reduce1(const StepArgs& a, int64_t off) {
    float s = 0.0f;
    for (int r = 0; r < a.n_slices; ++r)
        s = __fadd_rn(s, Half16<GDT>::widen(static_cast<const uint16_t*>(a.slices[r])[off]));
    return s;
}

// ---------------------------------------------------------------- per-step control
// What a kernel needs of the step that is not in its arguments for a chained
// step: the scalars, the multiplier, S, and which state set is read.
struct Ctl {
    float ss, rb2;      // the step-dependent AdamW scalars (the others stay in a.sc)
    float k;            // the fused pass's gradient multiplier, fp32(1/S)
    bool sw;            // the state sets are used the other way round (chain->cur == 1)
    bool bad;           // a chained step outside its scalar table: nothing is updated
};

// S of the step (read again where it is needed, rather than kept live).
__device__ __forceinline__ double step_S(const StepArgs& a) {
    return a.chain ? __ldcg(&a.chain->loss_scale) : a.loss_scale;
}

__device__ __forceinline__ bool step_bad(const StepArgs& a) {
    if (!a.chain) return false;
    const int64_t i = __ldcg(&a.chain->step) - a.t0;
    return i < 0 || i >= a.n_table;
}

__device__ __forceinline__ Ctl step_ctl(const StepArgs& a) {
    Ctl c;
    c.ss = a.sc.ss;
    c.rb2 = a.sc.rb2;
    c.k = a.k;
    c.sw = false;
    c.bad = false;
    if (a.chain) {
        const int cur = __ldcg(&a.chain->cur);
        const int64_t t = __ldcg(&a.chain->step);
        c.k = (float)(1.0 / __ldcg(&a.chain->loss_scale));
        c.sw = cur != 0;
        const int64_t i = t - a.t0;
        if (i < 0 || i >= a.n_table) {
            c.bad = true;
        } else {
            c.ss = __ldg(a.sc_table + 2 * i);
            c.rb2 = __ldg(a.sc_table + 2 * i + 1);
        }
    }
    return c;
}

// A shard's state set read and state set written.
struct StatePtrs {
    const float *mi, *mmi, *vi;
    float *mo, *mmo, *vo;
};

__device__ __forceinline__ StatePtrs state_ptrs(const ShardDev& d, bool sw) {
    if (!sw) return StatePtrs{d.mi, d.mmi, d.vi, d.mo, d.mmo, d.vo};
    return StatePtrs{d.mo, d.mmo, d.vo, const_cast<float*>(d.mi), const_cast<float*>(d.mmi),
                     const_cast<float*>(d.vi)};
}

// ---------------------------------------------------------------- one element at a time
// The per-element bodies of the passes, for the elements the vector loops do
// not cover (a shard's unaligned head and ragged tail, or everything on the
// scalar path).  Same arithmetic as the vector bodies.
template <int GDT, int PDT>
__device__ __forceinline__ void fused_elem(const StepArgs& a, const ShardDev& d, int64_t i, const Ctl& c,
                                           SumSq& sumsq, int& ovf) {
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    const uint32_t h = average16<GDT>(reduce1<GDT>(a, d.grad_off + i), a.divisor);
    ovf |= Half16<GDT>::nonfinite(h);
    const float af = Half16<GDT>::widen(h);
    sumsq.add_fp64(af);
    const StatePtrs p = state_ptrs(d, c.sw);
    float th = p.mi[i], mm = p.mmi[i], vv = p.vi[i];
    adamw1(th, mm, vv, af, c.k, a.sc, c.ss, c.rb2);
    p.mo[i] = th;
    p.mmo[i] = mm;
    p.vo[i] = vv;
    P[d.param_off + i] = (uint16_t)Half16<PDT>::narrow(th);
}

template <int GDT>
__device__ __forceinline__ void reduce_elem(const StepArgs& a, const ShardDev& d, int64_t i, SumSq& sumsq, int& ovf) {
    const uint32_t h = average16<GDT>(reduce1<GDT>(a, d.grad_off + i), a.divisor);
    ovf |= Half16<GDT>::nonfinite(h);
    sumsq.add_fp64(Half16<GDT>::widen(h));
    static_cast<uint16_t*>(d.gshard)[i] = (uint16_t)h;
}

template <int GDT, int PDT>
__device__ __forceinline__ void apply_elem(const StepArgs& a, const ShardDev& d, int64_t i, float k, const Ctl& c) {
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    const StatePtrs p = state_ptrs(d, c.sw);
    float th = p.mi[i], mm = p.mmi[i], vv = p.vi[i];
    adamw1(th, mm, vv, Half16<GDT>::widen(static_cast<const uint16_t*>(d.gshard)[i]), k, a.sc, c.ss, c.rb2);
    p.mo[i] = th;
    p.mmo[i] = mm;
    p.vo[i] = vv;
    P[d.param_off + i] = (uint16_t)Half16<PDT>::narrow(th);
}

// ---------------------------------------------------------------- K1a: fused single pass
// Reads the slices and the *_in state once, writes the *_out state and the
// 16-bit parameters once.  Speculative: the skip decision is global, so the
// *_out state is only committed by the caller when result->applied; the
// parameters are restored by k_recover on overflow.
// NS: 0 = the generic slice loop for many slices, 4 blocks per SM (at most
// 64 registers; chained steps 3, at most 85); NS_FEW = the same loop for at
// most FEW_SLICES slices, 2 blocks per SM (up to 128 registers: every load of
// a vector is in flight at once); NS = 4 = the loop unrolled for exactly 4
// slices, 2 blocks per SM.  Measured on the GPT-2 step (8 slices): 9.51 ms
// with NS_FEW, against 9.72 ms for the loop unrolled for exactly 8 slices at
// 64 registers and 10.77 ms for the 64-register generic loop; on the ZeRO-3
// unit passes (4 slices): 0.3130 ms with NS = 4 against 0.3200 ms with
// NS_FEW, and 0.341 ms with NS = 4 at 3 blocks per SM.
// CHAIN: a chained step (t, S and the state set from a.chain); the other
// instantiations take everything from their arguments.
template <int GDT, int PDT, int VEC, int NS, bool CHAIN = false, bool WIDE = false>
__global__ void __launch_bounds__(TILE_THREADS, NS == 0 ? (CHAIN ? 3 : 4) : 2)   // chained: 3, so no spills
k_step_fused(const __grid_constant__ StepArgs a) {
    constexpr int64_t TILE = (int64_t)TILE_THREADS * VEC;
    pdl_wait();             // a no-op unless launched early (partial passes, one per ZeRO-3 unit)
    pdl_launch_next();
    SumSq sumsq;
    int ovf = 0;
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    const Ctl c = CHAIN ? step_ctl(a) : Ctl{a.sc.ss, a.sc.rb2, a.k, false, false};
    const float k = c.k;
    int si = 0;
    for (int64_t tile = c.bad ? a.n_tiles : blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
        si = find_shard(a, tile, si);
        const ShardDev& d = a.shards[si];
        const int64_t it = tile - d.tile_begin;
        if (it == 0 && threadIdx.x < d.head && threadIdx.x < d.numel)
            fused_elem<GDT, PDT>(a, d, threadIdx.x, c, sumsq, ovf);      // the shard's unaligned head
        const int64_t j = d.head + it * TILE + (int64_t)threadIdx.x * VEC;
        if (j >= d.numel) continue;
        if (VEC == 8 && j + 8 <= d.numel) {
            const StatePtrs p = state_ptrs(d, c.sw);
            float4 t0, t1, m0, m1, v0, v1;
            ld_state8_ro<WIDE>(p.mi + j, t0, t1);
            ld_state8_ro<WIDE>(p.mmi + j, m0, m1);
            ld_state8_ro<WIDE>(p.vi + j, v0, v1);
            float s[8];
            reduce8<GDT, NS>(a, d.grad_off + j, s);
            float th[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
            float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float af[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t h = average16n<GDT, NS>(s[e], a.divisor);
                ovf |= Half16<GDT>::nonfinite(h);
                af[e] = Half16<GDT>::widen(h);
                adamw1(th[e], mm[e], vv[e], af[e], k, a.sc, c.ss, c.rb2);
            }
            uint32_t hp[8];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const uint32_t w = Half16<PDT>::narrow2(th[e], th[e + 1]);
                hp[e] = w & 0xFFFFu;
                hp[e + 1] = w >> 16;
            }
            sumsq.add8(af);
            st_state8<WIDE>(p.mo + j, th);
            st_state8<WIDE>(p.mmo + j, mm);
            st_state8<WIDE>(p.vo + j, vv);
            store8(P, d.param_off + j, hp);
        } else {
            const int64_t end = (VEC == 8) ? d.numel : j + 1;
            for (int64_t i = j; i < end; ++i) fused_elem<GDT, PDT>(a, d, i, c, sumsq, ovf);
        }
    }
    double acc = sumsq.total();
    block_reduce(acc, ovf);
    if (!publish_partial(a, acc, ovf)) return;
    double sum;
    int flag;
    combine_partials(a, sum, flag);
    if (threadIdx.x == 0 && a.stats) {
        // a partial pass: its statistics join the step's, decided later by k_commit
        zero_stats st = a.accumulate ? *a.stats : zero_stats{0.0, 0, 0};
        st.sumsq += sum;
        st.overflow |= flag;
        *a.stats = st;
    } else if (threadIdx.x == 0) {
        zero_result r;
        r.overflow = (flag | a.extra_overflow) ? 1 : 0;
        r.status = (CHAIN && step_bad(a)) ? ZERO_ELIMIT : 0;
        r.applied = (r.overflow || r.status) ? 0 : 1;
        r.path = 1;
        r.sumsq = sum + a.extra_sumsq;
        r.grad_norm = sqrt(r.sumsq) / (CHAIN ? step_S(a) : a.loss_scale);
        r.clip_coef = 1.0;
        r.grad_mult = CHAIN ? (float)(1.0 / step_S(a)) : a.k;
        r.reserved = 0.0f;
        *a.result = r;
    }
}

// ---------------------------------------------------------------- K1r: restore parameters after a skipped fused step
template <int PDT>
__global__ void __launch_bounds__(TILE_THREADS) k_recover(const __grid_constant__ StepArgs a) {
    if (__ldcg(&a.result->applied)) return;
    const bool sw = a.chain && __ldcg(&a.chain->cur) != 0;     // the set the step read (not yet flipped)
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    for (int si = 0; si < a.n_shards; ++si) {
        const ShardDev& d = a.shards[si];
        const float* M = state_ptrs(d, sw).mi;
        for (int64_t i = (int64_t)blockIdx.x * TILE_THREADS + threadIdx.x; i < d.numel;
             i += (int64_t)gridDim.x * TILE_THREADS)
            P[d.param_off + i] = (uint16_t)Half16<PDT>::narrow(M[i]);
    }
}

// ---------------------------------------------------------------- K1b / K4: reduce + statistics
template <int GDT, int VEC, int NS>
__global__ void __launch_bounds__(TILE_THREADS)
k_reduce(const __grid_constant__ StepArgs a) {
    constexpr int64_t TILE = (int64_t)TILE_THREADS * VEC;
    pdl_wait();
    pdl_launch_next();
    SumSq sumsq;
    int ovf = 0;
    int si = 0;
    for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
        si = find_shard(a, tile, si);
        const ShardDev& d = a.shards[si];
        const int64_t it = tile - d.tile_begin;
        if (it == 0 && threadIdx.x < d.head && threadIdx.x < d.numel)
            reduce_elem<GDT>(a, d, threadIdx.x, sumsq, ovf);              // the shard's unaligned head
        const int64_t j = d.head + it * TILE + (int64_t)threadIdx.x * VEC;
        if (j >= d.numel) continue;
        uint16_t* G = static_cast<uint16_t*>(d.gshard);
        if (VEC == 8 && j + 8 <= d.numel) {
            float s[8];
            reduce8<GDT, NS>(a, d.grad_off + j, s);
            uint32_t h[8];
            float af[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                h[e] = average16n<GDT, NS>(s[e], a.divisor);
                ovf |= Half16<GDT>::nonfinite(h[e]);
                af[e] = Half16<GDT>::widen(h[e]);
            }
            sumsq.add8(af);
            store8(G, j, h);
        } else {
            const int64_t end = (VEC == 8) ? d.numel : j + 1;
            for (int64_t i = j; i < end; ++i) reduce_elem<GDT>(a, d, i, sumsq, ovf);
        }
    }
    double acc = sumsq.total();
    block_reduce(acc, ovf);
    if (!publish_partial(a, acc, ovf)) return;
    double sum;
    int flag;
    combine_partials(a, sum, flag);
    if (threadIdx.x == 0) {
        zero_stats st = a.accumulate ? *a.stats : zero_stats{0.0, 0, 0};
        st.sumsq += sum;
        st.overflow |= flag;
        *a.stats = st;
    }
}

// ---------------------------------------------------------------- K1c: apply
// One thread's 8-element vector of a tile: where it lies (when the tile holds
// a whole vector for this thread) and its loaded operands.
struct ApplyLoc {
    const ShardDev* d;
    int64_t j;
    bool full;
};

struct ApplyVec {
    float4 t0, t1, m0, m1, v0, v1;
    uint4 w;
};

// This thread's part of a tile: the scalar elements (the shard's unaligned
// head, a ragged tail) are done here; returns where its whole vector lies.
// si: the shard of this block's previous tile (updated).
template <int GDT, int PDT>
__device__ __forceinline__ ApplyLoc apply_locate(const StepArgs& a, int64_t tile, float k, const Ctl& c, int& si) {
    constexpr int64_t TILE = (int64_t)TILE_THREADS * 8;
    ApplyLoc L{nullptr, 0, false};
    if (tile >= a.n_tiles) return L;
    si = find_shard(a, tile, si);
    const ShardDev& d = a.shards[si];
    const int64_t it = tile - d.tile_begin;
    if (it == 0 && threadIdx.x < d.head && threadIdx.x < d.numel)
        apply_elem<GDT, PDT>(a, d, threadIdx.x, k, c);                       // the shard's unaligned head
    const int64_t j = d.head + it * TILE + (int64_t)threadIdx.x * 8;
    if (j >= d.numel) return L;
    if (j + 8 <= d.numel) return ApplyLoc{&d, j, true};
    for (int64_t i = j; i < d.numel; ++i) apply_elem<GDT, PDT>(a, d, i, k, c);
    return L;
}

template <bool WIDE>
__device__ __forceinline__ void apply_load(const ApplyLoc& L, bool sw, ApplyVec& x) {
    const StatePtrs p = state_ptrs(*L.d, sw);
    ld_state8<WIDE>(p.mi + L.j, x.t0, x.t1);
    ld_state8<WIDE>(p.mmi + L.j, x.m0, x.m1);
    ld_state8<WIDE>(p.vi + L.j, x.v0, x.v1);
    x.w = ld_stream(static_cast<const uint16_t*>(L.d->gshard) + L.j);
}

template <int GDT, int PDT, bool WIDE>
__device__ __forceinline__ void apply_finish(const StepArgs& a, const ApplyLoc& L, const ApplyVec& x, float k,
                                             const Ctl& c, uint16_t* P) {
    const StatePtrs p = state_ptrs(*L.d, c.sw);
    const int64_t j = L.j;
    const uint32_t u[4] = {x.w.x, x.w.y, x.w.z, x.w.w};
    float th[8] = {x.t0.x, x.t0.y, x.t0.z, x.t0.w, x.t1.x, x.t1.y, x.t1.z, x.t1.w};
    float mm[8] = {x.m0.x, x.m0.y, x.m0.z, x.m0.w, x.m1.x, x.m1.y, x.m1.z, x.m1.w};
    float vv[8] = {x.v0.x, x.v0.y, x.v0.z, x.v0.w, x.v1.x, x.v1.y, x.v1.z, x.v1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t h = (e & 1) ? (u[e >> 1] >> 16) : (u[e >> 1] & 0xFFFFu);
        adamw1(th[e], mm[e], vv[e], Half16<GDT>::widen(h), k, a.sc, c.ss, c.rb2);
    }
    uint32_t hp[8];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const uint32_t w = Half16<PDT>::narrow2(th[e], th[e + 1]);
        hp[e] = w & 0xFFFFu;
        hp[e + 1] = w >> 16;
    }
    st_state8<WIDE>(p.mo + j, th);
    st_state8<WIDE>(p.mmo + j, mm);
    st_state8<WIDE>(p.vo + j, vv);
    store8(P, L.d->param_off + j, hp);
}

// Every block derives the same skip / clip decision from the statistics.
// (Issuing the next tile's loads before updating and storing the current
// one measured 2.5% slower on one shard and no faster on eight.)
// WIDE: 256-bit state accesses (every shard's state arrays 32-byte aligned).
template <int GDT, int PDT, int VEC, bool WIDE = false>
__global__ void __launch_bounds__(TILE_THREADS)
k_apply(const __grid_constant__ StepArgs a) {
    const zero_stats st = *a.stats;
    const int overflow = (st.overflow | a.extra_overflow) ? 1 : 0;
    const double sumsq = st.sumsq + a.extra_sumsq;
    double norm, clip;
    const Ctl c = step_ctl(a);
    const float k = grad_multiplier(sumsq, step_S(a), a.max_norm, norm, clip);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        zero_result r;
        r.overflow = overflow;
        r.status = c.bad ? ZERO_ELIMIT : 0;
        r.applied = (overflow || c.bad) ? 0 : 1;
        r.path = 2;
        r.sumsq = sumsq;
        r.grad_norm = norm;
        r.clip_coef = clip;
        r.grad_mult = k;
        r.reserved = 0.0f;
        *a.result = r;
    }
    if (overflow || c.bad) return;
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    int si = 0;
    if (VEC != 8) {                                                          // one element at a time
        for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
            si = find_shard(a, tile, si);
            const ShardDev& d = a.shards[si];
            const int64_t i = (tile - d.tile_begin) * TILE_THREADS + threadIdx.x;
            if (i < d.numel) apply_elem<GDT, PDT>(a, d, i, k, c);
        }
        return;
    }
    for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
        const ApplyLoc L = apply_locate<GDT, PDT>(a, tile, k, c, si);
        if (!L.full) continue;
        ApplyVec x;
        apply_load<WIDE>(L, c.sw, x);
        apply_finish<GDT, PDT, WIDE>(a, L, x, k, c, P);
    }
}

// ---------------------------------------------------------------- K3: ZeRO-3 layer gather
// out[dst_off[p] + j] = src[p][j] for j < len[p]: the per-layer all-gather
// (equal parts, one per rank) and the owner broadcast (the pieces of the
// owners' contiguous segments a layer spans) are both this copy.
struct GatherArgs {
    const void* src[ZERO_MAX_SLICES];
    int64_t len[ZERO_MAX_SLICES];              // elements of each segment
    int64_t dst_off[ZERO_MAX_SLICES];          // where each segment starts in out
    int64_t tile_begin[ZERO_MAX_SLICES + 1];   // first tile of each segment; [n] = tile count
    int n;
    void* out;
};

// Each thread moves GATHER_UNROLL vectors per tile, all loads issued before
// the first store, so that a block keeps GATHER_UNROLL * 256 vectors in flight.
constexpr int GATHER_UNROLL = 8;

template <int VEC>
__global__ void __launch_bounds__(TILE_THREADS) k_gather(const __grid_constant__ GatherArgs a) {
    constexpr int U = VEC == 8 ? GATHER_UNROLL : 2;
    constexpr int64_t TILE = (int64_t)TILE_THREADS * VEC * U;
    pdl_wait();
    pdl_launch_next();
    const int64_t n_tiles = a.tile_begin[a.n];
    uint16_t* O = static_cast<uint16_t*>(a.out);
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        int p = 0;
        while (p + 1 < a.n && a.tile_begin[p + 1] <= tile) ++p;
        const int64_t t = tile - a.tile_begin[p];
        const int64_t L = a.len[p];
        const uint16_t* src = static_cast<const uint16_t*>(a.src[p]);
        uint16_t* dst = O + a.dst_off[p];
        const int64_t j0 = t * TILE + (int64_t)threadIdx.x * VEC;
        if (VEC == 8) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = j0 + (int64_t)u * TILE_THREADS * VEC;
                if (j + 8 <= L) w[u] = ld_stream(src + j);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = j0 + (int64_t)u * TILE_THREADS * VEC;
                if (j + 8 <= L) __stcs(reinterpret_cast<uint4*>(dst + j), w[u]);
                else for (int64_t i = j; i < L; ++i) dst[i] = src[i];
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = j0 + (int64_t)u * TILE_THREADS;
                if (j < L) dst[j] = src[j];
            }
        }
    }
}

}  // namespace zdp
