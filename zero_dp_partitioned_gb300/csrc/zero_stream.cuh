// zero_stream.cuh -- TMA-pipelined versions of the two write-heavy passes
// (the fused single pass for up to 8 gradient slices, and the apply pass),
// with one block-wide cycle per chunk; opt-in (ZERO_GB300_PATH=stream).  The
// producer/consumer passes in zero_ws.cu split the same work between a
// producer lane and consumer warps without that cycle.  This file also holds
// the PTX wrappers (mbarrier, bulk copies) the TMA kernels share.
//
// Why it was built: register-staged kernels bound the bytes they keep in
// flight, and with them the HBM bandwidth they reach, by their registers;
// seven 128-bit stores per thread per 8 elements also fill the store queue.
// (Measured since: a chunk's block-wide cycle costs more than the copies
// save -- 14.1 ms for the GPT-2 step -- and the register pass with every load
// of a vector in flight reaches the copy bandwidth.)  Here each array's
// chunk is moved by one bulk asynchronous copy (cp.async.bulk, executed by
// the TMA unit) into a ring of shared-memory stages tracked by mbarriers, and
// the results leave by bulk stores from a double-buffered output stage.
//
// Pipeline of one block (256 threads, chunks of CHUNK elements of one shard,
// chunk j of this block = global chunk blockIdx.x + j * gridDim.x):
//   thread 0 keeps S-1 chunks of loads in flight ahead of the chunk being
//   computed; every thread waits on the chunk's mbarrier, reads its 4 elements
//   from shared memory, computes, writes 4 results into the output stage;
//   a block barrier; thread 0 issues the bulk stores of the output stage.
//   An output stage is rewritten only after `cp.async.bulk.wait_group.read 1`
//   says the stores issued from it two chunks earlier have read it.
//
// Bulk copies need 16-byte aligned addresses and sizes that are multiples of
// 16 bytes: each chunk's bulk part is its length rounded down to 8 elements;
// the last few elements of a shard (fewer than 8) are read and written with
// plain loads and stores.  16-bit parameters whose shard offset is not a
// multiple of 8 elements are stored directly from registers.
//
// Every mbarrier wait is bounded (SPIN_LIMIT tries).  On a timeout the block
// records the timeout bit in its flags word, waits (bounded again) for the
// loads it still has in flight, and goes on to publish its partial so that the
// result is always written; the step is then reported as not applied.
#pragma once

#include "zero_kernels.cuh"

namespace zdp {

constexpr int CHUNK = 1024;                     // elements per chunk (4 per thread)
constexpr int MAX_STREAM_SLICES = 8;
constexpr unsigned SPIN_LIMIT = 1u << 22;
constexpr int FLAG_OVERFLOW = 1, FLAG_TIMEOUT = 2;

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// One bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned limit) {
    for (unsigned it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- shared-memory layout
// [0, 64): S full barriers (8 bytes each, S <= 8)
// then S input stages of `in_bytes`, then 2 output stages of `out_bytes`.
struct StreamLayout {
    int stages;
    uint32_t in_bytes, out_bytes;
    uint32_t grad_off, state_off;     // inside an input stage: grads first, then master|m|v
};

__host__ __device__ inline StreamLayout stream_layout(int n_grad_arrays, int stages) {
    StreamLayout L;
    L.stages = stages;
    L.grad_off = 0;
    L.state_off = (uint32_t)n_grad_arrays * CHUNK * 2;
    L.in_bytes = L.state_off + 3u * CHUNK * 4;
    L.out_bytes = 3u * CHUNK * 4 + CHUNK * 2;   // master | m | v | param
    return L;
}

__host__ __device__ inline size_t stream_smem_bytes(const StreamLayout& L) {
    return 64 + (size_t)L.stages * L.in_bytes + 2 * (size_t)L.out_bytes;
}

struct StreamArgs {
    StepArgs a;
    int stages;
    unsigned spin_limit;        // tries per wait (SPIN_LIMIT in production)
    unsigned drain_limit;       // tries per wait when draining after a timeout
    int param_bulk;             // 1 when every shard's parameter slot allows bulk stores
};

// Element e of a chunk of shard d starting at c0: where the chunk's bulk part ends.
__device__ __forceinline__ int64_t chunk_len(const ShardDev& d, int64_t c0) {
    const int64_t rem = d.numel - c0;
    return rem < CHUNK ? rem : CHUNK;
}

// Issue the bulk loads of one chunk into stage `st`.  FUSED: n slices of
// gradients; otherwise the shard's 16-bit reduced gradient.
template <bool FUSED>
__device__ __forceinline__ void issue_chunk(const StepArgs& a, const StreamLayout& L, uint8_t* smem, int st,
                                            int64_t chunk) {
    const int si = find_shard(a, chunk);
    const ShardDev& d = a.shards[si];
    const int64_t c0 = (chunk - d.tile_begin) * CHUNK;
    const int64_t len = chunk_len(d, c0);
    const uint32_t blen = (uint32_t)(len & ~int64_t(7));
    const uint32_t bar = smem_addr(smem) + 8u * st;
    uint8_t* stage = smem + 64 + (size_t)st * L.in_bytes;
    const int ng = FUSED ? a.n_slices : 1;
    mbar_expect_tx(bar, blen * (2u * ng + 12u));
    if (blen == 0) return;
    for (int r = 0; r < ng; ++r) {
        const uint16_t* src = FUSED ? static_cast<const uint16_t*>(a.slices[r]) + d.grad_off + c0
                                    : static_cast<const uint16_t*>(d.gshard) + c0;
        bulk_load(smem_addr(stage + L.grad_off + (size_t)r * CHUNK * 2), src, blen * 2u, bar);
    }
    const float* st_src[3] = {d.mi, d.mmi, d.vi};
    for (int q = 0; q < 3; ++q)
        bulk_load(smem_addr(stage + L.state_off + (size_t)q * CHUNK * 4), st_src[q] + c0, blen * 4u, bar);
}

// Store 4 16-bit values at dst + q with the widest stores the address allows.
__device__ __forceinline__ void store4(uint16_t* dst, int64_t q, const uint32_t (&h)[4]) {
    const int mis = (int)(reinterpret_cast<uintptr_t>(dst + q) & 7u);
    if (mis == 0) {
        *reinterpret_cast<uint2*>(dst + q) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    } else if ((mis & 3) == 0) {
        reinterpret_cast<unsigned*>(dst + q)[0] = h[0] | (h[1] << 16);
        reinterpret_cast<unsigned*>(dst + q + 2)[0] = h[2] | (h[3] << 16);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[q + e] = (uint16_t)h[e];
    }
}

// The streamed pass.  FUSED: reduce n slices (<= 8), statistics, AdamW with
// multiplier a.k, store, and (last block) the result -- as k_step_fused.
// Otherwise: AdamW from the reduced gradient shard with the decision taken
// from the statistics -- as k_apply.  Either way every block publishes its
// flags (and, fused, its partial sum of squares) and the last block to finish
// writes the result, so a timeout anywhere is reported.
template <int GDT, int PDT, bool FUSED>
__global__ void __launch_bounds__(TILE_THREADS) k_stream(const __grid_constant__ StreamArgs sa) {
    extern __shared__ __align__(128) uint8_t smem[];
    const StepArgs& a = sa.a;
    const StreamLayout L = stream_layout(FUSED ? a.n_slices : 1, sa.stages);
    const int S = L.stages;
    const int tid = threadIdx.x;

    // fused: the multiplier is given; apply: every block derives the same decision
    float k = a.k;
    int overflow_in = 0;
    double st_sumsq = 0.0, norm = 0.0, clip = 1.0;
    if (!FUSED) {
        const zero_stats st = *a.stats;
        overflow_in = (st.overflow | a.extra_overflow) ? 1 : 0;
        st_sumsq = st.sumsq + a.extra_sumsq;
        k = grad_multiplier(st_sumsq, a.loss_scale, a.max_norm, norm, clip);
    }

    SumSq sumsq;
    int flags = 0;
    uint16_t* P = static_cast<uint16_t*>(a.flat_param);
    const int64_t n_local = a.n_tiles > (int64_t)blockIdx.x ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (!overflow_in && n_local > 0) {
        if (tid == 0) {
            for (int s = 0; s < S; ++s) mbar_init(smem_addr(smem) + 8u * s, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0)
            for (int64_t j = 0; j < S - 1 && j < n_local; ++j)
                issue_chunk<FUSED>(a, L, smem, (int)j, blockIdx.x + j * gridDim.x);

        int64_t j = 0;
        for (; j < n_local; ++j) {
            const int st = (int)(j % S);
            const int64_t chunk = blockIdx.x + j * gridDim.x;
            if (tid == 0 && j + S - 1 < n_local)
                issue_chunk<FUSED>(a, L, smem, (int)((j + S - 1) % S), blockIdx.x + (j + S - 1) * gridDim.x);
            const bool ok = mbar_wait(smem_addr(smem) + 8u * st, (uint32_t)((j / S) & 1), sa.spin_limit);
            if (tid == 0) bulk_wait_read<1>();       // the output stage written two chunks ago has been read
            if (!__syncthreads_and(ok ? 1 : 0)) {
                flags |= FLAG_TIMEOUT;
                break;
            }
            const int si = find_shard(a, chunk);
            const ShardDev& d = a.shards[si];
            const int64_t c0 = (chunk - d.tile_begin) * CHUNK;
            const int64_t len = chunk_len(d, c0);
            const int64_t blen = len & ~int64_t(7);
            const uint8_t* in = smem + 64 + (size_t)st * L.in_bytes;
            uint8_t* out = smem + 64 + (size_t)S * L.in_bytes + (size_t)(j & 1) * L.out_bytes;
            const int e0 = 4 * tid;
            if (e0 + 4 <= blen) {
                uint32_t h4[4];
                if (FUSED) {
                    float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    for (int r = 0; r < a.n_slices; ++r) {
                        const uint2 w =
                            *reinterpret_cast<const uint2*>(in + L.grad_off + (size_t)r * CHUNK * 2 + e0 * 2);
                        s4[0] = __fadd_rn(s4[0], Half16<GDT>::widen(w.x & 0xFFFFu));
                        s4[1] = __fadd_rn(s4[1], Half16<GDT>::widen(w.x >> 16));
                        s4[2] = __fadd_rn(s4[2], Half16<GDT>::widen(w.y & 0xFFFFu));
                        s4[3] = __fadd_rn(s4[3], Half16<GDT>::widen(w.y >> 16));
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) h4[e] = average16<GDT>(s4[e], a.divisor);
                } else {
                    const uint2 w = *reinterpret_cast<const uint2*>(in + L.grad_off + e0 * 2);
                    h4[0] = w.x & 0xFFFFu;
                    h4[1] = w.x >> 16;
                    h4[2] = w.y & 0xFFFFu;
                    h4[3] = w.y >> 16;
                }
                const float4 t = *reinterpret_cast<const float4*>(in + L.state_off + e0 * 4);
                const float4 m = *reinterpret_cast<const float4*>(in + L.state_off + CHUNK * 4 + e0 * 4);
                const float4 v = *reinterpret_cast<const float4*>(in + L.state_off + 2 * CHUNK * 4 + e0 * 4);
                float th[4] = {t.x, t.y, t.z, t.w}, mm[4] = {m.x, m.y, m.z, m.w}, vv[4] = {v.x, v.y, v.z, v.w};
                float af[4];
                uint32_t hp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (FUSED && Half16<GDT>::nonfinite(h4[e])) flags |= FLAG_OVERFLOW;
                    af[e] = Half16<GDT>::widen(h4[e]);
                    adamw1(th[e], mm[e], vv[e], af[e], k, a.sc);
                    hp[e] = Half16<PDT>::narrow(th[e]);
                }
                if (FUSED) sumsq.add4(af);
                *reinterpret_cast<float4*>(out + e0 * 4) = make_float4(th[0], th[1], th[2], th[3]);
                *reinterpret_cast<float4*>(out + CHUNK * 4 + e0 * 4) = make_float4(mm[0], mm[1], mm[2], mm[3]);
                *reinterpret_cast<float4*>(out + 2 * CHUNK * 4 + e0 * 4) = make_float4(vv[0], vv[1], vv[2], vv[3]);
                if (sa.param_bulk)
                    *reinterpret_cast<uint2*>(out + 3 * CHUNK * 4 + e0 * 2) =
                        make_uint2(hp[0] | (hp[1] << 16), hp[2] | (hp[3] << 16));
                else
                    store4(P, d.param_off + c0 + e0, hp);
            } else if (e0 < len) {
                // the shard's last (fewer than 8) elements: plain loads and stores
                const int64_t end = (e0 + 4 < len) ? e0 + 4 : len;
                for (int64_t e = (e0 > blen ? e0 : blen); e < end; ++e) {
                    const int64_t i = c0 + e;
                    uint32_t h;
                    if (FUSED) {
                        h = average16<GDT>(reduce1<GDT>(a, d.grad_off + i), a.divisor);
                        if (Half16<GDT>::nonfinite(h)) flags |= FLAG_OVERFLOW;
                    } else {
                        h = static_cast<const uint16_t*>(d.gshard)[i];
                    }
                    const float af = Half16<GDT>::widen(h);
                    if (FUSED) sumsq.add_fp64(af);
                    float th = d.mi[i], mm = d.mmi[i], vv = d.vi[i];
                    adamw1(th, mm, vv, af, k, a.sc);
                    d.mo[i] = th;
                    d.mmo[i] = mm;
                    d.vo[i] = vv;
                    P[d.param_off + i] = (uint16_t)Half16<PDT>::narrow(th);
                }
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {
                if (blen > 0) {
                    const uint32_t ob = smem_addr(out);
                    bulk_store(d.mo + c0, ob, (uint32_t)blen * 4u);
                    bulk_store(d.mmo + c0, ob + CHUNK * 4, (uint32_t)blen * 4u);
                    bulk_store(d.vo + c0, ob + 2 * CHUNK * 4, (uint32_t)blen * 4u);
                    if (sa.param_bulk) bulk_store(P + d.param_off + c0, ob + 3 * CHUNK * 4, (uint32_t)blen * 2u);
                }
                bulk_commit();
            }
        }
        if ((flags & FLAG_TIMEOUT) && tid == 0) {
            // loads of chunks j .. j+S-1 may still be in flight: a bounded wait for each
            for (int64_t q = j; q < n_local && q <= j + S - 1; ++q)
                mbar_wait(smem_addr(smem) + 8u * (int)(q % S), (uint32_t)((q / S) & 1), sa.drain_limit);
        }
        if (tid == 0) bulk_wait_all();
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
            r.grad_norm = sqrt(r.sumsq) / a.loss_scale;
            r.clip_coef = 1.0;
            r.grad_mult = a.k;
        } else {
            r.overflow = overflow_in;
            r.sumsq = st_sumsq;
            r.grad_norm = norm;
            r.clip_coef = clip;
            r.grad_mult = k;
        }
        r.status = (flag & FLAG_TIMEOUT) ? ZERO_ETIMEOUT : 0;
        r.applied = (r.overflow || r.status) ? 0 : 1;
        r.path = FUSED ? 3 : 4;
        r.reserved = 0.0f;
        *a.result = r;
    }
}

}  // namespace zdp
