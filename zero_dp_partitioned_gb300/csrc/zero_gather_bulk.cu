// zero_gather_bulk.cu -- the ZeRO-3 gather moved by the TMA unit, on as many
// CTAs as the caller allows.
//
// A unit's parameters are rebuilt in one layer buffer from its pieces (each
// rank's part, or the pieces of the owners' segments) before the unit's
// forward and again before its backward.  In a pipelined schedule the gather
// of the next unit runs while the current unit computes.  On one GPU both
// want the SMs: the register-staged gather (k_gather) fills every SM with
// warps that each keep a few 16-byte loads in flight, and a tensor-core
// consumer launched beside it waits for SMs; the two barely overlap.  Here
// the copy is issued by one thread per CTA as bulk asynchronous copies
// (cp.async.bulk: global -> shared memory -> global), so a few CTAs keep a
// deep pipeline of bytes in flight with almost no issue slots, and the caller
// bounds the CTA count, leaving the other SMs to the consumer.
//
// Pieces: every piece's source and its destination slot must agree modulo
// 16 bytes (the bulk copies need 16-byte aligned addresses and sizes).  A
// piece's bytes before its first 16-byte boundary and after its last one
// (fewer than 16 each) are copied with plain byte stores by the other lanes
// of CTA 0; the aligned middle is cut into chunks of `chunk` bytes, dealt to
// the CTAs round-robin.
//
// Pipeline of one CTA (thread 0): loads of the first `stages` chunks are
// issued at once, one mbarrier per stage; for each chunk in turn: wait for its
// load, issue its bulk store from the same stage, and reload the stage the
// previous chunk used once `cp.async.bulk.wait_group.read 1` says that
// chunk's store has read it.  Every wait is bounded: a CTA whose wait runs out
// records it in *status (bit 0), waits (bounded again) for the loads it still
// has in flight and for its stores, and stops.
#include <cuda_runtime.h>

#include "zero_internal.h"
#include "zero_tma.cuh"

namespace zdp {

constexpr int BULK_HEADER = 256;           // S <= 8 mbarriers, then S destinations, then S sizes
constexpr int BULK_MAX_STAGES = 8;

__global__ void __launch_bounds__(32, 1) k_gather_bulk(const __grid_constant__ BulkGatherArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    if (threadIdx.x != 0) {
        pdl_wait();         // see the programmatic dependent launch note in zero_kernels.cuh
        pdl_launch_next();
        // CTA 0's other lanes: the unaligned bytes at both ends of every piece
        if (blockIdx.x == 0) {
            for (int p = threadIdx.x - 1; p < a.n; p += 31) {
                const uint8_t* s = a.src[p];
                uint8_t* d = a.out + a.dst_off[p];
                for (int64_t i = 0; i < a.head[p]; ++i) d[i] = s[i];
                for (int64_t i = a.head[p] + a.mid[p]; i < a.bytes[p]; ++i) d[i] = s[i];
            }
        }
        return;
    }
    const int S = a.stages;
    const int64_t G = gridDim.x;
    const int64_t total = a.chunk_begin[a.n];
    const int64_t n = total > blockIdx.x ? (total - blockIdx.x + G - 1) / G : 0;
    if (n == 0) return;
    const uint32_t bars = smem_addr(smem);
    const uint32_t base = bars + BULK_HEADER;
    uint8_t** stage_dst = reinterpret_cast<uint8_t**>(smem + 8 * BULK_MAX_STAGES);
    uint32_t* stage_bytes = reinterpret_cast<uint32_t*>(smem + 16 * BULK_MAX_STAGES);
    for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
    // Set-up above touches only this CTA's shared memory, so it overlaps the
    // previous kernel's tail; global memory is touched only after the wait.
    pdl_wait();
    pdl_launch_next();

    // Load cursor: the piece holding the next chunk to load, kept in registers
    // (this CTA's chunks only move forward through the pieces).
    int p = 0;
    int64_t p_begin = a.chunk_begin[0], p_end = a.chunk_begin[1], p_mid = a.mid[0];
    const uint8_t* p_src = a.src[0] + a.head[0];
    uint8_t* p_dst = a.out + a.dst_off[0] + a.head[0];
    auto issue = [&](int64_t c, int st) {
        while (c >= p_end) {
            ++p;
            p_begin = p_end;
            p_end = a.chunk_begin[p + 1];
            p_mid = a.mid[p];
            p_src = a.src[p] + a.head[p];
            p_dst = a.out + a.dst_off[p] + a.head[p];
        }
        const int64_t off = (c - p_begin) * a.chunk;
        const int64_t rem = p_mid - off;
        const uint32_t b = (uint32_t)(rem < a.chunk ? rem : a.chunk);
        stage_dst[st] = p_dst + off;
        stage_bytes[st] = b;
        mbar_expect_tx(bars + 8 * st, b);
        bulk_load(base + (uint32_t)st * (uint32_t)a.chunk, p_src + off, b, bars + 8 * st);
    };

    int64_t next_load = 0;              // this CTA's chunks [0, next_load) have had their loads issued
    for (; next_load < n && next_load < S; ++next_load) issue(blockIdx.x + next_load * G, (int)next_load);
    bool ok = true;
    int st = 0, prev_st = 0;
    uint32_t phase = 0;
    int64_t k = 0;
    for (; k < n; ++k) {
        if (!mbar_wait(bars + 8 * st, phase, a.spin_limit)) {
            ok = false;
            break;
        }
        bulk_store(stage_dst[st], base + (uint32_t)st * (uint32_t)a.chunk, stage_bytes[st]);
        bulk_commit();
        if (k >= 1 && next_load < n) {
            // next_load == k - 1 + S: it takes the stage of chunk k - 1 once that chunk's store has read it
            bulk_wait_read<1>();
            issue(blockIdx.x + next_load * G, prev_st);
            ++next_load;
        }
        prev_st = st;
        if (++st == S) {
            st = 0;
            phase ^= 1u;
        }
    }
    if (!ok) {
        for (int64_t c = k; c < next_load; ++c)
            mbar_wait(bars + 8 * (int)(c % S), (uint32_t)((c / S) & 1), a.drain_limit);
        atomicOr(a.status, 1);
    }
    bulk_wait_all();
}

size_t gather_bulk_smem(int chunk, int stages) { return BULK_HEADER + (size_t)stages * chunk; }

int launch_gather_bulk(const BulkGatherArgs& a, int grid, cudaStream_t s) {
    const size_t smem = gather_bulk_smem(a.chunk, a.stages);
    int rc = cuda_fail(cudaFuncSetAttribute(k_gather_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                       "bulk gather shared-memory size");
    if (rc != ZERO_OK) return rc;
    void* args[] = {const_cast<BulkGatherArgs*>(&a)};
    return cuda_fail(launch_after_previous((const void*)k_gather_bulk, grid, 32, args, smem, s),
                     "bulk gather launch");
}

}  // namespace zdp
