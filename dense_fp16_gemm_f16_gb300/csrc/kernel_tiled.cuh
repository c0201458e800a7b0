// kernel_tiled.cuh -- persistent, warp-specialised tcgen05 GEMM D = A * B^T.
//
// The data path is the Blackwell one of "Building a Tiled GEMM" (MLC),
// sections "GEMM data path" and steps 1-3: operand tiles GMEM -> SMEM
// (128-byte swizzle, 128-byte K chunks: 64 fp16/bf16 or 128 8-bit values),
// tcgen05.mma into a TMEM fp32
// accumulator that stays in place across the K loop (step 2), one output tile
// per unit of work (step 3).  Past those steps it applies the chapter's
// optimisation roadmap ("Optimisation roadmap"): TMA loads tracked by
// mbarriers, a multi-stage SMEM ring so loads overlap MMAs, a persistent tile
// loop, warp specialisation (producer / MMA / writeback), and, for CG == 2, a
// CTA pair that computes one larger MMA tile together.
//
// Roles (kThreads = 192):
//   warp 0             TMA producer: for every tile and K block, wait for a
//                      free stage, then load this CTA's A rows and B rows.
//   warp 1             allocates / frees TMEM; in the leader CTA it issues the
//                      MMAs (one thread issues, as step 1 of the chapter
//                      requires) and commits them to barriers.
//   warps 2-5          epilogue: TMEM -> registers (fused transform) -> D's
//                      type (fp16 or bf16) -> swizzled SMEM
//                      -> TMA store, clipped at the edges of D.
// Warps 0 and 1 run their loops with all 32 lanes and let one elected lane
// issue each copy, MMA and commit.  The loop's values (stage addresses,
// descriptors) are then warp-uniform, which keeps the issuing thread fast
// enough: run by a lone lane, the MMA loop took longer per stage than the
// tensor pipe does (measured on GB300: the pipe idled 11 % of its cycles,
// against under 4 % this way).
// The accumulator is double-buffered in TMEM, so the epilogue of one tile
// runs while the MMAs of the next tile are issued.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "config.h"
#include "epilogue.cuh"
#include "ptx.cuh"
#include "wait.cuh"

namespace gemm_gb300 {

// ---------------------------------------------------------------- split K
// With p.ksplit = S > 1 a cluster of S * CG CTAs works on one tile: MMA group
// j (a CTA pair, or one CTA) runs the j-th of S pieces of the tile's K loop,
// and the S fp32 partials are summed in distributed shared memory.  Group j
// finishes the j-th slice of the tile's columns (the BN / 8 groups of 8
// columns dealt out evenly), for the rows its CTAs hold: every CTA stores
// each column's partial into the receive buffer of the CTA of the same rank
// in the group that finishes it, the cluster meets at a barrier, and each CTA
// adds the S partials of its slice in ascending piece order -- a fixed order,
// so the result does not depend on timing -- then applies the fused transform
// and writes D.  The receive buffer takes the operand ring's space (the ring
// is idle once every MMA of the cluster has finished, which the first of two
// cluster barriers establishes).  No CTA waits on another cluster, so the
// clusters need not be resident together.

// First 8-column group of column slice j of a tile of kGroups groups.
__device__ __forceinline__ int split_group_begin(int j, int k_groups, int S) { return j * k_groups / S; }
// The slice that holds 8-column group g.
__device__ __forceinline__ int split_slice_of(int g, int k_groups, int S) { return ((g + 1) * S - 1) / k_groups; }

// Receive buffer layout: [S pieces][slice_quads][128 rows][4] fp32, where
// slice_quads = 2 * ceil(k_groups / S) column quads: a thread (one row) moves
// four consecutive columns with one 16-byte access, and consecutive rows are
// consecutive 16-byte words (no bank conflicts on either side).
__device__ __forceinline__ uint32_t split_recv_offset(int piece, int quad, int row, int slice_quads) {
    return static_cast<uint32_t>(((piece * slice_quads + quad) * 128 + row) * 16);
}

// Exchange: this CTA (group `piece`, pair rank `rank`) sends every 8-column
// group of its partial (TMEM lane = row) to the CTA of the same rank in the
// group that finishes the group's slice.  `ready` = the accumulator is valid
// (else zeros are sent, so every receiver still gets every word it waits for).
template <class Cfg>
__device__ __forceinline__ void split_k_send(uint32_t recv_base, uint32_t t_row, bool ready, int piece, uint32_t rank,
                                             int row, int S) {
    constexpr int kGroups = Cfg::BN / 8;
    const int slice_quads = 2 * ((kGroups + S - 1) / S);
#pragma unroll 1
    for (int c = 0; c < Cfg::BN / 64; ++c) {
        uint32_t v[64];
        if (ready) {
            ptx::tmem_ld_x32(t_row + c * 64, v);
            ptx::tmem_ld_x32(t_row + c * 64 + 32, v + 32);
            ptx::tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = 0u;
        }
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
            const int g = c * 8 + g8;
            const int dest = split_slice_of(g, kGroups, S);
            const int quad = 2 * (g - split_group_begin(dest, kGroups, S));
            const uint32_t dest_cta = static_cast<uint32_t>(dest * Cfg::CG) + rank;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t addr = ptx::mapa(recv_base + split_recv_offset(piece, quad + h, row, slice_quads), dest_cta);
                ptx::st_cluster_v4(addr, v[8 * g8 + 4 * h], v[8 * g8 + 4 * h + 1], v[8 * g8 + 4 * h + 2],
                                   v[8 * g8 + 4 * h + 3]);
            }
        }
    }
}

// Sum of the S partials of this CTA's slice for row `row` (D row grow), in
// ascending piece order, with the fused transform, written to D.
template <class Cfg, class T>
__device__ __forceinline__ void split_k_reduce(const uint8_t* recv, const TiledParams& p, int piece, int row,
                                               int64_t grow, int64_t n0, int S) {
    constexpr int kGroups = Cfg::BN / 8;
    const int slice_quads = 2 * ((kGroups + S - 1) / S);
    const int g0 = split_group_begin(piece, kGroups, S);
    const int g1 = split_group_begin(piece + 1, kGroups, S);
    T* D = static_cast<T*>(p.D);
    if (grow >= p.M) return;
#pragma unroll 1
    for (int g = g0; g < g1; ++g) {
        const int64_t gcol = n0 + 8 * g;
        if (gcol >= p.N) break;                       // N % 8 == 0: groups are all in or all out
        const uint4 cv = p.epi.on ? epi_load_c8<T>(p.epi, grow, gcol, p.M, p.N) : make_uint4(0u, 0u, 0u, 0u);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        const int quad = 2 * (g - g0);
#pragma unroll 1
        for (int i = 0; i < S; ++i) {
            const float4 lo = *reinterpret_cast<const float4*>(recv + split_recv_offset(i, quad, row, slice_quads));
            const float4 hi = *reinterpret_cast<const float4*>(recv + split_recv_offset(i, quad + 1, row, slice_quads));
            acc[0] += lo.x; acc[1] += lo.y; acc[2] += lo.z; acc[3] += lo.w;
            acc[4] += hi.x; acc[5] += hi.y; acc[6] += hi.z; acc[7] += hi.w;
        }
        if (p.epi.on) epi_apply8_c<T>(p.epi, acc, cv, gcol);
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = Elem<T>::pack2(acc[2 * e], acc[2 * e + 1]);
        *reinterpret_cast<uint4*>(D + grow * static_cast<int64_t>(p.N) + gcol) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// T is the element type of D (and C, bias); F8 selects 8-bit operands
// (kind::f8f6f4, 128 K elements per stage) instead of 16-bit ones of type T;
// KA = K blocks per ring stage (a compile-time constant, so the one-block
// loops compile to straight-line issue code).
template <class Cfg, class T, bool F8, int KA = 1>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
gemm_tiled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmBpiece, const __grid_constant__ CUtensorMap tmD,
                  const TiledParams p) {
    constexpr int CG = Cfg::CG;
    constexpr int CONS = Cfg::CONS;
    static_assert(split_recv_fits(Cfg::BN, Cfg::RING_BYTES, CG == 2 ? kSplitMaxPieces : kSplitMaxPieces1),
                  "the split-K receive buffer must fit the operand ring");
    constexpr int MAXS = Cfg::MAX_STAGES;
    constexpr int kStageK = stage_k(F8 ? 1 : 2);
    extern __shared__ uint8_t smem_raw[];
    // Align the working area to 1024 bytes (the 128-byte swizzle atom); every
    // CTA of a pair gets the same offsets, which the pair MMA relies on.
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const uint32_t sbase = ptx::smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // A cluster is one MMA group (a CTA pair, or one CTA), or with split K
    // (p.ksplit = S > 1) S groups on the same tile.  rank = this CTA's rank in
    // its pair; piece = its group in the cluster (the K piece with split K);
    // leader = cluster rank of the group's first CTA, which issues the MMAs
    // (they commit to barriers in both CTAs of a pair).
    const bool split = p.ksplit > 1;
    const int csize = CG * (split ? p.ksplit : 1);
    const uint32_t crank = (csize > 1) ? ptx::cluster_ctarank() : 0u;
    const uint32_t rank = crank % CG;
    const int piece = static_cast<int>(crank / CG);
    const uint32_t leader = static_cast<uint32_t>(piece * CG);
    const uint16_t pair_mask = static_cast<uint16_t>(((1u << CG) - 1u) << leader);

    const uint32_t bar0 = sbase + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (MAXS + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * MAXS + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * MAXS + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * MAXS + 4);
    // ring geometry of this launch (the same in every role and both CTAs of a pair)
    // ring of this launch: slots of `stride` bytes (one K block of A and B),
    // grouped into STAGES stages of KA consecutive slots
    const uint32_t stride = static_cast<uint32_t>(ring_stride(p, Cfg::A_BYTES, Cfg::B_BYTES));
    const int STAGES = static_cast<int>(Cfg::RING_BYTES / stride) / KA;
    auto slot_addr = [&](int s, int a) { return sbase + static_cast<uint32_t>(s * KA + a) * stride; };
    const uint32_t slot = sbase + Cfg::OFF_SLOT;

    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmBpiece);
        ptx::prefetch_tensormap(&tmD);
        for (int s = 0; s < MAXS; ++s) {
            ptx::mbar_init(full_bar(s), 1);   // the leader's expect_tx arrival + TMA bytes
            ptx::mbar_init(empty_bar(s), 1);   // one MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);                 // one MMA commit
            ptx::mbar_init(tempty_bar(b), Cfg::EPI_WARPS * CG);   // every epilogue warp of the pair
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_SLOT);
    // Everything above touched only this CTA's shared memory and TMEM, so it
    // overlaps the previous kernel's tail; global memory is used only below.
    // (Every kernel here takes more than half of an SM's shared memory, so a
    // CTA of this grid never shares an SM, or its TMEM, with one of the last.)
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();

    const int64_t cluster_idx = blockIdx.x / csize;
    const int64_t num_clusters = gridDim.x / csize;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop, so its values stay warp-uniform; one
        // elected lane issues the barrier arrivals and copies.
        {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t round = 0;
            for (int64_t u = cluster_idx; ok && u < p.num_units; u += num_clusters, ++round) {
                int64_t tm, n0;
                int nw, kb0, kb1;
                work_unit(u, p, Cfg::BN, piece, tm, n0, nw, kb0, kb1);
                // Odd rounds walk K downwards: a round starts on the K blocks the
                // previous round (on the same tile rows) read last, which are the
                // ones still in L2.  Only the load order changes (the MMA takes
                // stages as they come); split-K pieces keep one direction.
                const bool reverse = (round & 1u) && p.ksplit == 1;
                // each CTA of a pair supplies nw / CG rows of B to the MMA; a
                // column piece of a tail tile loads only those rows (box of the
                // second B map) instead of the whole tile's
                // A rows of consumer h: tile row tm * BM + h * MMA_M + rank * 128
                const int32_t a_row = static_cast<int32_t>(tm * Cfg::BM + rank * 128);
                const int32_t b_row = static_cast<int32_t>(n0 + rank * (nw / CG));
                const bool piece = nw < Cfg::BN;
                const CUtensorMap* b_map = piece ? &tmBpiece : &tmB;
                const uint32_t stage_bytes = Cfg::A_BYTES + (piece ? Cfg::B_BYTES / p.split : Cfg::B_BYTES);
                for (int kb = kb0; kb < kb1; kb += KA) {
                    const int na = (KA == 1 || kb1 - kb >= KA) ? KA : kb1 - kb;
                    if (!wait_phase_warp(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerEmpty,
                                         p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (ptx::elect_one()) {
                        // Both CTAs' bytes of a pair complete on the leader's full
                        // barrier; the leader announces the pair's total.
                        const uint32_t bar = CG == 1 ? full_bar(stage) : ptx::mapa(full_bar(stage), leader);
                        if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(stage), CG * na * stage_bytes);
#pragma unroll
                        for (int a = 0; a < KA; ++a) {
                            if (a >= na) break;
                            const uint32_t a_dst = slot_addr(stage, a);
                            const uint32_t b_dst = a_dst + Cfg::A_BYTES;
                            const int kx = (reverse ? (kb1 - 1 - (kb + a - kb0)) : kb + a) * kStageK;
                            if constexpr (CG == 1) {
#pragma unroll
                                for (int h = 0; h < CONS; ++h)
                                    ptx::tma_load_2d(a_dst + h * Cfg::A_HALF_BYTES, &tmA, bar, kx,
                                                     a_row + h * Cfg::MMA_M);
                                ptx::tma_load_2d(b_dst, b_map, bar, kx, b_row);
                            } else {
#pragma unroll
                                for (int h = 0; h < CONS; ++h)
                                    ptx::tma_load_2d_pair(a_dst + h * Cfg::A_HALF_BYTES, &tmA, bar, kx,
                                                          a_row + h * Cfg::MMA_M);
                                ptx::tma_load_2d_pair(b_dst, b_map, bar, kx, b_row);
                            }
                        }
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Do not leave while an MMA commit may still arrive on this CTA's
            // barriers: wait until the MMA has released every stage.
            for (int i = 0; ok && i < STAGES; ++i) {
                ok = wait_phase_warp(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerTail, p.timeout_ns);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (split) {   // the epilogue's two exchange barriers
            ptx::cluster_sync();
            ptx::cluster_sync();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        // The whole warp runs the loop, so every value it computes is
        // warp-uniform; one elected lane (always the same one: the warp is
        // converged) issues each tcgen05 instruction.
        if (rank == 0) {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t it = 0;
            for (int64_t u = cluster_idx; ok && u < p.num_units; u += num_clusters, ++it) {
                int64_t tm, n0;
                int nw, kb0, kb1;
                work_unit(u, p, Cfg::BN, piece, tm, n0, nw, kb0, kb1);
                const uint32_t idesc = ptx::instr_desc(Cfg::MMA_M, nw, p.ab_format);
                // accumulator buffer (two per consumer, alternating) and its use count
                const uint32_t buf = Cfg::ACC_BUFS == 2 ? (it & 1u) : 0u;
                const uint32_t use = Cfg::ACC_BUFS == 2 ? ((it >> 1) & 1u) : (it & 1u);
                if (!wait_phase_warp(tempty_bar(buf), use ^ 1u, p.status, kSiteMmaTmemEmpty, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * CONS * Cfg::BN;   // consumer h adds h * BN
                // the producer's K order for this unit (odd rounds walk K downwards)
                const bool reverse = (it & 1u) && p.ksplit == 1;
                for (int kb = kb0; kb < kb1; kb += KA) {
                    const int na = (KA == 1 || kb1 - kb >= KA) ? KA : kb1 - kb;
                    if (!wait_phase_warp(full_bar(stage), phase, p.status, kSiteMmaFull, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (ptx::elect_one()) {
#pragma unroll
                        for (int a = 0; a < KA; ++a) {
                            if (a >= na) break;
                            const uint64_t a_desc = ptx::sw128_kmajor_desc(slot_addr(stage, a));
                            const uint64_t b_desc = ptx::sw128_kmajor_desc(slot_addr(stage, a) + Cfg::A_BYTES);
                            // the last K block holds only p.last_k_steps 32-byte steps of
                            // real data (the rest is TMA zero fill): skip the MMAs of the others
                            const int blk = reverse ? (kb1 - 1 - (kb + a - kb0)) : kb + a;
                            const int steps = (blk == p.k_blocks - 1) ? p.last_k_steps : kMmaPerStage;
                            const bool first = kb == kb0 && a == 0;
                            // each consumer's MMAs read its own 128 rows of A and the shared B
#pragma unroll
                            for (int h = 0; h < CONS; ++h)
#pragma unroll
                                for (int k = 0; k < kMmaPerStage; ++k)   // 32 bytes of K each
                                    if (k < steps)
                                        ptx::mma<CG, F8>(d_tmem + h * Cfg::BN,
                                                         a_desc + h * (Cfg::A_HALF_BYTES >> 4) + 2u * k,
                                                         b_desc + 2u * k, idesc, (!first || k != 0) ? 1u : 0u);
                        }
                        if constexpr (CG == 1) ptx::mma_commit(empty_bar(stage));
                        else ptx::mma_commit_pair(empty_bar(stage), pair_mask);
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (ptx::elect_one()) {
                    if constexpr (CG == 1) ptx::mma_commit(tfull_bar(buf));
                    else ptx::mma_commit_pair(tfull_bar(buf), pair_mask);
                }
                __syncwarp();
            }
            if (ptx::elect_one()) {
                if constexpr (CG == 1) ptx::mma_commit(drain_bar);
                else ptx::mma_commit_pair(drain_bar, static_cast<uint16_t>(1u << leader));
            }
            __syncwarp();
            wait_phase_warp(drain_bar, 0, p.status, kSiteMmaDrain, p.timeout_ns);
        }
        if (split) {   // the epilogue's two exchange barriers
            ptx::cluster_sync();
            ptx::cluster_sync();
        }
    } else if (split) {
        // ------------------------------------------------------------ epilogue, split K
        // One tile per cluster (the planner launches exactly one cluster per
        // tile).  Every thread reaches both barriers, whatever happened before.
        const int q = warp & 3;
        const int row = q * 32 + lane;    // this CTA's accumulator row (TMEM lane)
        const int64_t u = cluster_idx;
        int64_t tm = 0, n0 = 0;
        int nw = 0, kb0 = 0, kb1 = 0;
        if (u < p.num_units) work_unit(u, p, Cfg::BN, piece, tm, n0, nw, kb0, kb1);
        const bool ready = u < p.num_units &&
                           wait_phase_warp(tfull_bar(0), 0, p.status, kSiteEpilogueTmemFull, p.timeout_ns);
        if (ready) ptx::tc_fence_after();
        // A: every MMA of the cluster is done, so every operand ring is free
        ptx::cluster_sync();
        split_k_send<Cfg>(sbase, tmem_base + (static_cast<uint32_t>(q * 32) << 16), ready, piece, rank, row,
                          p.ksplit);
        // B: every partial of this CTA's slice is in its receive buffer
        ptx::cluster_sync();
        if (ready) split_k_reduce<Cfg, T>(smem, p, piece, row, tm * Cfg::BM + rank * 128 + row, n0, p.ksplit);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;    // TMEM lanes 32q .. 32q+31 are readable by this warp
        const int ew = warp - 2;   // owner of staging buffers 2ew, 2ew+1
        const int h = ew / kEpiWarps;   // the consumer (accumulator) this warp drains
        const uint32_t tempty_leader0 = (CG == 2) ? ptx::mapa(tempty_bar(0), leader) : tempty_bar(0);
        // which parts of the fused transform run (warp-uniform, for the whole launch)
        const bool epi_c = p.epi.on && p.epi.C != nullptr && p.epi.beta != 0.0f;
        // only the column factors alpha * s[n] (the 8-bit dequantisation): a loop without branches
        const bool epi_scale_only = p.epi.on && !epi_c && p.epi.bias == nullptr && p.epi.act == 0;
        uint8_t* cols_area = smem + Cfg::OFF_COLS + ew * Cfg::COLS_BYTES;
        uint32_t it = 0;
        int ebuf = 0;
        for (int64_t u = cluster_idx; u < p.num_units; u += num_clusters, ++it) {
            int64_t tm, n0;
            int nw, kb0, kb1;
            work_unit(u, p, Cfg::BN, piece, tm, n0, nw, kb0, kb1);
            const int chunks = nw / Cfg::EPI_COLS;
            const uint32_t buf = Cfg::ACC_BUFS == 2 ? (it & 1u) : 0u;
            const uint32_t use = Cfg::ACC_BUFS == 2 ? ((it >> 1) & 1u) : (it & 1u);
            // the per-column scales and bias of the whole unit, fetched before its
            // accumulator is waited for (ev[0] always holds the current chunk's)
            constexpr int kChunks = Cfg::BN / Cfg::EPI_COLS;
            EpiCols64<T> ev[kChunks];
            if (p.epi.on) {
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    if (c < chunks) ev[c].load(p.epi, n0 + c * Cfg::EPI_COLS, lane, p.N);
            }
            if (!wait_phase_warp(tfull_bar(buf), use, p.status, kSiteEpilogueTmemFull, p.timeout_ns)) break;
            ptx::tc_fence_after();
            const int64_t row0 = tm * Cfg::BM + h * Cfg::MMA_M + rank * 128 + q * 32;  // D row of lane 0
            const bool rows_in = row0 < p.M;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + (buf * CONS + h) * Cfg::BN;
#pragma unroll 1
            for (int c = 0; c < chunks; ++c) {
                const int64_t col0 = n0 + c * Cfg::EPI_COLS;
                const bool store = rows_in && col0 < p.N;  // warp-uniform
                // this chunk's C values, in flight while TMEM is read
                uint4 cv[8] = {};
                if (epi_c) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        cv[j] = (store && col0 + 8 * j < p.N) ? epi_load_c8<T>(p.epi, row0 + lane, col0 + 8 * j, p.M, p.N)
                                                             : make_uint4(0u, 0u, 0u, 0u);
                }
                uint32_t v[64];
                ptx::tmem_ld_x32(t_row + c * 64, v);
                ptx::tmem_ld_x32(t_row + c * 64 + 32, v + 32);
                ptx::tmem_wait_ld();
                if (c == chunks - 1) {
                    // this warp has read its part of the buffer: return it to the MMA
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (CG == 2) ptx::mbar_arrive_cluster(tempty_leader0 + 8u * buf);
                        else ptx::mbar_arrive(tempty_bar(buf));
                    }
                }
                // the TMA store issued two chunks ago from this buffer has read it
                if (lane == 0) ptx::bulk_wait_group_read<1>();
                __syncwarp();
                uint8_t* sb = smem + Cfg::OFF_EPI + (ew * 2 + ebuf) * Cfg::EPI_BUF_BYTES;
                if (store) {
                    // row `lane` of the box, 16-byte chunk j at position j ^ (row % 8):
                    // the layout the 128-byte-swizzled tensor map expects
                    uint8_t* row_ptr = sb + lane * (Cfg::EPI_COLS * 2);
                    if (p.epi.on) {
                        ev[0].stage(cols_area, lane);
                        __syncwarp();
                    }
                    if (epi_scale_only) {
                        const float4* f4 = reinterpret_cast<const float4*>(cols_area);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 s0 = f4[2 * j], s1 = f4[2 * j + 1];
                            const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                            uint32_t h[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                h[e] = Elem<T>::pack2(__uint_as_float(v[8 * j + 2 * e]) * sc[2 * e],
                                                      __uint_as_float(v[8 * j + 2 * e + 1]) * sc[2 * e + 1]);
                            *reinterpret_cast<uint4*>(row_ptr + ((j ^ (lane & 7)) << 4)) =
                                make_uint4(h[0], h[1], h[2], h[3]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float x[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[8 * j + e]);
                            if (p.epi.on && col0 + 8 * j < p.N) epi_apply8_s<T>(p.epi, x, cv[j], epi_c, cols_area, j);
                            uint32_t h[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) h[e] = Elem<T>::pack2(x[2 * e], x[2 * e + 1]);
                            *reinterpret_cast<uint4*>(row_ptr + ((j ^ (lane & 7)) << 4)) =
                                make_uint4(h[0], h[1], h[2], h[3]);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    if (store)
                        ptx::tma_store_2d(&tmD, ptx::smem_u32(sb), static_cast<int32_t>(col0),
                                          static_cast<int32_t>(row0));
                    ptx::bulk_commit_group();
                }
                ebuf ^= 1;
#pragma unroll
                for (int i = 0; i + 1 < kChunks; ++i) ev[i] = ev[i + 1];
            }
        }
        if (lane == 0) ptx::bulk_wait_group<0>();
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_gb300
