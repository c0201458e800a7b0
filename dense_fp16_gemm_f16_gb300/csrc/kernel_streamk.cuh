// kernel_streamk.cuh -- small-M GEMM (M <= 64): D^T = B * A^T with split K.
//
// With M this small a 128-row MMA over M would be mostly padding and the
// run time is set by reading B (the N x K weights) once from HBM -- the
// "small batch leaves memory bandwidth unused" situation of the GEMM blog
// post (section 5.4).  So the operands swap roles: each MMA is
// tcgen05.mma M=128 (128 rows of B, i.e. 128 output columns) x N=MN (the M
// rows of A, padded to 16/32/64 by TMA zero fill) x K=16 (32 for 8-bit
// operands), both operands
// K-major exactly as stored.  The accumulator tile in TMEM is D^T: TMEM lane
// = output column n, TMEM column = output row m.
//
// Work split: the (n-tile, k-block) units are laid out tile-major and cut into
// G contiguous ranges, one per CTA (G = number of SMs), so every SM streams
// the same number of B bytes.  A tile whose K loop lies inside one CTA's range
// is written straight to D.  A tile cut across CTAs gets one fp32 partial per
// CTA in a workspace; the CTA that finishes last (per-tile counter) adds the
// partials in ascending CTA order -- a fixed order, so results are bitwise
// reproducible -- applies the fused transform if any, rounds to D's type
// (fp16, or bf16), writes D and re-arms the counter.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "config.h"
#include "epilogue.cuh"
#include "ptx.cuh"
#include "wait.cuh"

namespace gemm_gb300 {

// T is the element type of D (and C, bias); F8 selects 8-bit operands.
template <class Cfg, class T, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
gemm_streamk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const StreamKParams p) {
    constexpr int MN = Cfg::MN;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const uint32_t sbase = ptx::smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t slot = sbase + Cfg::OFF_SLOT;
    volatile uint32_t* last_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_SLOT + 4);

    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmW);
        ptx::prefetch_tensormap(&tmX);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), kEpiWarps);
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc<1>(slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish<1>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_SLOT);
    // Everything above touched only this CTA's shared memory and TMEM, so it
    // overlaps the previous kernel's tail; global memory is used only below.
    // (Every kernel here takes more than half of an SM's shared memory, so a
    // CTA of this grid never shares an SM, or its TMEM, with one of the last.)
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();

    constexpr int kStageK = stage_k(F8 ? 1 : 2);
    const uint32_t idesc = ptx::instr_desc(128, MN, p.ab_format);
    const int64_t G = p.num_ctas;
    const int64_t W = p.units;
    const int64_t KB = p.k_blocks;
    const int64_t c = blockIdx.x;
    const int64_t u0 = unit_begin(c, W, G);
    const int64_t u1 = unit_begin(c + 1, W, G);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // (whole warp; one elected lane issues, as in the tiled kernel)
        {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            // B streams past (evict first when it cannot stay in L2); A is
            // re-read by every CTA and stays
            const uint64_t pol_w = p.stream_b ? ptx::policy_evict_first() : ptx::policy_evict_normal();
            const uint64_t pol_x = ptx::policy_evict_last();
            for (int64_t u = u0; u < u1; ++u) {
                const int64_t t = div_nonneg(u, KB);
                const int32_t kx = static_cast<int32_t>((u - t * KB) * kStageK);
                if (!wait_phase_warp(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerEmpty, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(full_bar(stage), Cfg::STAGE_BYTES);
                    ptx::tma_load_2d_hint(sbase + Cfg::OFF_W + stage * Cfg::W_BYTES, &tmW, full_bar(stage), kx,
                                          static_cast<int32_t>(t * 128), pol_w);
                    ptx::tma_load_2d_hint(sbase + Cfg::OFF_X + stage * Cfg::X_BYTES, &tmX, full_bar(stage), kx, 0, pol_x);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            for (int i = 0; ok && i < STAGES; ++i) {
                ok = wait_phase_warp(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerTail, p.timeout_ns);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        // (whole warp; one elected lane issues every tcgen05 instruction)
        {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t seg = 0;
            for (int64_t u = u0; ok && u < u1; ++seg) {
                const int64_t t = div_nonneg(u, KB);
                const int64_t seg_end = (t + 1) * KB < u1 ? (t + 1) * KB : u1;
                const uint32_t buf = seg & 1u;
                const uint32_t use = (seg >> 1) & 1u;
                if (!wait_phase_warp(tempty_bar(buf), use ^ 1u, p.status, kSiteMmaTmemEmpty, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * MN;
                for (const int64_t seg_start = u; u < seg_end; ++u) {
                    if (!wait_phase_warp(full_bar(stage), phase, p.status, kSiteMmaFull, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t w_desc = ptx::sw128_kmajor_desc(sbase + Cfg::OFF_W + stage * Cfg::W_BYTES);
                    const uint64_t x_desc = ptx::sw128_kmajor_desc(sbase + Cfg::OFF_X + stage * Cfg::X_BYTES);
                    if (ptx::elect_one()) {
#pragma unroll
                        for (int k = 0; k < kMmaPerStage; ++k)
                            ptx::mma<1, F8>(d_tmem, w_desc + 2u * k, x_desc + 2u * k, idesc,
                                            (u != seg_start || k != 0) ? 1u : 0u);
                        ptx::mma_commit(empty_bar(stage));
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (ptx::elect_one()) ptx::mma_commit(tfull_bar(buf));
                __syncwarp();
            }
            if (ptx::elect_one()) ptx::mma_commit(drain_bar);
            __syncwarp();
            wait_phase(drain_bar, 0, p.status, kSiteMmaDrain, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int r = q * 32 + lane;                     // row of the 128-row tile = output column
        const int etid = threadIdx.x - 64;               // 0..127 among the epilogue threads
        T* D = static_cast<T*>(p.D);
        const int64_t first_tile = div_nonneg(u0, KB);
        uint32_t seg = 0;
        for (int64_t u = u0; u < u1; ++seg) {
            const int64_t t = div_nonneg(u, KB);
            const int64_t seg_end = (t + 1) * KB < u1 ? (t + 1) * KB : u1;
            const uint32_t buf = seg & 1u;
            const uint32_t use = (seg >> 1) & 1u;
            // all four epilogue warps take the same decision: they meet at
            // named barriers below
            const bool ready = wait_phase(tfull_bar(buf), use, p.status, kSiteEpilogueTmemFull, p.timeout_ns);
            if (!ptx::named_bar_and(1, 32 * kEpiWarps, ready)) break;
            ptx::tc_fence_after();
            uint32_t v[MN];
            ptx::tmem_ld_cols<MN>(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * MN, v);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(buf));

            const int64_t n = t * 128 + r;
            const int64_t c_first = cta_of_unit(t * KB, W, G);
            const int64_t c_last = cta_of_unit(t * KB + KB - 1, W, G);
            if (c_first == c_last) {
                // the whole K loop of this tile ran here
                if (n < p.N) {
                    if (p.epi.on) {
                        EpiColumn<T, MN> ec;
                        ec.load(p.epi, n, p.M, p.N);
#pragma unroll
                        for (int m = 0; m < MN; ++m)
                            if (m < p.M)
                                D[m * static_cast<int64_t>(p.N) + n] =
                                    Elem<T>::from_float(ec.apply(p.epi, __uint_as_float(v[m]), m));
                    } else {
#pragma unroll
                        for (int m = 0; m < MN; ++m)
                            if (m < p.M) D[m * static_cast<int64_t>(p.N) + n] = Elem<T>::from_float(__uint_as_float(v[m]));
                    }
                }
            } else {
                // The piece holding k = 0 ends the range of the CTA before the
                // tile's other pieces, so it usually finishes last.  Its owner
                // checks first: if every other piece is already in, it adds them
                // to its own values directly (no write and re-read of its own
                // partial).  Otherwise -- and always for the other pieces -- the
                // piece is published and the last to arrive sums the tile.
                const bool owner = (c == c_first);
                if (owner && etid == 0) {
                    const uint32_t done = ptx::ld_acquire_gpu(p.counters + t);
                    *last_flag = (done == static_cast<uint32_t>(c_last - c_first)) ? 2u : 0u;
                }
                if (owner) ptx::named_bar_sync(1, 32 * kEpiWarps);
                if (!(owner && *last_flag == 2u)) {
                    // a piece's partial is [MN / 4][128 rows][4] fp32: a thread (row r)
                    // moves four consecutive columns with one 16-byte access, and the
                    // 32 lanes of a warp cover one contiguous 512-byte run
                    float4* mine = reinterpret_cast<float4*>(
                                       p.partials + ((c * p.max_tiles_per_cta + (t - first_tile)) * MN) * 128) + r;
                    const uint64_t pol_keep = ptx::policy_evict_last();   // read back soon by the reducer
#pragma unroll
                    for (int q = 0; q < MN / 4; ++q)
                        ptx::st_global_hint_v4(mine + q * 128,
                                               make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])),
                                               pol_keep);
                    ptx::named_bar_sync(1, 32 * kEpiWarps);
                    if (etid == 0) {
                        const uint32_t prev = ptx::atom_add_acq_rel_gpu(p.counters + t, 1u);
                        *last_flag = (prev == static_cast<uint32_t>(c_last - c_first)) ? 1u : 0u;
                    }
                    ptx::named_bar_sync(1, 32 * kEpiWarps);
                }
                if (*last_flag) {
                    const bool self_in_regs = (*last_flag == 2u);
                    if (n < p.N) {
                        EpiColumn<T, MN> ec;
                        if (p.epi.on) ec.load(p.epi, n, p.M, p.N);   // in flight during the sum
                        // Sum the pieces in ascending CTA order.  Pieces are fetched
                        // CH at a time, every 16-byte load of a batch issued before
                        // any of them is used, so their latencies overlap; the
                        // additions keep the fixed order.
                        constexpr int CH = 64 / MN;
                        float acc[MN];
#pragma unroll
                        for (int m = 0; m < MN; ++m) acc[m] = 0.0f;
                        for (int64_t c0 = c_first; c0 <= c_last; c0 += CH) {
                            float4 pv[CH][MN / 4];
#pragma unroll
                            for (int i = 0; i < CH; ++i) {
                                const int64_t cc = c0 + i;
                                const bool load = cc <= c_last && !(self_in_regs && cc == c);
                                const int64_t j = load ? t - div_nonneg(unit_begin(cc, W, G), KB) : 0;
                                const float4* src = reinterpret_cast<const float4*>(
                                                        p.partials + ((cc * p.max_tiles_per_cta + j) * MN) * 128) + r;
#pragma unroll
                                for (int q = 0; q < MN / 4; ++q)
                                    pv[i][q] = load ? __ldcg(src + q * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int i = 0; i < CH; ++i) {
                                const int64_t cc = c0 + i;
                                if (cc > c_last) continue;
                                if (self_in_regs && cc == c) {   // own piece, still in registers
#pragma unroll
                                    for (int m = 0; m < MN; ++m) acc[m] += __uint_as_float(v[m]);
                                } else {
#pragma unroll
                                    for (int q = 0; q < MN / 4; ++q) {
                                        acc[4 * q] += pv[i][q].x;
                                        acc[4 * q + 1] += pv[i][q].y;
                                        acc[4 * q + 2] += pv[i][q].z;
                                        acc[4 * q + 3] += pv[i][q].w;
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int m = 0; m < MN; ++m) {
                            if (m < p.M) {
                                const float x = p.epi.on ? ec.apply(p.epi, acc[m], m) : acc[m];
                                D[m * static_cast<int64_t>(p.N) + n] = Elem<T>::from_float(x);
                            }
                        }
                    }
                    if (etid == 0) p.counters[t] = 0u;  // re-armed for the next call on this stream
                }
                ptx::named_bar_sync(1, 32 * kEpiWarps);  // last_flag is reused by the next segment
            }
            u = seg_end;
        }
    }

    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_gb300
