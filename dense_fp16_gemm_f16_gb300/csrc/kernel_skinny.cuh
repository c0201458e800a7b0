// kernel_skinny.cuh -- small-M GEMM (M <= 64): D^T = B * A^T over column
// ranges of B, each range's K loop split over the CTAs of one cluster.
//
// With M this small a 128-row MMA over M would be mostly padding, and the run
// time is set by reading B (the N x K weights) once from HBM: the "small batch
// leaves memory bandwidth unused" situation of the GEMM blog post (section
// 5.4).  So the operands swap roles: each MMA is tcgen05.mma M=128 (up to 128
// rows of B, i.e. output columns) x N=MN (the M rows of A, padded to 16/32/64
// by TMA zero fill) x K=16 (32 for 8-bit operands), both operands K-major as
// stored.  The accumulator in TMEM is D^T: TMEM lane = output column n, TMEM
// column = output row m.
//
// Work split.  N is cut into R ranges of `width` (<= 128) columns, so that
// every SM streams about the same number of B bytes.  A range belongs to one
// cluster of P CTAs, and CTA j of the cluster runs the j-th of P pieces of the
// K loop over the range's B rows (a B box of `width` rows; the MMA's other
// rows read whatever the slot holds and their TMEM lanes are never used).
// The P fp32 partials of a range meet in distributed shared memory: CTA j
// finishes output rows [j MN/P, (j+1) MN/P), every CTA stores each row's
// partial into the receive buffer of the CTA that finishes it, a cluster
// barrier (release / acquire) makes the stores visible, and each CTA adds the
// P partials of its rows in ascending piece order -- a fixed order, so the
// result is bitwise reproducible -- applies the fused transform, rounds to D's
// type and writes D.  Nothing goes through global memory but A, B and D, and
// no CTA waits on another cluster, so the grid needs no co-residency beyond
// the cluster's own.  With P = 1 a CTA may own several ranges, one after the
// other, with the accumulator double-buffered in TMEM so a range's epilogue
// overlaps the next range's loads and MMAs.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "config.h"
#include "epilogue.cuh"
#include "ptx.cuh"
#include "wait.cuh"

namespace gemm_gb300 {

// The output block held in TMEM at `taddr` (this warp's lanes): the sum of
// its ACCS accumulators, added in ascending order.
template <int MN, int ACCS>
__device__ __forceinline__ void skinny_acc_sum(uint32_t taddr, uint32_t (&v)[MN]) {
    ptx::tmem_ld_cols<MN>(taddr, v);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int a = 1; a < ACCS; ++a) {
        uint32_t w[MN];
        ptx::tmem_ld_cols<MN>(taddr + static_cast<uint32_t>(a * MN), w);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < MN; ++m) v[m] = __float_as_uint(__uint_as_float(v[m]) + __uint_as_float(w[m]));
    }
}

// T is the element type of D (and C, bias); F8 selects 8-bit operands.
template <class Cfg, class T, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const SkinnyParams p) {
    constexpr int MN = Cfg::MN;
    constexpr int MAXS = Cfg::MAX_STAGES;
    constexpr int kStageK = stage_k(F8 ? 1 : 2);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const uint32_t sbase = ptx::smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (MAXS + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * MAXS + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * MAXS + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * MAXS + 4);
    const uint32_t slot = sbase + Cfg::OFF_SLOT;
    // ring of this launch: `stages` stages of KA K blocks each; a stage's B
    // slots (w_stride bytes per K block) first, the A slots after all of them
    const int STAGES = p.stages;
    const int KA = p.stage_atoms;
    auto w_slot = [&](int s, int a) { return sbase + static_cast<uint32_t>((s * KA + a) * p.w_stride); };
    auto x_slot = [&](int s, int a) {
        return sbase + static_cast<uint32_t>(STAGES * KA * p.w_stride + (s * KA + a) * Cfg::X_BYTES);
    };
    // K pieces per range = CTAs per cluster (the same for the whole grid)
    const int P = p.pieces;
    const bool clustered = P > 1;

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
    // in a cluster, this also guarantees every CTA of it is running before any
    // of them stores into another's shared memory
    if (clustered) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_SLOT);

    const int j = clustered ? static_cast<int>(ptx::cluster_ctarank()) : 0;   // this CTA's K piece
    const int64_t cid = blockIdx.x / P;            // cluster index
    const int64_t C = gridDim.x / P;               // clusters in the grid
    const int kb0 = static_cast<int>(div_nonneg(static_cast<int64_t>(j) * p.k_blocks, P));
    const int kb1 = static_cast<int>(div_nonneg(static_cast<int64_t>(j + 1) * p.k_blocks, P));
    // While the previous kernel in the stream finishes, start pulling the B
    // blocks of this CTA's first ring fill into L2 (a prefetch cannot expose
    // stale data, so it may run before the dependency wait below).
    if (warp == 0 && lane == 0 && cid < p.ranges) {
        const int n_pre = (kb1 - kb0) < p.prefetch_blocks ? (kb1 - kb0) : p.prefetch_blocks;
        for (int i = 0; i < n_pre; ++i)
            ptx::tma_prefetch_2d(&tmW, (kb0 + i) * kStageK, static_cast<int32_t>(cid * p.width));
    }
    // Everything above touched only this CTA's shared memory and TMEM (and
    // L2 by prefetch), so it overlaps the previous kernel's tail; global memory
    // is read and written only below.  (Every kernel here takes more than half
    // of an SM's shared memory, so a CTA of this grid never shares an SM, or
    // its TMEM, with one of the last.)
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // (whole warp; one elected lane issues the arrivals and copies)
        bool ok = true;
        int stage = 0;
        uint32_t phase = 0;
        // B streams past (evict first when it cannot stay in L2); A is re-read
        // by every range and stays
        const uint64_t pol_w = p.stream_b ? ptx::policy_evict_first() : ptx::policy_evict_normal();
        const uint64_t pol_x = ptx::policy_evict_last();
        const uint32_t stage_bytes = static_cast<uint32_t>(p.width) * kStageRowBytes + Cfg::X_BYTES;
        for (int64_t r = cid; ok && r < p.ranges; r += C) {
            const int32_t y = static_cast<int32_t>(r * p.width);
            for (int kb = kb0; kb < kb1; kb += KA) {
                const int na = (kb1 - kb) < KA ? (kb1 - kb) : KA;
                if (!wait_phase_warp(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerEmpty, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(full_bar(stage), static_cast<uint32_t>(na) * stage_bytes);
                    for (int a = 0; a < na; ++a) {
                        ptx::tma_load_2d_hint(w_slot(stage, a), &tmW, full_bar(stage), (kb + a) * kStageK, y, pol_w);
                        ptx::tma_load_2d_hint(x_slot(stage, a), &tmX, full_bar(stage), (kb + a) * kStageK, 0, pol_x);
                    }
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        // do not leave while an MMA commit may still arrive on this CTA's barriers
        for (int i = 0; ok && i < STAGES; ++i) {
            ok = wait_phase_warp(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerTail, p.timeout_ns);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (clustered) ptx::cluster_sync();   // meets the epilogue's exchange barrier
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        // (whole warp; one elected lane issues every tcgen05 instruction)
        bool ok = true;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t it = 0;
        const uint32_t idesc = ptx::instr_desc(128, MN, p.ab_format);
        for (int64_t r = cid; ok && r < p.ranges; r += C, ++it) {
            const uint32_t buf = it & 1u;
            const uint32_t use = (it >> 1) & 1u;
            if (!wait_phase_warp(tempty_bar(buf), use ^ 1u, p.status, kSiteMmaTmemEmpty, p.timeout_ns)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * Cfg::ACC_COLS;
            for (int kb = kb0; kb < kb1; kb += KA) {
                const int na = (kb1 - kb) < KA ? (kb1 - kb) : KA;
                if (!wait_phase_warp(full_bar(stage), phase, p.status, kSiteMmaFull, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                    for (int a = 0; a < na; ++a) {
                        const uint64_t w_desc = ptx::sw128_kmajor_desc(w_slot(stage, a));
                        const uint64_t x_desc = ptx::sw128_kmajor_desc(x_slot(stage, a));
#pragma unroll
                        for (int k = 0; k < kMmaPerStage; ++k)
                            ptx::mma<1, F8>(d_tmem + static_cast<uint32_t>((k % Cfg::ACCS) * MN), w_desc + 2u * k,
                                            x_desc + 2u * k, idesc,
                                            (kb != kb0 || a != 0 || k >= Cfg::ACCS) ? 1u : 0u);
                    }
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
        wait_phase_warp(drain_bar, 0, p.status, kSiteMmaDrain, p.timeout_ns);
        if (clustered) ptx::cluster_sync();   // meets the epilogue's exchange barrier
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int n_local = q * 32 + lane;   // TMEM lane = column within the range
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        T* D = static_cast<T*>(p.D);
        if (!clustered) {
            // one whole K loop per range: straight from TMEM to D
            uint32_t it = 0;
            for (int64_t r = cid; r < p.ranges; r += C, ++it) {
                const uint32_t buf = it & 1u;
                const uint32_t use = (it >> 1) & 1u;
                const int64_t n = r * p.width + n_local;
                const bool col_in = n_local < p.width && n < p.N;
                // this column's C values, factor and bias, fetched while the K loop runs
                EpiColumn<T, MN> ec;
                if (p.epi.on && col_in) ec.load(p.epi, n, p.M, p.N);
                if (!wait_phase_warp(tfull_bar(buf), use, p.status, kSiteEpilogueTmemFull, p.timeout_ns)) break;
                ptx::tc_fence_after();
                uint32_t v[MN];
                skinny_acc_sum<MN, Cfg::ACCS>(t_lane + buf * Cfg::ACC_COLS, v);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(tempty_bar(buf));
                if (col_in) {
                    if (p.epi.on) {
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
            }
        } else {
            // One range per cluster (the planner launches exactly R clusters).
            // Every thread reaches the exchange barrier, whatever happened before.
            const int64_t r = cid;
            const int64_t n = r * p.width + n_local;
            const bool col_in = r < p.ranges && n_local < p.width && n < p.N;
            // this column's factor alpha * s[n] and bias, fetched while the K loop runs
            EpiColumnFactors<T> cf;
            if (p.epi.on && col_in) cf.load(p.epi, n);
            const bool ready = r < p.ranges &&
                               wait_phase_warp(tfull_bar(0), 0, p.status, kSiteEpilogueTmemFull, p.timeout_ns);
            uint32_t v[MN];
            if (ready) {
                ptx::tc_fence_after();
                skinny_acc_sum<MN, Cfg::ACCS>(t_lane, v);
            } else {
#pragma unroll
                for (int m = 0; m < MN; ++m) v[m] = 0u;
            }
            // CTA d finishes rows [d MS, (d+1) MS) (MS = MN / P, P a power of two).
            // Its receive buffer is [P pieces][128 columns][MS rows] fp32: a
            // column's rows bound for one CTA are contiguous, so they travel as
            // 16-byte stores (8-byte when MS = 2), a quarter of the remote
            // transactions of one store per value.
            const int ms_shift = (__ffs(MN) - 1) - (__ffs(P) - 1);
            const int MS = 1 << ms_shift;
            const uint32_t recv = sbase + Cfg::OFF_RECV;
            const uint32_t mine = recv + static_cast<uint32_t>((j * 128 + n_local) * MS * 4);
            if (MS >= 4) {
#pragma unroll
                for (int m = 0; m < MN; m += 4) {
                    const int d = m >> ms_shift;
                    const uint32_t off = static_cast<uint32_t>((m - (d << ms_shift)) * 4);
                    ptx::st_cluster_v4(ptx::mapa(mine + off, static_cast<uint32_t>(d)), v[m], v[m + 1], v[m + 2], v[m + 3]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < MN; m += 2) {
                    const int d = m >> ms_shift;
                    const uint32_t off = static_cast<uint32_t>((m - (d << ms_shift)) * 4);
                    ptx::st_cluster_v2(ptx::mapa(mine + off, static_cast<uint32_t>(d)), v[m], v[m + 1]);
                }
            }
            ptx::cluster_sync();   // exchange barrier: every partial of this CTA's rows is in
            if (ready && col_in) {
                // this column's rows [j MS, (j+1) MS), the P partials added in
                // ascending piece order
                const uint32_t col = recv + static_cast<uint32_t>(n_local * MS * 4);
                const uint32_t piece_bytes = static_cast<uint32_t>(128 * MS * 4);
                auto finish = [&](int ml, float acc) {
                    const int m = j * MS + ml;
                    if (m < p.M) {
                        const float x = p.epi.on ? cf.apply(p.epi, acc, m, n, p.N) : acc;
                        D[m * static_cast<int64_t>(p.N) + n] = Elem<T>::from_float(x);
                    }
                };
                if (MS >= 4) {
                    for (int c = 0; c < MS; c += 4) {
                        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        for (int i = 0; i < P; ++i) {
                            float t[4];
                            ptx::ld_shared_v4(col + i * piece_bytes + static_cast<uint32_t>(c * 4), t);
#pragma unroll
                            for (int r = 0; r < 4; ++r) acc[r] += t[r];
                        }
#pragma unroll
                        for (int r = 0; r < 4; ++r) finish(c + r, acc[r]);
                    }
                } else {
                    float acc[2] = {0.0f, 0.0f};
                    for (int i = 0; i < P; ++i) {
                        float t[2];
                        ptx::ld_shared_v2(col + i * piece_bytes, t);
                        acc[0] += t[0];
                        acc[1] += t[1];
                    }
                    finish(0, acc[0]);
                    finish(1, acc[1]);
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    // (no CTA reads another's shared memory after the exchange barrier, so a
    // CTA may leave while the others of its cluster still run)
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_gb300
