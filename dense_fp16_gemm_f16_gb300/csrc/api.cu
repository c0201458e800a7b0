// api.cu -- the C ABI declared in include/gemm_f16.h: argument validation,
// the host-side planner, CUtensorMap encoding, per-stream workspaces and the
// launch of the chosen kernel.  Every step of the GEMM itself runs in the
// kernels; nothing here computes on the CPU.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "config.h"
#include "epilogue.cuh"
#include "gemm_f16.h"
#include "launch.h"
#include "wait.cuh"

using namespace gemm_gb300;

namespace {

// Device status word: 0, or the first timeout any kernel recorded (see wait.cuh).
__device__ uint32_t g_status_word;
// A counter nothing ever increments (the failure-detection self-test waits on it).
__device__ uint32_t g_never_set;

// Failure-detection self-test: one thread waits, with the kernels' own bounded
// waits, on an mbarrier phase that never completes and on a counter that
// nothing increments; both give up after timeout_ns and record a timeout in
// the status word, and the kernel returns.
__global__ void selftest_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
    wait_phase(b, 0, status, kSiteSelfTest, timeout_ns);   // no arrival ever completes phase 0
    wait_count(&g_never_set, 1, status, kSiteSelfTest, timeout_ns);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    bool unsupported = false;
    int sms = 0;
    uint32_t* status = nullptr;
    int max_clusters_2cta = 0;   // co-resident 2-CTA clusters of the 256x256 kernel
    int max_clusters_2cta2c = 0; // co-resident 2-CTA clusters of the two-consumer 512x256 kernel
    int per_sm_1cta128 = 0;      // co-resident CTAs per SM
    int per_sm_1cta256 = 0;
    int skinny_clusters[kSkinnyMaxPieces + 1] = {};   // co-resident small-M clusters of P CTAs
    int split_clusters[kSplitMaxPieces + 1] = {};     // co-resident split-K clusters of S CTA pairs
    int split1_clusters[kSplitMaxPieces1 + 1] = {};   // co-resident split-K clusters of S single CTAs
};

struct Workspace {
    float* partials = nullptr;
    size_t partial_bytes = 0;
    uint32_t* counters = nullptr;
    size_t n_counters = 0;
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
std::map<std::pair<int, void*>, Workspace> g_workspaces;
EncodeTiledFn g_encode = nullptr;

constexpr int64_t kMaxDim = INT32_MAX;
// Raster groups hold as many tile rows as keep the group's A rows (tile rows x
// BM x K fp16) within this many bytes, so they stay in L2 while the group's
// B blocks stream past; the tile rows are then shared out evenly over the
// fewest groups that respect the limit.  Measured on GB300 with the K
// direction alternating per round: 11 tile rows per group at 8192^3 (1.5 %
// faster and 12 % less DRAM traffic than 8), 12 at 6144^3, all 16 at
// 4000 x 11000 x 4104.  GEMM_GROUP_M fixes the group size instead.
constexpr int64_t kL2GroupBytes = 48ll << 20;
// AUTO's choice for shapes whose 256x256 pair tiles fill less than one round
// of CTA pairs: the fastest of four plans by a small cost model, each term
// fitted to back-to-back launches on GB300 (fp16 and E4M3, K blocks of 128
// bytes; 14 mid shapes from 256x256x8192 to 2048x2048x2048):
//  - 128x256 tiles on single CTAs, cut into column pieces of width w to
//    fill the SMs (two K blocks per ring stage): kMidFixedUs + kb * t(w),
//    t(64) = 0.20, t(128) = 0.24, t(256) = 0.40 us per K block;
//  - whole 256x256 tiles on pairs (kb >= kPairMinBlocks): kMidFixedUs + 1 +
//    kb * 0.33 us;
//  - split K over a cluster of S pairs: 11.0 + ceil(kb / S) * 0.31 us;
//  - split K over a cluster of S single CTAs (S up to 8, so a larger S fits
//    one wave): 12.5 + ceil(kb / S) * 0.35 us.
// A split launch costs ~10 us more than an unsplit one (exchanging the fp32
// partials through distributed shared memory ~3 us, the cluster barriers
// ~2 us, the slice sums and D stores ~2 us, a slower ramp and teardown).
// Measured (fp16, us; unsplit 128x256 pieces / pair split / 1-CTA split):
// 1024x1024x4096 15.6 / 18.3 / 18.0; 512x2048x8192 26.6 / 24.4 / 24.1;
// 256x256x8192 25.8 / 19.3 / 17.3; 768x2048x6144 26.3 / 25.0 / 26.9;
// 128x512x16384 48.1 / 28.9 / 23.9.  Against every plan forced in turn on 20
// mid shapes, AUTO's choice was the fastest or within 2 % of it.
constexpr double kMidFixedUs = 3.0;
constexpr double kMidBlockUs64 = 0.20, kMidBlockUs128 = 0.24, kMidBlockUs256 = 0.40;
constexpr double kMidPairBlockUs = 0.33;
constexpr double kSplitPairFixedUs = 11.0, kSplitPairBlockUs = 0.31;
constexpr double kSplit1FixedUs = 12.5, kSplit1BlockUs = 0.35;
// Whole pair tiles enter the comparison only from this many K blocks on (their
// halved operand traffic per FLOP pays only in long K loops).
constexpr int64_t kPairMinBlocks = 48;
// Even when the pair tiles fill the GPU, K loops this short (each tile mostly
// epilogue) run faster on 128x256 CTAs.  Interleaved A/B on GB300: E4M3 with
// per-column scales, up to 12 K blocks, 9-12 % faster (4096x4096x1024 19.7
// against 22.0 us on pairs, 6144x6144x1536 45.5 against 50.2, 8192x8192x512
// 63.8 against 71.2); fp16 at 8 blocks 6-9 % faster (4096x8192x512 29.4
// against 32.4) but at 12 blocks 2-8 % slower (6144x6144x768 46.6 against
// 43.4), and from 16 blocks on the pairs win in both.
constexpr int64_t kShortKBlocks16 = 8;
constexpr int64_t kShortKBlocks8 = 12;
// When a row of K elements is not a whole number of 32-byte sectors, every
// other row of A and B starts 16 bytes into a sector, each 128-byte TMA row
// touches five sectors, and L2 delivery (not DRAM, not the tensor pipe)
// bounds the pair kernel (ncu at 4000 x 11000 x 4104: DRAM traffic 1.01x the
// compulsory bytes, tensor pipe idle a third of its active cycles).  The
// two-consumer kernel stages B once for 512 rows instead of 256, a quarter
// less operand traffic per FLOP, and wins there despite its single-buffered
// accumulators, given at least two rounds of its 512 x 256 tiles (GB300,
// back-to-back launches, pairs against two consumers: 4000 x 11000 x 4104
// 250-265 / 243-256 us, K = 4136 270-274 / 257-258, 6144 x 6144 x 6152 354 /
// 311; with rows on sectors the pairs win: 8192^3 533-555 / 567-578,
// 4000 x 11000 x 4112 221-230 / 253-255).

int64_t raster_group(int64_t m_tiles, int tile_m, int64_t K, int in_bytes) {
#ifdef GEMM_GROUP_M
    const int64_t g = GEMM_GROUP_M;
#else
    const int64_t g_max = kL2GroupBytes / (static_cast<int64_t>(tile_m) * K * in_bytes);
    const int64_t groups = g_max < 1 ? m_tiles : cdiv(m_tiles, g_max);
    const int64_t g = cdiv(m_tiles, groups);
#endif
    return g < 1 ? 1 : (g > m_tiles ? m_tiles : g);
}

int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// in_bytes: bytes per element of A and B (2, or 1 for 8-bit operands).  Rows
// of A, B and D must be whole 16-byte units (TMA row pitches).
gemm_status_t check_sizes(int64_t M, int64_t N, int64_t K, int in_bytes = 2) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;
    if ((K * in_bytes) % 16 != 0 || N % 8 != 0) return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

int dtype_in_bytes(int dtype) { return dtype >= GEMM_DTYPE_E4M3 ? 1 : 2; }
bool dtype_valid(int dtype) { return dtype >= GEMM_DTYPE_F16 && dtype <= GEMM_DTYPE_E5M2; }
// element type of D, C and bias: fp16 for fp16 operands, bf16 otherwise
int dtype_out(int dtype) { return dtype == GEMM_DTYPE_F16 ? GEMM_DTYPE_F16 : GEMM_DTYPE_BF16; }
// operand format field of the MMA instruction descriptor
uint32_t dtype_ab_format(int dtype) {
    return (dtype == GEMM_DTYPE_BF16 || dtype == GEMM_DTYPE_E5M2) ? 1u : 0u;
}

// ----------------------------------------------------------------- planner
struct Limits {
    int sms;
    int max_clusters_2cta;
    int max_clusters_2cta2c;
    int per_sm_1cta128;
    int per_sm_1cta256;
    int skinny_clusters[kSkinnyMaxPieces + 1];   // index P: co-resident clusters of P CTAs (0: unknown)
    int split_clusters[kSplitMaxPieces + 1];     // index S: co-resident clusters of S CTA pairs
    int split1_clusters[kSplitMaxPieces1 + 1];   // index S: co-resident clusters of S single CTAs
};

// A pure-host planner's view of a GPU with `sms` SMs (nothing queried).
Limits host_limits(int sms) {
    Limits lim{sms, sms / 2, sms / 2, 1, 1, {}, {}, {}};
    for (int pc = 1; pc <= kSkinnyMaxPieces; pc *= 2) lim.skinny_clusters[pc] = sms / pc;
    for (int s = 1; s <= kSplitMaxPieces; ++s) lim.split_clusters[s] = sms / (2 * s);
    for (int s = 1; s <= kSplitMaxPieces1; ++s) lim.split1_clusters[s] = sms / s;
    return lim;
}

// Column ranges x K pieces of the small-M kernel (kernel_skinny.cuh).  For P
// in {1, 2, 4, 8} pieces per range: with P > 1 one range per cluster and all
// clusters resident at once, R = min(SMs / P, resident clusters, N) ranges,
// and R must reach ceil(N / 128) (ranges of at most 128 columns); with P = 1
// ranges are dealt to at most one CTA per SM, in as many rounds as needed.
// Each choice is timed with a simple model and the fastest wins (ties keep
// the smaller P).  A CTA runs rounds * ceil(kb / P) K blocks of (width + M)
// rows of 128 bytes (its B rows and A's M rows), in ring stages of
// skinny_stage_atoms() blocks; it takes the longer of those bytes at its share
// of HBM bandwidth and of its issue time (kSkinnyStageUs per stage plus
// kSkinnyAtomUs per K block), plus a quarter of the shorter one (the two
// never overlap perfectly), plus the in-cluster sum when P > 1.  The issue
// costs are measured on GB300 with P forced (builds fixing P) and the blocks
// per stage varied: 16 x 1024 x 8192 on 152 ranges of 7 columns (P = 1) takes
// 35.8 / 24.5 / 20.2 us with 1 / 2 / 4 K blocks per stage, 0.28 / 0.38 /
// 0.63 us per stage whatever the bytes.  At N = 8192 ranges of 108 columns in
// pairs beat 152 ranges of 54 by 0.5-2.4 us (fp16 and E4M3, M = 1-64).
constexpr double kSkinnyHbmBytesPerUs = 6.7e6;
constexpr double kSkinnyOverlapLoss = 0.25;
constexpr double kSkinnyStageUs = 0.18;
constexpr double kSkinnyAtomUs = 0.10;
constexpr double kSkinnyExchangeUs = 0.5;

struct SkinnyShape {
    int pieces;
    int64_t ranges, width, rounds, grid;
};

// K blocks the small-M ring holds for ranges of `width` columns.
int skinny_ring_atoms(const SkinnyOps& ops, int64_t width) {
    return std::min(ops.max_atoms, ops.ring_bytes / (skinny_w_stride(static_cast<int>(width)) + ops.x_bytes));
}

SkinnyShape plan_skinny(int64_t M, int64_t N, int64_t kb, const Limits& lim, const SkinnyOps& ops) {
    const int64_t G = lim.sms;
    const int64_t r_min = cdiv(N, 128);
    SkinnyShape best{1, 0, 0, 0, 0};
    double best_t = 0.0;
    for (int pc = 1; pc <= kSkinnyMaxPieces; pc *= 2) {
        if (pc > kb) break;
#ifdef GEMM_SKINNY_PIECES
        // a build that fixes P (where the shape allows it), for measurements
        if (pc != GEMM_SKINNY_PIECES && best.ranges != 0) continue;
#endif
        SkinnyShape sh{pc, 0, 0, 1, 0};
        if (pc == 1) {
            sh.rounds = cdiv(r_min, G);
            sh.ranges = std::min<int64_t>(sh.rounds * G, N);
            sh.grid = std::min<int64_t>(sh.ranges, G);
        } else {
            const int64_t cap = std::min<int64_t>(G / pc, lim.skinny_clusters[pc]);
            if (cap < r_min) continue;
            sh.ranges = std::min<int64_t>(cap, N);
            sh.grid = sh.ranges * pc;
        }
        sh.width = cdiv(N, sh.ranges);
        const int64_t per_range = cdiv(kb, pc);
        const int64_t ka = skinny_stage_atoms(skinny_ring_atoms(ops, sh.width));
        const double atoms = static_cast<double>(sh.rounds * per_range);
        const double stages = static_cast<double>(sh.rounds * cdiv(per_range, ka));
        const double bytes = atoms * static_cast<double>((sh.width + M) * kStageRowBytes);
        const double t_bytes = bytes * static_cast<double>(sh.grid) / kSkinnyHbmBytesPerUs;
        const double t_issue = stages * kSkinnyStageUs + atoms * kSkinnyAtomUs;
        double t = std::max(t_bytes, t_issue) + kSkinnyOverlapLoss * std::min(t_bytes, t_issue) +
                   (pc > 1 ? kSkinnyExchangeUs : 0.0);
#ifdef GEMM_SKINNY_PIECES
        if (pc == GEMM_SKINNY_PIECES) t = -1.0;
#endif
        if (best.ranges == 0 || t < best_t - 1e-9) {
            best = sh;
            best_t = t;
        }
    }
    return best;
}

// B blocks (width rows of 128 bytes) each small-M CTA prefetches into L2
// before its dependency wait, while the previous kernel in the stream
// finishes: the whole grid prefetches at most kSkinnyPrefetchPct percent of
// B and at most kSkinnyPrefetchBytes (at least one block per CTA).
#ifndef GEMM_SKINNY_PREFETCH_MB
#define GEMM_SKINNY_PREFETCH_MB 48
#endif
#ifndef GEMM_SKINNY_PREFETCH_PCT
#define GEMM_SKINNY_PREFETCH_PCT 50
#endif
constexpr int64_t kSkinnyPrefetchBytes = int64_t{GEMM_SKINNY_PREFETCH_MB} << 20;
constexpr int64_t kSkinnyPrefetchPct = GEMM_SKINNY_PREFETCH_PCT;

int32_t skinny_prefetch_blocks(const gemm_plan_t& pl, int64_t b_bytes) {
    const int64_t per_block = static_cast<int64_t>(pl.grid_ctas) * pl.tile_n * kStageRowBytes;
    const int64_t piece = cdiv(pl.k_blocks, pl.k_split);
    const int64_t budget = std::min<int64_t>(kSkinnyPrefetchBytes, b_bytes / 100 * kSkinnyPrefetchPct);
    const int64_t n = per_block > 0 ? budget / per_block : 1;
    return static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(n, piece)));
}

int skinny_mn(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

// K blocks per ring stage of the tiled kernel.  A launch made only of column
// pieces (narrow MMAs: a stage's MMAs take less time than the stage's barrier
// round trip) takes two K blocks per stage where the configuration has that
// form (the 1-CTA ones); otherwise one.  Measured on GB300
// (fp16, back to back): 1024 x 1024 x 2048 on 128 pieces of 128 x 64, 13.2 ->
// 10.8 us with two; whole 128 x 256 tiles at 2048^3 15.97 -> 17.05 us and pair
// tiles 1-4 % slower with two.
int32_t tiled_stage_atoms(const gemm_plan_t& pl, int max_atoms) {
    int32_t a = (pl.num_full_tiles == 0 && pl.tail_split > 1 && pl.k_split == 1) ? 2 : 1;
    if (a > max_atoms) a = max_atoms;
    while (a > 1 && pl.stages / a < 2) --a;
    return a;
}

// The ops table of a tiled variant.
const TiledOps& tiled_ops_of(gemm_variant_t v, int dtype) {
    switch (v) {
        case GEMM_VARIANT_TILE_1CTA_128x128: return tiled_ops_1cta128(dtype);
        case GEMM_VARIANT_TILE_1CTA_128x256:
        case GEMM_VARIANT_TILE_1CTA_SPLITK: return tiled_ops_1cta256(dtype);
        case GEMM_VARIANT_TILE_2CTA_512x256: return tiled_ops_2cta512(dtype);
        default: return tiled_ops_2cta256(dtype);   // TILE_2CTA_256x256, TILE_2CTA_SPLITK
    }
}

// AUTO for shapes whose pair tiles fill less than one round (see kMidFixedUs).
gemm_variant_t mid_shape_variant(int64_t M, int64_t N, int64_t kb, const Limits& lim) {
    const int64_t t1 = cdiv(M, 128) * cdiv(N, 256);
    const int64_t t2 = cdiv(M, 256) * cdiv(N, 256);
    const double k = static_cast<double>(kb);
    // 128x256 tiles on single CTAs, the last round cut into column pieces
    const int per256 = lim.per_sm_1cta256 > 0 ? lim.per_sm_1cta256 : 1;
    const int64_t slots1 = static_cast<int64_t>(lim.sms) * per256;
    int64_t full1;
    int split1;
    tail_split(t1, slots1, 256, 1, full1, split1);
    const double per_block = split1 == 4 ? kMidBlockUs64 : (split1 == 2 ? kMidBlockUs128 : kMidBlockUs256);
    const int64_t rounds1 = cdiv(full1, slots1) + cdiv((t1 - full1) * split1, slots1);
    double best = kMidFixedUs + static_cast<double>(rounds1) * k * per_block;
    gemm_variant_t v = t1 >= 2 ? GEMM_VARIANT_TILE_1CTA_128x256 : GEMM_VARIANT_TILE_1CTA_128x128;
    // whole pair tiles, long K loops
    if (kb >= kPairMinBlocks) {
        const double t = kMidFixedUs + 1.0 + k * kMidPairBlockUs;
        if (t < best) { best = t; v = GEMM_VARIANT_TILE_2CTA_256x256; }
    }
    // split K over pairs, or over single CTAs
    const int s2 = choose_ksplit(t2, lim.split_clusters, kb);
    if (s2 > 1) {
        const double t = kSplitPairFixedUs + static_cast<double>(cdiv(kb, s2)) * kSplitPairBlockUs;
        if (t < best) { best = t; v = GEMM_VARIANT_TILE_2CTA_SPLITK; }
    }
    const int s1 = choose_ksplit(t1, lim.split1_clusters, kb, kSplitMaxPieces1);
    if (s1 > 1) {
        const double t = kSplit1FixedUs + static_cast<double>(cdiv(kb, s1)) * kSplit1BlockUs;
        if (t < best) { best = t; v = GEMM_VARIANT_TILE_1CTA_SPLITK; }
    }
    return v;
}

gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, gemm_variant_t variant, const Limits& lim,
                        gemm_plan_t* pl, int in_bytes = 2) {
    std::memset(pl, 0, sizeof(*pl));
    const gemm_status_t st = check_sizes(M, N, K, in_bytes);
    if (st != GEMM_OK) return st;
    const int64_t bk = stage_k(in_bytes);
    if (variant < GEMM_VARIANT_AUTO || variant > GEMM_VARIANT_TILE_1CTA_SPLITK) return GEMM_ERR_INVALID_VALUE;
    if ((variant == GEMM_VARIANT_SKINNY_SPLITK || variant == GEMM_VARIANT_SKINNY_STREAMK) && M > 64)
        return GEMM_ERR_INVALID_VALUE;
    if (lim.sms <= 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t pairs = lim.max_clusters_2cta > 0 ? lim.max_clusters_2cta : lim.sms / 2;

    if (variant == GEMM_VARIANT_AUTO) {
        if (M <= 64) {
            variant = GEMM_VARIANT_SKINNY_SPLITK;
        } else {
            // The pair kernel when its 256x256 tiles fill at least one round of
            // CTA pairs (4000x11000x4104: 253 us on pairs vs 350 us on 128x256
            // CTAs), with the exceptions below; under one round, the cost
            // model of mid_shape_variant (128x256 column pieces on single
            // CTAs, whole pair tiles, or split K over pairs or single CTAs).
            const int64_t t2 = cdiv(M, 256) * cdiv(N, 256);
            const int64_t kb = cdiv(K, bk);
            if (t2 >= pairs && kb <= (in_bytes == 1 ? kShortKBlocks8 : kShortKBlocks16))
                variant = GEMM_VARIANT_TILE_1CTA_128x256;
            else if (t2 >= pairs && (K * in_bytes) % 32 != 0 && cdiv(M, 512) * cdiv(N, 256) >= 2 * pairs)
                variant = GEMM_VARIANT_TILE_2CTA_512x256;
            else if (t2 >= pairs)
                variant = GEMM_VARIANT_TILE_2CTA_256x256;
            else
                variant = mid_shape_variant(M, N, kb, lim);
        }
    }
    pl->variant = variant;
    pl->tile_k = static_cast<int32_t>(bk);
    pl->k_blocks = cdiv(K, bk);

    if (variant == GEMM_VARIANT_SKINNY_SPLITK) {
        const int mn = skinny_mn(M);
        const SkinnyOps& ops = skinny_ops(mn, 0);
        pl->cta_group = 1;
        pl->tile_m = mn;
        pl->stages = skinny_ring_atoms(ops, 128);
        pl->smem_bytes = ops.smem_bytes;
        pl->tmem_cols = ops.tmem_cols;
        pl->m_tiles = 1;
        pl->tile_n = 128;
        pl->n_tiles = cdiv(N, 128);
        if (M == 0 || N == 0 || K == 0) return GEMM_OK;
        const SkinnyShape sh = plan_skinny(M, N, pl->k_blocks, lim, ops);
        pl->tile_n = static_cast<int32_t>(sh.width);
        // K blocks in flight: B slots sized to the range width (narrow ranges get more)
        pl->stages = skinny_ring_atoms(ops, pl->tile_n);
        pl->n_tiles = sh.ranges;
        pl->k_split = sh.pieces;
        pl->grid_ctas = static_cast<int32_t>(sh.grid);
        pl->max_tiles_per_cta = static_cast<int32_t>(sh.rounds);
        pl->workspace_bytes = 0;
        return GEMM_OK;
    }

    if (variant == GEMM_VARIANT_SKINNY_STREAMK) {
        const int mn = skinny_mn(M);
        const StreamKOps& ops = streamk_ops(mn, 0);
        pl->cta_group = 1;
        pl->tile_m = mn;
        pl->tile_n = 128;
        pl->stages = ops.stages;
        pl->smem_bytes = ops.smem_bytes;
        pl->tmem_cols = ops.tmem_cols;
        pl->m_tiles = 1;
        pl->n_tiles = cdiv(N, 128);
        if (M == 0 || N == 0 || K == 0) return GEMM_OK;
        const int64_t units = pl->n_tiles * pl->k_blocks;
        const int64_t G = units < lim.sms ? units : lim.sms;
        int64_t max_t = 1;
        for (int64_t c = 0; c < G; ++c) {
            const int64_t u0 = unit_begin(c, units, G), u1 = unit_begin(c + 1, units, G);
            const int64_t span = (u1 - 1) / pl->k_blocks - u0 / pl->k_blocks + 1;
            if (span > max_t) max_t = span;
        }
        pl->grid_ctas = static_cast<int32_t>(G);
        pl->max_tiles_per_cta = static_cast<int32_t>(max_t);
        pl->workspace_bytes = round_up(G * max_t * mn * 128 * 4, 256) + round_up(pl->n_tiles * 4, 256);
        return GEMM_OK;
    }

    if (variant == GEMM_VARIANT_TILE_2CTA_SPLITK &&
        choose_ksplit(cdiv(M, 256) * cdiv(N, 256), lim.split_clusters, pl->k_blocks) < 2)
        variant = GEMM_VARIANT_TILE_2CTA_256x256;   // too many tiles for one wave of clusters: no split
    if (variant == GEMM_VARIANT_TILE_1CTA_SPLITK &&
        choose_ksplit(cdiv(M, 128) * cdiv(N, 256), lim.split1_clusters, pl->k_blocks, kSplitMaxPieces1) < 2)
        variant = GEMM_VARIANT_TILE_1CTA_128x256;
    pl->variant = variant;
    const bool ksplit_variant = variant == GEMM_VARIANT_TILE_2CTA_SPLITK || variant == GEMM_VARIANT_TILE_1CTA_SPLITK;
    const TiledOps& ops = tiled_ops_of(variant, 0);
    pl->cta_group = ops.cta_group;
    pl->tile_m = ops.tile_m;
    pl->tile_n = ops.tile_n;
    pl->stages = ops.stages;
    pl->smem_bytes = ops.smem_bytes;
    pl->tmem_cols = ops.tmem_cols;
    pl->m_tiles = cdiv(M, ops.tile_m);
    pl->n_tiles = cdiv(N, ops.tile_n);
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;
    const int64_t tiles = pl->m_tiles * pl->n_tiles;
    // slots = clusters (or CTAs) that can be resident at once
    int64_t slots;
    if (ops.cta_group == 2) {
        const int c = variant == GEMM_VARIANT_TILE_2CTA_512x256 ? lim.max_clusters_2cta2c : lim.max_clusters_2cta;
        slots = c > 0 ? c : lim.sms / 2;
    } else {
        const int per_sm = variant == GEMM_VARIANT_TILE_1CTA_128x128 ? lim.per_sm_1cta128 : lim.per_sm_1cta256;
        slots = static_cast<int64_t>(lim.sms) * (per_sm > 0 ? per_sm : 1);
    }
    if (slots <= 0) return GEMM_ERR_INVALID_VALUE;
    int64_t num_full;
    int split;
    int ksplit = 1;
    int64_t clusters;
    if (ksplit_variant) {
        // one cluster of ksplit MMA groups per tile, all resident in one wave
        ksplit = variant == GEMM_VARIANT_TILE_1CTA_SPLITK
                     ? choose_ksplit(tiles, lim.split1_clusters, pl->k_blocks, kSplitMaxPieces1)
                     : choose_ksplit(tiles, lim.split_clusters, pl->k_blocks);
        num_full = tiles;
        split = 1;
        clusters = tiles;
        pl->grid_ctas = static_cast<int32_t>(tiles * ksplit * ops.cluster);
    } else {
        tail_split(tiles, slots, ops.tile_n, ops.cta_group, num_full, split);
        const int64_t units = num_full + (tiles - num_full) * split;
        clusters = units < slots ? units : slots;
        pl->grid_ctas = static_cast<int32_t>(clusters * ops.cluster);
    }
    pl->k_split = ksplit;
    pl->num_full_tiles = num_full;
    pl->tail_split = split;
    pl->group_m = static_cast<int32_t>(raster_group(pl->m_tiles, ops.tile_m, K, in_bytes));
    return GEMM_OK;
}

// ----------------------------------------------------------------- device set-up
gemm_status_t get_device(DeviceState** out, int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_devices[dev];
    if (d.unsupported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            d.unsupported = true;
            return GEMM_ERR_UNSUPPORTED_DEVICE;
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        void* status = nullptr;
        if (cudaGetSymbolAddress(&status, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        const TiledOps* tiled[3] = {&tiled_ops_2cta256(0), &tiled_ops_1cta128(0), &tiled_ops_1cta256(0)};
        for (int dt : {0, 1, 2}) {   // fp16, bf16, 8-bit (one kernel for both formats)
            const TiledOps* all[4] = {&tiled_ops_2cta256(dt), &tiled_ops_1cta128(dt), &tiled_ops_1cta256(dt),
                                      &tiled_ops_2cta512(dt)};
            for (const TiledOps* t : all)
                if (t->prepare() != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
            for (int mn : {16, 32, 64})
                if (skinny_ops(mn, dt).prepare() != cudaSuccess || streamk_ops(mn, dt).prepare() != cudaSuccess) {
                    cudaGetLastError();
                    return GEMM_ERR_CUDA;
                }
        }
        int clusters = 0, per128 = 0, per256 = 0, clusters2c = 0;
        if (tiled[0]->max_active(&clusters) != cudaSuccess || tiled[1]->max_active(&per128) != cudaSuccess ||
            tiled[2]->max_active(&per256) != cudaSuccess || tiled_ops_2cta512(0).max_active(&clusters2c) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        d.sms = sms;
        d.status = static_cast<uint32_t*>(status);
        d.max_clusters_2cta = clusters;
        d.max_clusters_2cta2c = clusters2c;
        d.per_sm_1cta128 = per128;
        d.per_sm_1cta256 = per256;
        // co-resident clusters of each size the planner may use (a size the
        // device cannot run at all counts as zero: the planner avoids it)
        d.skinny_clusters[1] = sms;
        for (int pc = 2; pc <= kSkinnyMaxPieces; pc *= 2) {
            if (skinny_ops(16, 0).max_active(pc, &d.skinny_clusters[pc]) != cudaSuccess) {
                cudaGetLastError();
                d.skinny_clusters[pc] = 0;
            }
        }
        d.split_clusters[1] = clusters;
        for (int sp = 2; sp <= kSplitMaxPieces; ++sp) {
            if (tiled[0]->max_active_split(sp, &d.split_clusters[sp]) != cudaSuccess) {
                cudaGetLastError();
                d.split_clusters[sp] = 0;
            }
        }
        d.split1_clusters[1] = sms * per256;
        for (int sp = 2; sp <= kSplitMaxPieces1; ++sp) {
            if (tiled[2]->max_active_split(sp, &d.split1_clusters[sp]) != cudaSuccess) {
                cudaGetLastError();
                d.split1_clusters[sp] = 0;
            }
        }
        d.ready = true;
    }
    *out = &d;
    if (dev_out) *dev_out = dev;
    return GEMM_OK;
}

Limits limits_of(const DeviceState& d) {
    Limits lim{d.sms, d.max_clusters_2cta, d.max_clusters_2cta2c, d.per_sm_1cta128, d.per_sm_1cta256, {}, {}, {}};
    for (int pc = 1; pc <= kSkinnyMaxPieces; ++pc) lim.skinny_clusters[pc] = d.skinny_clusters[pc];
    for (int sp = 1; sp <= kSplitMaxPieces; ++sp) lim.split_clusters[sp] = d.split_clusters[sp];
    for (int sp = 1; sp <= kSplitMaxPieces1; ++sp) lim.split1_clusters[sp] = d.split1_clusters[sp];
    return lim;
}

// L2 promotion of the tiled kernels' operand loads: a 128-byte box row pulls
// in the 256-byte L2 line around it, which the next K block of the same rows
// reads.  Measured on GB300 against none / 64 / 128 bytes: 8192^3 627 against
// 665-672 us, 4000 x 11000 x 4112 214 against 232-238 us.  The small-M
// kernels stream B once with an evict-first policy and take no promotion
// (16 x 8192 x 8192: 22.4 against 24.8 us with 256 bytes).
constexpr CUtensorMapL2promotion kTiledL2Promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
constexpr CUtensorMapL2promotion kStreamL2Promotion = CU_TENSOR_MAP_L2_PROMOTION_NONE;

// 2-D tensor map of a gemm_dtype_t's elements (fp16, bf16, or bytes for the
// 8-bit types): `inner` contiguous elements per row, `outer` rows, box of
// box_inner x box_outer elements, 128-byte swizzle, zero fill outside.
bool encode_2d(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, uint32_t box_inner,
               uint32_t box_outer, int dtype = 0, CUtensorMapL2promotion promotion = kTiledL2Promotion) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * dtype_in_bytes(dtype)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t elem[2] = {1, 1};
    const CUtensorMapDataType type = dtype >= GEMM_DTYPE_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == GEMM_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = g_encode(map, type, 2, const_cast<void*>(base), dims,
                                strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, promotion,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

gemm_status_t get_workspace(int dev, gemm_stream_t stream, size_t partial_bytes, size_t n_counters,
                            Workspace** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = g_workspaces[std::make_pair(dev, static_cast<void*>(stream))];
    if (w.partial_bytes < partial_bytes) {
        // growing: the old buffer may still be in use by work queued on this stream
        if (w.partials) {
            if (cudaStreamSynchronize(stream) != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
            cudaFree(w.partials);
            w.partials = nullptr;
            w.partial_bytes = 0;
        }
        if (cudaMalloc(&w.partials, partial_bytes) != cudaSuccess) {
            cudaGetLastError();
            w.partials = nullptr;
            return GEMM_ERR_CUDA;
        }
        w.partial_bytes = partial_bytes;
    }
    if (w.n_counters < n_counters) {
        if (w.counters) {
            if (cudaStreamSynchronize(stream) != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
            cudaFree(w.counters);
            w.counters = nullptr;
            w.n_counters = 0;
        }
        if (cudaMalloc(&w.counters, n_counters * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            w.counters = nullptr;
            return GEMM_ERR_CUDA;
        }
        // counters start at zero; every call leaves them at zero again
        if (cudaMemset(w.counters, 0, n_counters * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        w.n_counters = n_counters;
    }
    *out = &w;
    return GEMM_OK;
}

bool ranges_overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    if (a_bytes <= 0 || b_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t timeout_for(int64_t k_blocks) {
    // two seconds plus a generous 2 us per K block of the longest tile
    return 2000000000ull + static_cast<uint64_t>(k_blocks) * 2000ull;
}

// Elementwise D = act(beta * C + bias) for K == 0 (the empty sum) when a fused
// epilogue is asked for.
template <class T>
__global__ void epilogue_only_kernel(T* D, int64_t M, int64_t N, EpiParams e) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / N, col = i - (i / N) * N;
        D[i] = Elem<T>::from_float(epi_apply1<T>(e, 0.0f, row, col, N));
    }
}

EpiParams epi_params(const gemm_epilogue_t* e) {
    EpiParams p;
    p.alpha = 1.0f;
    p.beta = 0.0f;
    p.C = nullptr;
    p.bias = nullptr;
    p.scale_n = nullptr;
    p.act = 0;
    p.on = 0;
    if (e == nullptr) return p;
    p.alpha = e->alpha;
    p.beta = e->beta;
    p.C = e->beta != 0.0f ? e->C : nullptr;
    p.bias = e->bias;
    p.scale_n = e->scale_n;
    p.act = e->activation;
    p.on = (p.alpha != 1.0f || p.C != nullptr || p.bias != nullptr || p.scale_n != nullptr || p.act != 0) ? 1 : 0;
    return p;
}

gemm_status_t run(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                  gemm_variant_t variant, gemm_stream_t stream, int dtype = 0,
                  const gemm_epilogue_t* epilogue = nullptr) {
    // ---- host-only argument checks (nothing touches a device before these pass)
    if (!dtype_valid(dtype)) return GEMM_ERR_INVALID_VALUE;
    const int in_bytes = dtype_in_bytes(dtype);
    gemm_status_t st = check_sizes(M, N, K, in_bytes);
    if (st != GEMM_OK) return st;
    const EpiParams epi = epi_params(epilogue);
    if (epilogue != nullptr) {
        if (epilogue->activation != GEMM_ACT_NONE && epilogue->activation != GEMM_ACT_RELU)
            return GEMM_ERR_INVALID_VALUE;
        if (epilogue->beta != 0.0f && epilogue->C == nullptr) return GEMM_ERR_INVALID_VALUE;
        if ((epi.C && !aligned16(epi.C)) || (epi.bias && !aligned16(epi.bias)) ||
            (epi.scale_n && !aligned16(epi.scale_n)))
            return GEMM_ERR_MISALIGNED;
        // C may be D itself (an in-place update); it may not partly overlap D, and
        // neither the bias nor the scales may overlap D at all
        if (M > 0 && N > 0) {
            if (epi.C && epi.C != D && ranges_overlap(epi.C, M * N * 2, D, M * N * 2)) return GEMM_ERR_INVALID_VALUE;
            if (epi.bias && ranges_overlap(epi.bias, N * 2, D, M * N * 2)) return GEMM_ERR_INVALID_VALUE;
            if (epi.scale_n && ranges_overlap(epi.scale_n, N * 4, D, M * N * 2)) return GEMM_ERR_INVALID_VALUE;
        }
    }
    if (variant < GEMM_VARIANT_AUTO || variant > GEMM_VARIANT_TILE_1CTA_SPLITK) return GEMM_ERR_INVALID_VALUE;
    if ((variant == GEMM_VARIANT_SKINNY_SPLITK || variant == GEMM_VARIANT_SKINNY_STREAMK) && M > 64)
        return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (D == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_VALUE;
    const int64_t a_bytes = M * K * in_bytes, b_bytes = N * K * in_bytes, d_bytes = M * N * 2;
    if (ranges_overlap(D, d_bytes, A, a_bytes) || ranges_overlap(D, d_bytes, B, b_bytes))
        return GEMM_ERR_INVALID_VALUE;
    if (!aligned16(D) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return GEMM_ERR_MISALIGNED;

    DeviceState* dev = nullptr;
    int dev_id = 0;
    st = get_device(&dev, &dev_id);
    if (st != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int out_dtype = dtype_out(dtype);
    const int bk = stage_k(in_bytes);

    if (K == 0) {  // the empty sum
        if (epi.on) {
            const int blocks = static_cast<int>(std::min<int64_t>(cdiv(M * N, 256), 8 * dev->sms));
            if (out_dtype == GEMM_DTYPE_BF16)
                epilogue_only_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16*>(D), M, N, epi);
            else
                epilogue_only_kernel<__half><<<blocks, 256, 0, s>>>(static_cast<__half*>(D), M, N, epi);
            if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
            return GEMM_OK;
        }
        if (cudaMemsetAsync(D, 0, static_cast<size_t>(d_bytes), s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }

    gemm_plan_t pl;
    st = make_plan(M, N, K, variant, limits_of(*dev), &pl, in_bytes);
    if (st != GEMM_OK) return st;

    if (pl.variant == GEMM_VARIANT_SKINNY_SPLITK) {
        const SkinnyOps& ops = skinny_ops(pl.tile_m, dtype);
        CUtensorMap tw, tx;
        if (!encode_2d(&tw, B, K, N, bk, static_cast<uint32_t>(pl.tile_n), dtype, kStreamL2Promotion) ||
            !encode_2d(&tx, A, K, M, bk, static_cast<uint32_t>(ops.mn), dtype, kStreamL2Promotion))
            return GEMM_ERR_INVALID_VALUE;
        SkinnyParams p;
        p.M = static_cast<int32_t>(M);
        p.N = static_cast<int32_t>(N);
        p.K = static_cast<int32_t>(K);
        p.k_blocks = static_cast<int32_t>(pl.k_blocks);
        p.width = pl.tile_n;
        p.ranges = static_cast<int32_t>(pl.n_tiles);
        p.pieces = pl.k_split;
        p.stage_atoms = skinny_stage_atoms(pl.stages);
        p.stages = pl.stages / p.stage_atoms;
        p.w_stride = skinny_w_stride(pl.tile_n);
        p.D = D;
        p.epi = epi;
        p.status = dev->status;
        p.timeout_ns = timeout_for(pl.k_blocks);
        p.stream_b = b_bytes >= kStreamBBytes ? 1 : 0;
        p.ab_format = dtype_ab_format(dtype);
        p.prefetch_blocks = skinny_prefetch_blocks(pl, b_bytes);
        if (ops.launch(tw, tx, p, pl.grid_ctas, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        return GEMM_OK;
    }

    if (pl.variant == GEMM_VARIANT_SKINNY_STREAMK) {
        const StreamKOps& ops = streamk_ops(pl.tile_m, dtype);
        CUtensorMap tw, tx;
        if (!encode_2d(&tw, B, K, N, bk, 128, dtype) ||
            !encode_2d(&tx, A, K, M, bk, static_cast<uint32_t>(ops.mn), dtype))
            return GEMM_ERR_INVALID_VALUE;
        Workspace* ws = nullptr;
        const size_t partial_bytes = static_cast<size_t>(pl.grid_ctas) * pl.max_tiles_per_cta * ops.mn * 128 * 4;
        st = get_workspace(dev_id, stream, partial_bytes, static_cast<size_t>(pl.n_tiles), &ws);
        if (st != GEMM_OK) return st;
        // Every completed call leaves the tile counters at zero, but one that
        // gave up waiting (a timeout) may not; clear them on the stream so a
        // later call never starts from counts an earlier one left behind.
        if (cudaMemsetAsync(ws->counters, 0, static_cast<size_t>(pl.n_tiles) * sizeof(uint32_t), s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        StreamKParams p;
        p.M = static_cast<int32_t>(M);
        p.N = static_cast<int32_t>(N);
        p.K = static_cast<int32_t>(K);
        p.n_tiles = static_cast<int32_t>(pl.n_tiles);
        p.k_blocks = static_cast<int32_t>(pl.k_blocks);
        p.num_ctas = pl.grid_ctas;
        p.max_tiles_per_cta = pl.max_tiles_per_cta;
        p.units = pl.n_tiles * pl.k_blocks;
        p.partials = ws->partials;
        p.counters = ws->counters;
        p.D = D;
        p.epi = epi;
        p.status = dev->status;
        p.timeout_ns = timeout_for(pl.k_blocks);
        p.stream_b = b_bytes >= kStreamBBytes ? 1 : 0;
        p.ab_format = dtype_ab_format(dtype);
        if (ops.launch(tw, tx, p, pl.grid_ctas, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        return GEMM_OK;
    }

    const TiledOps& ops = tiled_ops_of(static_cast<gemm_variant_t>(pl.variant), dtype);
    CUtensorMap ta, tb, tbp, td;
    const uint32_t b_rows = static_cast<uint32_t>(ops.b_box_rows);
    if (!encode_2d(&ta, A, K, M, bk, 128, dtype) || !encode_2d(&tb, B, K, N, bk, b_rows, dtype) ||
        !encode_2d(&tbp, B, K, N, bk, b_rows / static_cast<uint32_t>(pl.tail_split), dtype) ||
        !encode_2d(&td, D, N, M, 64, 32, out_dtype))
        return GEMM_ERR_INVALID_VALUE;
    TiledParams p;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.k_blocks = static_cast<int32_t>(pl.k_blocks);
    p.m_tiles = pl.m_tiles;
    p.n_tiles = pl.n_tiles;
    p.num_tiles = pl.m_tiles * pl.n_tiles;
    p.group_m = pl.group_m;
    p.num_full = pl.num_full_tiles;
    p.split = pl.tail_split;
    p.ksplit = pl.k_split;
    p.ab_format = dtype_ab_format(dtype);
    p.last_k_steps = static_cast<int32_t>(cdiv(K * in_bytes - (pl.k_blocks - 1) * kStageRowBytes, 32));
    p.num_units = pl.k_split > 1 ? p.num_tiles
                                 : pl.num_full_tiles + (p.num_tiles - pl.num_full_tiles) * pl.tail_split;
    p.stage_atoms = tiled_stage_atoms(pl, ops.max_stage_atoms);
    p.D = D;
    p.epi = epi;
    p.status = dev->status;
    p.timeout_ns = timeout_for(pl.k_blocks);
    if (ops.launch(ta, tb, tbp, td, p, pl.grid_ctas, s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

// ----------------------------------------------------------------- no-allocation entry
// Scratch for gemm_f16_nt_noalloc: one fixed array per device that loads this
// library, laid out as [per-tile counters, 256-byte padded][fp32 partials].
// It exists from module load until the process exits; nothing here ever calls
// cudaMalloc or cudaFree for it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[GEMM_F16_NOALLOC_SCRATCH_BYTES];

constexpr int kNoAllocMaxDevices = 64;
uint8_t* g_noalloc_ptr[kNoAllocMaxDevices] = {};  // device address of the array, per device

// Set-up, once per device, with that device current: the array's name in host
// code is only a host-side stand-in, so fetch its device address.
gemm_status_t noalloc_scratch(int dev, uint8_t** out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return GEMM_OK;
}

gemm_status_t run_noalloc(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                          gemm_stream_t stream) {
    gemm_status_t st = check_sizes(M, N, K);
    if (st != GEMM_OK) return st;
    if (M > 64) return GEMM_ERR_INVALID_VALUE;  // only the small-M kernel uses scratch
    if (M == 0 || N == 0) return GEMM_OK;
    if (D == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_VALUE;
    const int64_t a_bytes = M * K * 2, b_bytes = N * K * 2, d_bytes = M * N * 2;
    if (ranges_overlap(D, d_bytes, A, a_bytes) || ranges_overlap(D, d_bytes, B, b_bytes))
        return GEMM_ERR_INVALID_VALUE;
    if (!aligned16(D) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return GEMM_ERR_MISALIGNED;

    DeviceState* dev = nullptr;
    int dev_id = 0;
    st = get_device(&dev, &dev_id);
    if (st != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        if (cudaMemsetAsync(D, 0, static_cast<size_t>(d_bytes), s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }

    gemm_plan_t pl;
    st = make_plan(M, N, K, GEMM_VARIANT_SKINNY_STREAMK, limits_of(*dev), &pl);
    if (st != GEMM_OK) return st;
    const StreamKOps& ops = streamk_ops(pl.tile_m, 0);
    const size_t counter_bytes = static_cast<size_t>(round_up(pl.n_tiles * 4, 256));
    const size_t partial_bytes = static_cast<size_t>(pl.grid_ctas) * pl.max_tiles_per_cta * ops.mn * 128 * 4;
    if (counter_bytes + partial_bytes > static_cast<size_t>(GEMM_F16_NOALLOC_SCRATCH_BYTES))
        return GEMM_ERR_INVALID_VALUE;  // larger than the fixed scratch: nothing is launched

    uint8_t* scratch = nullptr;
    st = noalloc_scratch(dev_id, &scratch);
    if (st != GEMM_OK) return st;
    CUtensorMap tw, tx;
    if (!encode_2d(&tw, B, K, N, kBK, 128) || !encode_2d(&tx, A, K, M, kBK, static_cast<uint32_t>(ops.mn)))
        return GEMM_ERR_INVALID_VALUE;
    // The counters must start at zero.  Every completed call leaves them at
    // zero, but the array is shared by all calls, so clear them on the stream
    // rather than trust what an earlier (possibly cut-short) call left.
    if (cudaMemsetAsync(scratch, 0, counter_bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    StreamKParams p;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.n_tiles = static_cast<int32_t>(pl.n_tiles);
    p.k_blocks = static_cast<int32_t>(pl.k_blocks);
    p.num_ctas = pl.grid_ctas;
    p.max_tiles_per_cta = pl.max_tiles_per_cta;
    p.units = pl.n_tiles * pl.k_blocks;
    p.partials = reinterpret_cast<float*>(scratch + counter_bytes);
    p.counters = reinterpret_cast<uint32_t*>(scratch);
    p.D = D;
    p.epi = epi_params(nullptr);
    p.status = dev->status;
    p.timeout_ns = timeout_for(pl.k_blocks);
    p.stream_b = N * K * 2 >= kStreamBBytes ? 1 : 0;
    p.ab_format = dtype_ab_format(GEMM_DTYPE_F16);
    if (ops.launch(tw, tx, p, pl.grid_ctas, s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace

extern "C" {

GEMM_API gemm_status_t gemm_f16_nt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                                   gemm_stream_t stream) {
    return run(A, B, D, M, N, K, GEMM_VARIANT_AUTO, stream);
}

GEMM_API gemm_status_t gemm_f16_nt_variant(const void* A, const void* B, void* D, int64_t M, int64_t N,
                                           int64_t K, gemm_variant_t variant, gemm_stream_t stream) {
    return run(A, B, D, M, N, K, variant, stream);
}

GEMM_API gemm_status_t gemm_bf16_nt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                                    gemm_stream_t stream) {
    return run(A, B, D, M, N, K, GEMM_VARIANT_AUTO, stream, GEMM_DTYPE_BF16, nullptr);
}

GEMM_API gemm_status_t gemm_nt_ex(gemm_dtype_t dtype, const void* A, const void* B, void* D, int64_t M, int64_t N,
                                  int64_t K, const gemm_epilogue_t* epilogue, gemm_variant_t variant,
                                  gemm_stream_t stream) {
    return run(A, B, D, M, N, K, variant, stream, static_cast<int>(dtype), epilogue);
}

GEMM_API gemm_status_t gemm_f16_nt_check(gemm_stream_t stream) {
    DeviceState* dev = nullptr;
    int dev_id = 0;
    gemm_status_t st = get_device(&dev, &dev_id);
    if (st != GEMM_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (word == 0) return GEMM_OK;
    // clear the word, and re-arm the skinny counters a cut-short kernel may have left set
    cudaMemset(dev->status, 0, sizeof(uint32_t));
    {
        std::lock_guard<std::mutex> lock(g_mu);
        for (auto& kv : g_workspaces)
            if (kv.first.first == dev_id && kv.second.counters)
                cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(uint32_t));
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    const uint32_t code = word & 0xFFu;
    return code == GEMM_ERR_TIMEOUT ? GEMM_ERR_TIMEOUT : GEMM_ERR_CUDA;
}

GEMM_API const char* gemm_status_string(gemm_status_t status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE: bad size, pointer, overlap or variant";
        case GEMM_ERR_MISALIGNED:
            return "GEMM_ERR_MISALIGNED: pointers must be 16-byte aligned, N a multiple of 8 and K of 8 "
                   "(16 for 8-bit operands)";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3 (sm_103a)";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch failed";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a kernel gave up waiting on a barrier";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA runtime call failed";
    }
    return "unknown gemm_status_t";
}

GEMM_API gemm_status_t gemm_f16_nt_plan(int64_t M, int64_t N, int64_t K, gemm_variant_t variant,
                                        int32_t num_sms, gemm_plan_t* plan) {
    if (plan == nullptr) return GEMM_ERR_INVALID_VALUE;
    Limits lim;
    if (num_sms > 0) {
        lim = host_limits(num_sms);
    } else {
        DeviceState* dev = nullptr;
        const gemm_status_t st = get_device(&dev, nullptr);
        if (st != GEMM_OK) return st;
        lim = limits_of(*dev);
    }
    return make_plan(M, N, K, variant, lim, plan);
}

GEMM_API gemm_status_t gemm_nt_plan_ex(gemm_dtype_t dtype, int64_t M, int64_t N, int64_t K, gemm_variant_t variant,
                                       int32_t num_sms, gemm_plan_t* plan) {
    if (plan == nullptr || !dtype_valid(dtype)) return GEMM_ERR_INVALID_VALUE;
    Limits lim;
    if (num_sms > 0) {
        lim = host_limits(num_sms);
    } else {
        DeviceState* dev = nullptr;
        const gemm_status_t st = get_device(&dev, nullptr);
        if (st != GEMM_OK) return st;
        lim = limits_of(*dev);
    }
    return make_plan(M, N, K, variant, lim, plan, dtype_in_bytes(dtype));
}

GEMM_API gemm_status_t gemm_selftest_timeout(int32_t timeout_us, gemm_stream_t stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return GEMM_ERR_INVALID_VALUE;
    DeviceState* dev = nullptr;
    const gemm_status_t st = get_device(&dev, nullptr);
    if (st != GEMM_OK) return st;
    selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        dev->status, static_cast<uint64_t>(timeout_us) * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

GEMM_API gemm_status_t gemm_f16_nt_noalloc(const void* A, const void* B, void* D, int64_t M, int64_t N,
                                           int64_t K, gemm_stream_t stream) {
    return run_noalloc(A, B, D, M, N, K, stream);
}

}  // extern "C"
