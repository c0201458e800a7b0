// config.h -- tile configurations and the index arithmetic that the host
// planner and the kernels must agree on (grouped tile raster, the skinny
// kernel's split of the K loop across CTAs).  Host and device code.
#pragma once

#include <cstdint>

#include "epilogue.cuh"
#include "ptx.cuh"

#if defined(__CUDACC__)
#define GEMM_HD __host__ __device__ __forceinline__
#else
#define GEMM_HD inline
#endif

namespace gemm_gb300 {

// One pipeline stage moves one 128-byte row of A and of B per tile row: the
// width of the 128-byte swizzle ("Building a Tiled GEMM", step 1: BLK_K = 64
// fp16 with a 128-byte-swizzled SMEM layout).  That is 64 K elements of fp16
// or bf16 and 128 of an 8-bit type.  One MMA instruction takes 32 bytes of
// each row (K = 16 for 16-bit types, 32 for 8-bit ones): four per stage.
constexpr int kStageRowBytes = 128;
constexpr int kMmaPerStage = kStageRowBytes / 32;
GEMM_HD constexpr int stage_k(int elem_bytes) { return kStageRowBytes / elem_bytes; }
constexpr int kBK = stage_k(2);   // K elements per stage for 16-bit operands
// Warp roles of every kernel: warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs, warps 2..5 are the epilogue warpgroup (warp w reads TMEM
// lanes 32*(w%4) .. 32*(w%4)+31).
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxDynSmem = 232448;  // 227 KB per CTA on sm_100-class GPUs

GEMM_HD int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// a / b for a >= 0, b > 0.  On the device a 64-bit division is a long
// software sequence; when both fit in 32 bits (every realistic problem) the
// 32-bit division gives the same quotient much faster.
GEMM_HD int64_t div_nonneg(int64_t a, int64_t b) {
#if defined(__CUDA_ARCH__)
    if ((static_cast<uint64_t>(a) | static_cast<uint64_t>(b)) <= 0xFFFFFFFFull)
        return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
#endif
    return a / b;
}


// ------------------------------------------------------------------ tiled
// Persistent, warp-specialised kernel.  CG = CTAs per MMA (1, or 2 for a
// cta_group::2 pair in a 2-CTA cluster), BN = output columns per tile.  With
// one consumer a tile is 128*CG rows by BN columns; each CTA of a pair loads
// its own 128 rows of A and its own BN/CG rows of B and owns 128 accumulator
// rows in its TMEM.  Reuse of A and B blocks between tiles comes from L2
// (grouped raster below).
// CONS = MMA consumers per CTA sharing each staged B tile ("Building a Tiled
// GEMM", optimisation roadmap, last item): with 2, each CTA stages 2 x 128 rows
// of A and its BN/CG rows of B once, and two MMAs per K step (one per 128-row
// half of A) feed two accumulators -- a tile of 2*128*CG rows -- each drained
// by its own epilogue warpgroup.  B then crosses from L2 once for twice the
// rows, a quarter less operand traffic per FLOP; the two accumulators fill
// TMEM, so they are single-buffered and the epilogue no longer hides under
// the next tile's MMAs.
template <int CG_, int BN_, int STAGES_, int CONS_ = 1>
struct TiledConfig {
    static constexpr int CG = CG_;
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int CONS = CONS_;
    static constexpr int MMA_M = 128 * CG;                   // rows of one MMA
    static constexpr int BM = MMA_M * CONS;                  // rows of a tile
    static constexpr int A_ROWS = 128 * CONS;                // per CTA
    static constexpr int B_ROWS = BN / CG;
    static constexpr int A_BYTES = A_ROWS * kStageRowBytes;
    static constexpr int A_HALF_BYTES = 128 * kStageRowBytes;   // one consumer's A rows
    static constexpr int B_BYTES = B_ROWS * kStageRowBytes;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // per CTA
    static constexpr int EPI_WARPS = kEpiWarps * CONS;      // one warpgroup per consumer
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int ACC_BUFS = CONS == 1 ? 2 : 1;       // accumulator buffers per consumer
    static constexpr int TMEM_COLS = ACC_BUFS * CONS * BN;
    static constexpr int EPI_COLS = 64;                      // columns per TMA store box
    static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;  // one warp's 32 rows
    // The operand ring holds STAGES whole stages of [A tile | B tile].  A launch
    // made only of column pieces (see tail_split) needs only B_BYTES / split of
    // B per stage, so it packs more, smaller stages into the same ring: more
    // bytes in flight for the latency-bound small problems.
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int MAX_SPLIT = (BN / 64 < 4) ? BN / 64 : 4;
    static constexpr int MAX_STAGES = RING_BYTES / (A_BYTES + B_BYTES / MAX_SPLIT);
    static constexpr int OFF_EPI = RING_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * 2 * EPI_BUF_BYTES;
    // full[MAX_STAGES], empty[MAX_STAGES], tmem_full[2], tmem_empty[2], drain
    static constexpr int NUM_BARS = 2 * MAX_STAGES + 5;
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    // per epilogue warp: the per-column scales (64 fp32) and bias (64 x 16 bit)
    // of the chunk it is writing, read back by every lane as broadcasts
    static constexpr int COLS_BYTES = EPI_COLS * 4 + EPI_COLS * 2;
    static constexpr int OFF_COLS = (OFF_SLOT + 16 + 15) / 16 * 16;
    static constexpr int SMEM_BYTES = OFF_COLS + EPI_WARPS * COLS_BYTES + 1024;  // + slack to align the base
    static_assert(A_BYTES % 1024 == 0 && (B_BYTES / MAX_SPLIT) % 1024 == 0, "stage tiles must stay 1024-aligned");
    static_assert(CONS == 1 || CONS == 2, "one or two consumers");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be a multiple of 64 up to 256");
    static_assert(B_ROWS <= 256, "TMA box rows are limited to 256");
    static_assert(SMEM_BYTES <= kMaxDynSmem, "shared memory budget exceeded");
    static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
};

using Cfg2cta256 = TiledConfig<2, 256, 6>;
using Cfg2cta512 = TiledConfig<2, 256, 3, 2>;   // two consumers: 512 x 256 per pair
using Cfg1cta128 = TiledConfig<1, 128, 6>;
using Cfg1cta256 = TiledConfig<1, 256, 4>;

struct TiledParams {
    int32_t M, N, K;
    int32_t k_blocks;
    int64_t m_tiles, n_tiles;
    int64_t num_tiles;
    int64_t group_m;          // tile rows per raster group
    int64_t num_full;         // tiles run whole: the persistent grid's full rounds
    int64_t num_units;        // num_full + (num_tiles - num_full) * split
    int32_t split;            // the remaining tiles are cut into `split` column pieces
    int32_t ksplit;           // > 1: every tile's K loop is cut into ksplit pieces, run by the
                              // ksplit MMA groups of one cluster (split K)
    uint32_t ab_format;       // operand format field of the MMA instruction descriptor
    int32_t last_k_steps;     // 32-byte K steps of real data in the last K block (1..4)
    int32_t stage_atoms;      // K blocks per ring stage (consecutive ring slots)
    void* D;                  // the output (fp16 or bf16 [M][N]); written directly by the
                              // split-K slice sums, through tmD otherwise
    EpiParams epi;            // fused output transform (epi.on == 0: plain D = A B^T)
    uint32_t* status;         // device status word (0 = ok)
    uint64_t timeout_ns;      // per-wait budget
};

// Grouped raster: tiles are numbered in groups of `group_m` tile rows; inside
// a group the tile row varies fastest, so CTAs working at the same time share
// A rows and B rows through L2.
GEMM_HD void tile_coords(int64_t t, int64_t m_tiles, int64_t n_tiles, int64_t group_m,
                         int64_t& tm, int64_t& tn) {
    const int64_t per_group = group_m * n_tiles;
    const int64_t g = div_nonneg(t, per_group);
    const int64_t first_m = g * group_m;
    const int64_t rows = (m_tiles - first_m < group_m) ? (m_tiles - first_m) : group_m;
    const int64_t r = t - g * per_group;
    tn = div_nonneg(r, rows);
    tm = first_m + (r - tn * rows);
}

// Bytes per ring stage of a launch: a whole [A | B] stage, or, when every
// unit is a column piece (no whole tiles), [A | B / split].
GEMM_HD int ring_stride(const TiledParams& p, int a_bytes, int b_bytes) {
    return (p.num_full == 0 && p.split > 1) ? a_bytes + b_bytes / p.split : a_bytes + b_bytes;
}

// Work unit u of the persistent loop -> (tile row tm, first column n0,
// column count nw, K blocks [kb0, kb1)).  The first num_full units are whole
// tiles in raster order; the tiles of the last, partly filled round are cut
// into `split` column pieces so that more CTA pairs share that round.  With
// split K, unit u is tile u and MMA group `group` of the cluster runs the
// group-th of ksplit even shares of its K blocks.
GEMM_HD void work_unit(int64_t u, const TiledParams& p, int BN, int group, int64_t& tm, int64_t& n0, int& nw,
                       int& kb0, int& kb1) {
    kb0 = 0;
    kb1 = p.k_blocks;
    if (p.ksplit > 1) {
        const int64_t t = u;
        const int j = group;
        int64_t tn;
        tile_coords(t, p.m_tiles, p.n_tiles, p.group_m, tm, tn);
        nw = BN;
        n0 = tn * BN;
        kb0 = static_cast<int>(div_nonneg(static_cast<int64_t>(j) * p.k_blocks, p.ksplit));
        kb1 = static_cast<int>(div_nonneg(static_cast<int64_t>(j + 1) * p.k_blocks, p.ksplit));
        return;
    }
    int64_t t = u, piece = 0;
    int s = 1;
    if (u >= p.num_full) {
        const int64_t v = u - p.num_full;
        s = p.split;
        const int64_t q = div_nonneg(v, s);
        t = p.num_full + q;
        piece = v - q * s;
    }
    int64_t tn;
    tile_coords(t, p.m_tiles, p.n_tiles, p.group_m, tm, tn);
    nw = BN / s;
    n0 = tn * BN + piece * nw;
}

// Split of the last round: whole rounds of `slots` tiles run first; the
// remaining tiles are cut into s column pieces (s = 1, 2 or 4, pieces at
// least 64 columns wide).  A piece does 1/s of the MMA work, but each CTA
// still loads all its 128 rows of A per K block, so its time is modelled as
// max(1/s, (128 + BN/(CG*s)) / (128 + BN/CG)) of a whole tile; the tail costs
// ceil(rem * s / slots) such piece times, and the cheapest s wins (ties keep
// the smaller s).
inline void tail_split(int64_t num_tiles, int64_t slots, int BN, int CG, int64_t& num_full, int& split) {
    num_full = (num_tiles / slots) * slots;
    const int64_t rem = num_tiles - num_full;
    split = 1;
    if (rem == 0) return;
    double best = static_cast<double>(cdiv(rem, slots));
    for (int s = 2; s <= 4 && BN / s >= 64; s *= 2) {
        const double load = (128.0 + static_cast<double>(BN) / (CG * s)) / (128.0 + static_cast<double>(BN) / CG);
        const double piece = load > 1.0 / s ? load : 1.0 / s;
        const double cost = static_cast<double>(cdiv(rem * s, slots)) * piece;
        if (cost < best - 1e-9) {
            best = cost;
            split = s;
        }
    }
}

// Split-K factor S (a cluster of S MMA groups per tile: S pairs, S <= 4, or S
// single CTAs, S <= 8, so that a cluster has at most the 8 CTAs every GPU of
// this class supports): the most pieces such that every tile's cluster is
// resident in one wave (tiles <= clusters[S], the co-resident clusters of S
// groups) and every piece keeps at least kSplitMinBlocks K blocks; 1 = no
// split.
constexpr int kSplitMaxPieces = 4;      // pairs
constexpr int kSplitMaxPieces1 = 8;     // single CTAs
constexpr int64_t kSplitMinBlocks = 4;
// Bytes of the split-K receive buffer ([S][2 ceil(bn/8 / S)][128 rows][16 B],
// kernel_tiled.cuh), which reuses the operand ring, and whether every S up to
// max_s fits a ring of ring_bytes.
GEMM_HD constexpr int split_recv_bytes(int bn, int s) { return s * 2 * ((bn / 8 + s - 1) / s) * 128 * 16; }
GEMM_HD constexpr bool split_recv_fits(int bn, int ring_bytes, int max_s) {
    for (int s = 2; s <= max_s; ++s)
        if (split_recv_bytes(bn, s) > ring_bytes) return false;
    return true;
}

inline int choose_ksplit(int64_t tiles, const int* clusters, int64_t k_blocks, int max_pieces = kSplitMaxPieces) {
#ifdef GEMM_SPLIT_PIECES
    // a build that fixes S (waves of clusters allowed), for measurements
    if (tiles > 0 && k_blocks >= kSplitMinBlocks * GEMM_SPLIT_PIECES) return GEMM_SPLIT_PIECES;
#endif
    for (int s = max_pieces; s >= 2; --s)
        if (tiles > 0 && tiles <= clusters[s] && k_blocks >= kSplitMinBlocks * s) return s;
    return 1;
}

// ------------------------------------------------------------------ small M
// Both small-M kernels compute D^T = B * A^T with the operands' roles
// swapped, so the 128-row MMA side runs over N (the weight rows) and the
// narrow MMA N side (MN = 16, 32 or 64) over M.
//
// Column-range kernel (the default).  N is cut into R ranges of `width` <= 128
// consecutive columns (B rows).  A range belongs to one cluster of P CTAs;
// CTA j of the cluster runs the j-th of P equal pieces of the K loop over the
// range's B rows, and the P fp32 partials are summed inside the cluster
// through distributed shared memory.  With P = 1 a CTA may own several
// ranges (persistent, one after the other).
// Accumulators per output block of the small-M kernel: with 4, MMA k of a K
// block adds into accumulator k (the epilogue adds the four in a fixed
// order).  Measured on GB300: 0.1 us faster at M <= 32 (16 x 8192 x 8192,
// fp16 and E4M3), 0.2 us slower at M = 64, where the epilogue's extra TMEM
// reads cost more than the MMAs gain.
#ifndef GEMM_SKINNY_ACCS
#define GEMM_SKINNY_ACCS 0   // 0: by MN as above
#endif
constexpr int skinny_accs(int mn) { return GEMM_SKINNY_ACCS != 0 ? GEMM_SKINNY_ACCS : (mn <= 32 ? 4 : 1); }

template <int MN_>
struct SkinnyConfig {
    static constexpr int MN = MN_;
    static constexpr int X_BYTES = MN * kStageRowBytes;    // activation (A) slot: MN rows
    // A B slot holds the range's `width` rows; slots are width * 128 bytes
    // rounded up to the 1024-byte swizzle atom, so narrow ranges pack more
    // stages (bytes in flight) into the ring.  The MMA reads 128 rows from a
    // slot's base: past a narrow slot it reads the next slot (or, for the last
    // one, the A slots and buffers behind the ring, all inside this CTA's
    // shared memory); those rows only feed TMEM lanes that are never used.
    static constexpr int MAX_STAGES = 32;   // ring stages (barrier pairs)
    static constexpr int MAX_ATOMS = 64;    // K blocks in flight (a stage holds one or more)
    // partials received from the cluster: [P][128 columns][MN / P rows] fp32 = MN * 128 fp32
    static constexpr int RECV_BYTES = MN * 128 * 4;
    static constexpr int NUM_BARS = 2 * MAX_STAGES + 5;
    // Each of the two accumulator buffers is ACCS MN-column accumulators
    // (MMA k of a K block adds into accumulator k % ACCS).
    static constexpr int ACCS = skinny_accs(MN);
    static_assert(ACCS == 1 || ACCS == 2 || ACCS == 4, "accumulators per block: 1, 2 or 4");
    static constexpr int ACC_COLS = ACCS * MN;
    static constexpr int TMEM_COLS = (2 * ACC_COLS < 32) ? 32 : 2 * ACC_COLS;
    // ring = [stages B slots][stages A slots], split at run time (ring_stages)
    static constexpr int RING_BYTES = (kMaxDynSmem - 1024 - RECV_BYTES - NUM_BARS * 8 - 16) / 1024 * 1024;
    static constexpr int OFF_RECV = RING_BYTES;
    static constexpr int OFF_BAR = OFF_RECV + RECV_BYTES;
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_SLOT + 16 + 1024;
    static_assert(X_BYTES % 1024 == 0, "activation tile must stay 1024-aligned");
    static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
    static_assert(RING_BYTES / (128 * kStageRowBytes + X_BYTES) >= 4, "at least four full-width stages");
    static_assert(RECV_BYTES + NUM_BARS * 8 >= 0, "layout");
    static_assert(MN == 16 || MN == 32 || MN == 64, "narrow side must be 16, 32 or 64");
    static_assert(SMEM_BYTES <= kMaxDynSmem, "shared memory budget exceeded");
};

// Stride of a B slot for ranges of `width` columns; a launch's ring holds
// min(MAX_ATOMS, RING_BYTES / (stride + X_BYTES)) K blocks, grouped into
// stages of skinny_stage_atoms() blocks.
GEMM_HD int skinny_w_stride(int width) { return (width * kStageRowBytes + 1023) / 1024 * 1024; }

// K blocks per ring stage for a ring of `atoms` K blocks: as many as leave at
// least three stages, at most 8.  Every stage costs a fixed ~0.18 us (its
// barrier round trip), each K block in it ~0.1 us more (its copies and four
// MMAs), so narrow ranges and 8-bit operands, whose K blocks are few bytes,
// need several per stage to keep up with HBM.
GEMM_HD int skinny_stage_atoms(int atoms) {
    const int a = atoms / 3;
    return a < 1 ? 1 : (a > 8 ? 8 : a);
}

using CfgSkinny16 = SkinnyConfig<16>;
using CfgSkinny32 = SkinnyConfig<32>;
using CfgSkinny64 = SkinnyConfig<64>;

// Largest cluster (K pieces per column range) of the column-range kernel.
constexpr int kSkinnyMaxPieces = 8;

struct SkinnyParams {
    int32_t M, N, K;
    int32_t k_blocks;
    int32_t width;            // columns per range (rows of a B box), 1..128
    int32_t ranges;           // R; range r covers columns [r * width, r * width + width) (clipped at N)
    int32_t pieces;           // P = CTAs per cluster; CTA j runs K blocks [j kb / P, (j + 1) kb / P)
    int32_t stages;           // ring stages, each stage_atoms B slots of w_stride bytes and as many A slots
    int32_t stage_atoms;      // K blocks (128-byte atoms of K) per ring stage
    int32_t w_stride;         // skinny_w_stride(width)
    void* D;                  // fp16 or bf16 [M][N]
    EpiParams epi;            // fused output transform (epi.on == 0: plain D = A B^T)
    uint32_t* status;
    uint64_t timeout_ns;
    int32_t stream_b;         // B is too large to stay in L2: load it evict-first
    uint32_t ab_format;       // operand format field of the MMA instruction descriptor
    int32_t prefetch_blocks;  // B blocks a CTA prefetches into L2 before its dependency wait
};

// Stream-K kernel (GEMM_VARIANT_SKINNY_STREAMK, and the no-allocation entry
// point).  The (n-tile, k-block) units are split into G contiguous ranges,
// one per CTA; tiles cut across ranges are summed in a fixed order, through a
// global-memory workspace, by the last CTA to finish one of their pieces.
template <int MN_>
struct StreamKConfig {
    static constexpr int MN = MN_;
    static constexpr int W_BYTES = 128 * kStageRowBytes;   // weight (B) tile: 128 rows
    static constexpr int X_BYTES = MN * kStageRowBytes;    // activation (A) tile: MN rows
    static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
    // This kernel streams B once and is bound by how many bytes are in flight,
    // so the ring takes every stage that fits beside the barriers (12 / 11 / 9).
    static constexpr int STAGES = (kMaxDynSmem - 2048) / STAGE_BYTES;
    static constexpr int TMEM_COLS = (2 * MN < 32) ? 32 : 2 * MN;
    static constexpr int OFF_W = 0;
    static constexpr int OFF_X = OFF_W + STAGES * W_BYTES;
    static constexpr int OFF_BAR = OFF_X + STAGES * X_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_SLOT + 16 + 1024;
    static_assert(X_BYTES % 1024 == 0, "activation tile must stay 1024-aligned");
    static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
    static_assert(STAGES >= 2, "at least a double-buffered ring");
    static_assert(MN == 16 || MN == 32 || MN == 64, "narrow side must be 16, 32 or 64");
    static_assert(SMEM_BYTES <= kMaxDynSmem, "shared memory budget exceeded");
};

using CfgStreamK16 = StreamKConfig<16>;
using CfgStreamK32 = StreamKConfig<32>;
using CfgStreamK64 = StreamKConfig<64>;

struct StreamKParams {
    int32_t M, N, K;
    int32_t n_tiles, k_blocks;
    int32_t num_ctas;         // G
    int32_t max_tiles_per_cta;
    int64_t units;            // n_tiles * k_blocks
    float* partials;          // [G][max_tiles_per_cta][MN][128] fp32
    uint32_t* counters;       // [n_tiles], zero between calls
    void* D;                  // fp16 or bf16 [M][N]
    EpiParams epi;            // fused output transform (epi.on == 0: plain D = A B^T)
    uint32_t* status;
    uint64_t timeout_ns;
    int32_t stream_b;         // B is too large to stay in L2: load it evict-first
    uint32_t ab_format;       // operand format field of the MMA instruction descriptor
};

// B of at least this many bytes is read once per call and cannot stay in the
// 129 MB L2 until the next one, so the small-M kernels stream it with an
// evict-first policy (keeping A and the fp32 partials in L2 instead).
constexpr int64_t kStreamBBytes = 96ll << 20;

// First unit of CTA c's range; CTA c owns [unit_begin(c), unit_begin(c+1)).
GEMM_HD int64_t unit_begin(int64_t c, int64_t units, int64_t G) { return div_nonneg(c * units, G); }

// The CTA whose range holds unit u.
GEMM_HD int64_t cta_of_unit(int64_t u, int64_t units, int64_t G) {
    return div_nonneg((u + 1) * G - 1, units);
}

}  // namespace gemm_gb300
