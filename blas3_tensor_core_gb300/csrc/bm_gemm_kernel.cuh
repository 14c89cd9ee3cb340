// bm_gemm_kernel.cuh -- persistent, warp-specialised BF16 GEMM / SYRK kernel for
// sm_103a (one CTA per SM; optionally a CTA pair per output tile).
//
//   C = alpha * op(A) * op(B) + beta * C      (GEMM)
//   C = alpha * op(A) * op(A)^T + beta * C    (SYRK, one triangle)
//
// This is the BLAS3 local compute of "BLASMp development notes" (section 1;
// stage B: SYRK's main compute is a GEMM), done with the staging ladder's last
// rung from "cp.async / ldmatrix ablation plan" (section 2.3: TMA with a
// multi-stage buffer, hardware 128-byte swizzle) and with the producer / MMA /
// accumulator-slot / epilogue roles that "fused A2A/GEMM Perfetto profile
// protocol" lists for its SM100/SM103 mainloop (MXFP8 hot-path table: load
// empty-stage acquire, TMA submission, MMA input-stage wait, reusable TMEM
// slot, MMA issue and stage release, epilogue).
//
// PAIR = 1: each CTA owns a 128 x BN output tile.
// PAIR = 2: a cluster of two CTAs on two SMs owns a 256 x BN tile. Each CTA
//   stages its own 128 rows of A and its own BN/2 rows of B; one
//   tcgen05.mma.cta_group::2 issued by CTA 0 reads both CTAs' shared memory and
//   writes 128 accumulator rows into each CTA's tensor memory. Per SM this
//   halves the B operand bytes that the tensor core reads from shared memory
//   per MMA (8 KB instead of 12 KB for a K = 16 step).
//
// Roles (320 threads per CTA):
//   warp 0, one lane  TMA producer: fills a STAGES-deep ring of shared-memory
//                     stages guarded by full/empty mbarriers (PAIR = 2: both
//                     CTAs' copies complete bytes on CTA 0's full barrier).
//   warp 1            MMA issuer (CTA 0 only; the warp waits, lane 0 issues):
//                     4 x tcgen05.mma (K = 16 each) per k-block, KPS k-blocks
//                     per stage, into one of two TMEM accumulators (128 lanes
//                     x BN fp32 columns per CTA); tcgen05.commit releases the
//                     stage (in both CTAs) and, at the end of a tile, signals
//                     the accumulator full. Warp 1 allocates and frees TMEM.
//   warps 2-9         epilogue, two warps per TMEM lane quadrant (warp w reads
//                     lanes 32 (w % 4) ..): TMEM -> registers (tcgen05.ld
//                     32x32b), alpha, then either a 128B-swizzled staging
//                     block stored by TMA (beta == 0 GEMM, split partials) or
//                     a transpose through shared memory with coalesced 16-byte
//                     loads of C (beta != 0) and stores; the SYRK triangle and
//                     the ragged edges of that path are masked per element.
// Tiles are handed out persistently (cluster c takes units c, c + clusters,
// ...), in grouped-raster order for GEMM and, for SYRK, over the referenced
// triangle only: the tiles across the diagonal first, then the inside tiles in
// groups of tile rows (tiles strictly on the other side of the diagonal are
// never visited).
//
// Every barrier wait is bounded: after the wait limit the thread records
// BM_ERR_TIMEOUT in the device status word and raises a shared abort flag that
// the other roles of its CTA poll; copies and MMAs in flight are waited for
// (again with a limit) and the CTA frees its tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "bm_ptx.cuh"

namespace bm {

enum : int { MODE_GEMM = 0, MODE_SYRK_LOWER = 1, MODE_SYRK_UPPER = 2 };
enum : int { EPI_FULL = 0, EPI_STORE = 1, EPI_COMBINE = 2 };  // epilogue paths compiled into a kernel copy
enum : int { DEV_ERR_TIMEOUT = 5 };

constexpr int CTA_M = 128;  // accumulator rows (TMEM lanes) per CTA
constexpr int TILE_K = 64;  // bf16 elements = 128 bytes = one swizzle row (a k-block)
constexpr int UMMA_K = 16;  // bf16 elements of one MMA = 32 bytes
// Operand element types: bf16 (kind::f16), FP8 E4M3 (kind::f8f6f4), or MXFP8:
// E4M3 with one UE8M0 scale per 32 elements of K (kind::mxf8f6f4, block-scaled).
// A k-block is 128 bytes of K in every case (64 bf16 or 128 FP8 elements) and one
// MMA consumes 32 bytes of K, so the shared-memory layout and descriptors are the
// same.
enum : int { ELEM_BF16 = 0, ELEM_E4M3 = 1, ELEM_MXF8 = 2 };
__host__ __device__ constexpr int kblock_elems(int elem) { return elem == ELEM_BF16 ? 64 : 128; }
// MXFP8 scale factors travel in atoms of 128 rows x 4 groups of 32 along K (one
// k-block): 512 bytes, byte (r % 32) * 16 + (r / 32) * 4 + g for row r and group
// g, the layout that tcgen05.cp 32x128b.warpx4 moves into tensor memory.
constexpr int SF_ATOM_BYTES = 512;
// Two epilogue warps per TMEM lane quadrant: warps w and w + 4 read the same 32
// accumulator rows and split the column chunks between them.
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int EPI_WARP_FLOATS = 32 * 32;  // one 32 x 32 fp32 staging block per epilogue warp
// The four warps of one half of the epilogue (one per quadrant) share their
// staging blocks as one 128-row x 128-byte block.
constexpr int GROUP_BLOCK_BYTES = 4 * EPI_WARP_FLOATS * 4;

struct GemmParams {
    int64_t m, n, k;   // output rows / columns (SYRK: m == n), reduction length
    void *C;
    int64_t ldc;
    float alpha, beta;
    int c_bf16;        // C element: 0 = fp32, 1 = bf16
    int a_mn_major;    // operand tiles in shared memory: 0 = K-major, 1 = M/N-major
    int b_mn_major;
    int mode;          // MODE_*
    int64_t tiles_m, tiles_n;
    int64_t num_tiles;  // GEMM: tiles_m * tiles_n; SYRK: tiles touching the triangle
    int64_t full_tiles; // tiles [0, full_tiles) run whole; each later tile is split k_splits (or n_split) ways
    int64_t num_units;  // full_tiles + (num_tiles - full_tiles) * (k_splits or n_split)
    int k_splits;       // > 1: split units write fp32 partials, summed in this kernel (fixup) or by a second one
    int n_split;        // 2: each later tile runs as two units of half its columns (256 x 256 pair
                        // tiles of GEMM only; MMA N = 128, no partial sums); k_splits is then 1
    int kb_per_split;   // k-blocks (128 bytes of K each) per split
    int kb_total;       // ceil(k / elements per k-block)
    int group_m;        // grouped raster: tile rows per group
    float *partial;     // [split tile][split][tile rows][tile columns] fp32 when k_splits > 1
    int *status;       // device status word (first error wins)
    uint64_t timeout_ns;
    int debug_stall;   // test hook: the first stage's copy is never issued
    int tma_c;         // tmC maps C for the epilogue's TMA copies (128B swizzle, box 128 bytes x
                       // 32 rows for per-warp stores when beta == 0, x 128 rows for the group
                       // load-combine-store when beta != 0)
    int syr2k_kb;      // SYR2K: k-blocks of one product; later k-blocks swap the roles of tmA and tmB
    int store_p_tma;   // split units: tmP maps the partial slots for TMA stores (fp32, box 32 x 32, 128B swizzle)
    int a_box3;        // tmA is a stage box: one 3-D copy brings a CTA's A tile for a whole stage
    int b_box3;        // same for tmB
    // In-kernel split-K reduction: split units run first; per epilogue warp region
    // of a split tile, the last of the k_splits units to store its partial sums the
    // slots and writes C (no reduce kernel). Counters are (seq << 16 | arrivals).
    int fixup;
    unsigned long long *fixup_ctr;  // split tiles x PAIR x NUM_EPI_WARPS counters
    unsigned long long seq;         // this launch's tag, 1 .. 2^48 - 1
    // MXFP8: tmSA / tmSB map the scale atoms of A and B as (256 bytes, 2, k-block,
    // 128-row block), one box of KPS k-blocks per stage.
};

// KPS: k-blocks per ring stage. With two k-blocks a stage, the MMA thread waits
// on a full barrier and commits once per 8 MMAs instead of once per 4; every
// such handshake leaves the tensor pipe idle for a while, so this pays wherever
// the ring still holds three stages.
//
// Stage layout (one CTA): the A tile of each k-block, then the B tile of each
// k-block. A K-major tile is rows x 128 bytes (8-row swizzle atoms, 1024 bytes
// apart); k-block s of it starts s tile sizes in. An M/N-major tile is split
// into chunks of 64 rows of M or N; chunk c holds the 64 x KPS k-rows of all
// the stage's k-blocks (128 bytes each), so k-block s starts 8 KB into it and
// the chunks are KPS x 8 KB apart. A 3-D "stage box" copy writes exactly this
// layout for a whole operand and stage; without one, each k-block (and chunk)
// is copied with a 2-D box into its place.
template <int BN, int STAGES, int PAIR, int ELEM, int KPS>
struct KernelCfg {
    static constexpr int TILE_M = CTA_M * PAIR;  // output rows per tile
    static constexpr int KB_ELEMS = kblock_elems(ELEM);  // K elements per k-block (128 bytes)
    static constexpr int B_ROWS = BN / PAIR;     // rows of op(B)^T staged by each CTA
    static constexpr int A_BYTES = CTA_M * TILE_K * 2;  // 128 rows x 128 bytes of K, any element type
    static constexpr int B_BYTES = B_ROWS * TILE_K * 2;
    static constexpr int STAGE_BYTES = KPS * (A_BYTES + B_BYTES);
    static constexpr int B_OFFSET = KPS * A_BYTES;       // B tiles follow the stage's A tiles
    static constexpr int CHUNK_BYTES = KPS * 8192;      // one 64-row M/N chunk of all k-blocks of a stage
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    // MXFP8 scale factors per k-block: this CTA's A atom (its 128 rows) and the B
    // atoms of all BN rows of the tile (each CTA of a pair holds all of them), in
    // shared memory after the ring and, for the MMAs, in tensor memory after the two
    // accumulators: four 32-bit columns per atom, one slot per ring k-block.
    static constexpr bool SCALED = ELEM == ELEM_MXF8;
    static constexpr int SF_B_ATOMS = BN / 128;
    static constexpr int SF_KB_BYTES = SCALED ? SF_ATOM_BYTES * (1 + SF_B_ATOMS) : 0;
    static constexpr int SF_STAGE_BYTES = KPS * SF_KB_BYTES;
    // (rounded up to 1 KB: the epilogue staging blocks that follow are 128B-swizzled
    // TMA sources and must start on 1024-byte boundaries)
    static constexpr int SF_BYTES = (STAGES * SF_STAGE_BYTES + 1023) / 1024 * 1024;
    static constexpr int SF_KB_COLS = SCALED ? 4 * (1 + SF_B_ATOMS) : 0;
    // Two accumulators (the epilogue drains one while the MMAs fill the other),
    // except for 256-wide MXFP8 tiles: two 256-column accumulators fill the tensor
    // memory, so those tiles use one and the next tile's MMAs wait until the
    // epilogue has read it (its stores still overlap the next mainloop).
    static constexpr int NUM_ACC = (SCALED && BN == 256) ? 1 : 2;
    static constexpr int ACC_COLS = NUM_ACC * BN;
    static constexpr int EPI_BYTES = NUM_EPI_WARPS * EPI_WARP_FLOATS * 4;
    // full, empty, acc full x2, acc empty x2, drain, C load x2 (one per epilogue half)
    static constexpr int NUM_BARS = 2 * STAGES + 7;
    static constexpr int BAR_BYTES = 8 * NUM_BARS + 16;
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + SF_BYTES + EPI_BYTES + BAR_BYTES;
    // allocation: a power of two of at least 32 columns
    static constexpr int TMEM_COLS = SCALED ? 512 : ACC_COLS;
    static_assert(BN == 128 || BN == 256, "BN");
    static_assert(PAIR == 1 || PAIR == 2, "PAIR");
    static_assert(KPS == 1 || KPS == 2, "k-blocks per stage");
    static_assert(B_ROWS % 64 == 0, "B rows per CTA");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert((RING_BYTES + SF_BYTES) % 1024 == 0 && EPI_WARP_FLOATS * 4 % 1024 == 0, "swizzled staging alignment");
    static_assert(!SCALED || ACC_COLS + STAGES * KPS * SF_KB_COLS <= TMEM_COLS, "tensor memory");
};

// ---------------------------------------------------------------- scheduling
struct Unit {
    int64_t tm, tn;
    int kb0, kb1;     // k-blocks of this unit
    int64_t slot;     // partial-sum slot (split units only), -1 for a whole tile
    int nh;           // N half of a tile split along N (0 or 1), -1 otherwise
};

// Does tile (tm, tn) (TM x BN) lie entirely in the referenced SYRK triangle?
template <int TM, int BN>
__host__ __device__ inline bool tile_inside_triangle(int mode, int64_t tm, int64_t tn)
{
    if (mode == MODE_SYRK_LOWER) return tm * TM >= (tn + 1) * BN - 1;  // smallest row >= largest column
    if (mode == MODE_SYRK_UPPER) return (tm + 1) * TM - 1 <= tn * BN;  // largest row <= smallest column
    return true;
}

// SYRK tile order in closed form. The tile shapes used (TM = BN, or BN = 2 TM)
// give every tile row tm exactly one tile across the diagonal, in tile column
// tm / Q with Q = BN / TM; the tiles strictly inside the triangle are, per row,
// the columns left of it (lower) or right of it (upper). syrk_inside_before(R)
// counts the inside tiles of rows [0, R).
template <int TM, int BN>
__host__ __device__ inline int64_t syrk_inside_before(int mode, int64_t R, int64_t tiles_n)
{
    constexpr int Q = BN / TM;
    static_assert(Q == 1 || Q == 2, "tile shapes with one diagonal tile per row");
    // sum over r < R of floor(r / Q)
    const int64_t h = R >> 1;
    const int64_t diag = Q == 1 ? R * (R - 1) / 2 : h * (h - 1) + (R & 1) * h;
    return mode == MODE_SYRK_LOWER ? diag : R * (tiles_n - 1) - diag;
}

// Inside tiles of a lower triangle of square tiles ((r, c) with c < r < T), in
// groups of SYRK_GROUP tile rows: group g holds rows [r0, r0 + gs), r0 = g G, and
// runs column by column, c = 0 .. r0 + gs - 2, each column's rows
// max(r0, c + 1) .. r0 + gs - 1 in order. While about one wave of tiles is in
// flight, the A panels it reads are the group's 16 row panels and a few column
// panels, so they stay in L2 beside the streaming C (row-by-row order re-read
// panels from DRAM; measured at 8192 x 4096, beta = 1: 171.3 -> 168.3 us, while
// groups of 4, 8, 24 and 32 rows gained nothing).
constexpr int64_t SYRK_GROUP = 16;

// inside tiles of the (full) groups before group g
__host__ __device__ inline int64_t syrk_group_prefix(int64_t g)
{
    constexpr int64_t G = SYRK_GROUP;
    return G * G * g * (g - 1) / 2 + g * (G * (G - 1) / 2);
}

// Inside tile v of the grouped lower order -> (r, c), in closed form: the group
// inverts the quadratic prefix above and the column inside the group's triangle
// (columns r0 + j of gs - 1 - j tiles) another quadratic; each from a square-root
// estimate and an exact integer correction of a step or two. The estimates are
// single precision: the integer steps make the result exact, and double-precision
// arithmetic is slow on this GPU (with it, the SYRK schedule cost 2.6 us per
// 8192 x 4096 call on the MMA and producer warps at the tile boundaries).
__host__ __device__ inline void syrk_lower_grouped(int64_t T, int64_t v, int64_t &r, int64_t &c)
{
    constexpr int64_t G = SYRK_GROUP;
    const int64_t groups = (T + G - 1) / G;
    int64_t g = static_cast<int64_t>((1.0f + sqrtf(1.0f + 8.0f * static_cast<float>(v))) / (2.0f * G));
    g = g < 0 ? 0 : (g > groups - 1 ? groups - 1 : g);
    while (g + 1 < groups && syrk_group_prefix(g + 1) <= v) ++g;
    while (g > 0 && syrk_group_prefix(g) > v) --g;
    const int64_t r0 = g * G;
    const int64_t gs = T - r0 < G ? T - r0 : G;
    int64_t local = v - syrk_group_prefix(g);
    if (local < r0 * gs) {  // columns left of the group: all gs rows each
        c = local / gs;
        r = r0 + local % gs;
        return;
    }
    local -= r0 * gs;
    // tiles before column r0 + j of the group's own triangle: S(j) = j (gs - 1) - j (j - 1) / 2
    const float b = static_cast<float>(gs) - 0.5f;
    const float disc = b * b - 2.0f * static_cast<float>(local);
    int64_t j = static_cast<int64_t>(b - sqrtf(disc > 0.0f ? disc : 0.0f));
    j = j < 0 ? 0 : (j > gs - 2 ? gs - 2 : j);
    while (j + 1 <= gs - 2 && (j + 1) * (gs - 1) - (j + 1) * j / 2 <= local) ++j;
    while (j > 0 && j * (gs - 1) - j * (j - 1) / 2 > local) --j;
    c = r0 + j;
    r = c + 1 + (local - (j * (gs - 1) - j * (j - 1) / 2));
}

// Tile t of the SYRK schedule -> (tile row, tile column). The tiles_m tiles
// across the diagonal come first (their epilogue masks each element and is
// slower, so it should overlap later tiles' mainloops rather than end the
// kernel), one per row; then the tiles inside the triangle. Square tiles take
// the grouped order above (the upper triangle its transpose: groups of 16 tile
// columns, each row by row). 128 x 256 tiles go row by row: the row of an
// inside tile inverts the quadratic count syrk_inside_before, a square-root
// estimate, then an exact integer correction of a step or two.
template <int TM, int BN>
__host__ __device__ inline void syrk_tile_coords(int mode, int64_t tiles_m, int64_t tiles_n, int64_t t, int64_t &tm,
                                                 int64_t &tn)
{
    constexpr int Q = BN / TM;
    if (t < tiles_m) {
        tm = t;
        tn = t / Q;
        return;
    }
    const int64_t v = t - tiles_m;
    if constexpr (Q == 1) {
        int64_t r, c;
        syrk_lower_grouped(tiles_m, v, r, c);
        tm = mode == MODE_SYRK_LOWER ? r : c;
        tn = mode == MODE_SYRK_LOWER ? c : r;
        return;
    }
    float est;  // (single precision, as above)
    if (mode == MODE_SYRK_LOWER) {
        // lower: about R^2 / (2 Q) inside tiles before row R
        est = 1.0f + 2.0f * sqrtf(static_cast<float>(v));
    } else {
        // upper: about R (T - 1/2) - R^2 / (2 Q) before row R, T = tiles_n
        const float b = static_cast<float>(tiles_n) - 0.5f;
        const float disc = b * b - 2.0f * static_cast<float>(v) / Q;
        est = Q * (b - sqrtf(disc > 0.0f ? disc : 0.0f));
    }
    int64_t r = static_cast<int64_t>(est);
    r = r < 0 ? 0 : (r > tiles_m - 1 ? tiles_m - 1 : r);
    while (r + 1 < tiles_m && syrk_inside_before<TM, BN>(mode, r + 1, tiles_n) <= v) ++r;
    while (r > 0 && syrk_inside_before<TM, BN>(mode, r, tiles_n) > v) --r;
    tm = r;
    const int64_t local = v - syrk_inside_before<TM, BN>(mode, r, tiles_n);
    tn = mode == MODE_SYRK_LOWER ? local : r / Q + 1 + local;
}

// Kernel copies that can run SYRK: bf16 operands with every epilogue path. The
// others (GEMM-only copies, FP8) leave the triangle order out.
__host__ __device__ constexpr bool syrk_capable(int elem, int epi) { return elem == ELEM_BF16 && epi == EPI_FULL; }

// Tile t -> (tile row, tile column): grouped raster for GEMM, the closed-form
// triangle order above for SYRK.
template <int TM, int BN, bool SYRK = true>
__device__ __forceinline__ void tile_coords(const GemmParams &p, int64_t t, int64_t &tm, int64_t &tn)
{
    tm = 0;
    tn = 0;
    if (p.mode == MODE_GEMM) {
        const int64_t per_group = static_cast<int64_t>(p.group_m) * p.tiles_n;
        const int64_t g = t / per_group;
        const int64_t first = g * p.group_m;
        const int64_t rows = (p.tiles_m - first) < p.group_m ? (p.tiles_m - first) : p.group_m;
        const int64_t local = t - g * per_group;
        tm = first + local % rows;
        tn = local / rows;
    } else if constexpr (SYRK && (BN == TM || BN == 2 * TM)) {
        // (the 256 x 128 MXFP8 tiles never run SYRK)
        syrk_tile_coords<TM, BN>(p.mode, p.tiles_m, p.tiles_n, t, tm, tn);
    }
}

// Output column of accumulator column j (a multiple of 32) of a unit whose tile
// starts at column col0. A whole tile maps j to col0 + j. A half unit (nh >= 0;
// 256-wide tiles on SM pairs) ran its MMAs with N = BN / 2 over rows nh * BN / 4 ..
// of each CTA's half of the tile's B rows, so its columns [0, BN / 4) are tile
// columns nh * BN / 4 + [0, BN / 4) and the rest lie BN / 2 further on.
template <int BN, int PAIR = 2>
__device__ __forceinline__ int64_t unit_col(int64_t col0, int nh, int j)
{
    if constexpr (!(PAIR == 2 && BN == 256)) return col0 + j;  // no half units in other copies
    if (nh < 0) return col0 + j;
    constexpr int q = BN / 4;
    return col0 + static_cast<int64_t>(j / q) * (BN / 2) + nh * q + (j % q);
}

// Work unit u: a whole tile, one K range of a split tile, or one N half of a
// tile split along N. With the reduce kernel (and with N halves) the split
// units come last, so with units handed out round-robin they fill the
// otherwise partly idle last wave. With the in-kernel reduction they
// come first: the reduction then runs in the epilogue while the next tile's
// mainloop proceeds, instead of after the last wave.
template <int TM, int BN, bool SYRK = true>
__device__ __forceinline__ Unit map_unit(const GemmParams &p, int64_t u)
{
    Unit r;
    int64_t t;
    r.nh = -1;
    if (p.n_split > 1) {
        // whole tiles first; then the two N halves of each later tile, one unit each
        const int64_t v = u - p.full_tiles;
        t = v < 0 ? u : p.full_tiles + (v >> 1);
        r.nh = v < 0 ? -1 : static_cast<int>(v & 1);
        r.kb0 = 0;
        r.kb1 = p.kb_total;
        r.slot = -1;
    } else {
        const int64_t split_units = p.num_units - p.full_tiles;
        const bool whole = p.fixup ? u >= split_units : u < p.full_tiles;
        if (whole) {
            t = p.fixup ? u - split_units : u;
            r.kb0 = 0;
            r.kb1 = p.kb_total;
            r.slot = -1;
        } else {
            const int64_t v = p.fixup ? u : u - p.full_tiles;
            const int64_t local = v / p.k_splits;
            const int split = static_cast<int>(v - local * p.k_splits);
            t = p.full_tiles + local;
            r.kb0 = split * p.kb_per_split;
            r.kb1 = min(p.kb_total, r.kb0 + p.kb_per_split);
            r.slot = p.k_splits > 1 ? v : -1;
        }
    }
    tile_coords<TM, BN, SYRK>(p, t, r.tm, r.tn);
    return r;
}

template <int PAIR>
__device__ __forceinline__ int64_t first_unit()
{
    if constexpr (PAIR == 1) return blockIdx.x;
    else return cluster_index();
}

template <int PAIR>
__device__ __forceinline__ int64_t unit_stride()
{
    if constexpr (PAIR == 1) return gridDim.x;
    else return cluster_count();
}

// ---------------------------------------------------------------- bounded waits
__device__ __noinline__ void signal_timeout(const GemmParams &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (p.status != nullptr) atomicCAS(p.status, 0, DEV_ERR_TIMEOUT);
}

template <bool CLUSTER>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    if constexpr (CLUSTER) return mbar_try_wait_cluster(bar, parity);
    else return mbar_try_wait(bar, parity);
}

// Single-thread wait: false when the limit passes or another role aborted.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int *abort_flag, uint64_t limit_ns)
{
    if (try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (try_wait<CLUSTER>(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Warp-uniform wait: every lane observes the phase (acquire) before any lane
// proceeds, and all lanes take the same exit.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag, uint64_t limit_ns)
{
    uint64_t t0 = 0;
    for (int it = 0;; ++it) {
        const bool ok = try_wait<CLUSTER>(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if (it == 0) t0 = global_timer_ns();
        if ((it & 15) == 15) {
            const bool stop = *abort_flag != 0 || (global_timer_ns() - t0 > limit_ns);
            if (__any_sync(0xffffffffu, stop)) return false;
        }
    }
}

__device__ __forceinline__ void spin_ns(uint64_t ns)
{
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

// ---------------------------------------------------------------- output
__device__ __forceinline__ bool in_output(const GemmParams &p, int64_t i, int64_t j)
{
    if (i >= p.m || j >= p.n) return false;
    if (p.mode == MODE_SYRK_LOWER) return i >= j;
    if (p.mode == MODE_SYRK_UPPER) return i <= j;
    return true;
}

// C[i, j..j+3] = v + beta * C (C read only when beta != 0), masked per element.
// j is a multiple of 4; C and ldc satisfy the 16-byte rule, so the vector
// accesses are aligned.
__device__ __forceinline__ void write_c4(const GemmParams &p, int64_t i, int64_t j, float v[4])
{
    bool all = (i < p.m) && (j + 3 < p.n);
    if (p.mode == MODE_SYRK_LOWER) all = all && (i >= j + 3);
    if (p.mode == MODE_SYRK_UPPER) all = all && (i <= j);
    const bool use_beta = p.beta != 0.0f;
    if (p.c_bf16) {
        __nv_bfloat16 *row = reinterpret_cast<__nv_bfloat16 *>(p.C) + i * p.ldc;
        if (all) {
            if (use_beta) {
                const uint2 old = *reinterpret_cast<const uint2 *>(row + j);
                const __nv_bfloat162 o01 = *reinterpret_cast<const __nv_bfloat162 *>(&old.x);
                const __nv_bfloat162 o23 = *reinterpret_cast<const __nv_bfloat162 *>(&old.y);
                v[0] = fmaf(p.beta, __low2float(o01), v[0]);
                v[1] = fmaf(p.beta, __high2float(o01), v[1]);
                v[2] = fmaf(p.beta, __low2float(o23), v[2]);
                v[3] = fmaf(p.beta, __high2float(o23), v[3]);
            }
            const __nv_bfloat162 r01 = __floats2bfloat162_rn(v[0], v[1]);
            const __nv_bfloat162 r23 = __floats2bfloat162_rn(v[2], v[3]);
            uint2 out;
            out.x = *reinterpret_cast<const uint32_t *>(&r01);
            out.y = *reinterpret_cast<const uint32_t *>(&r23);
            *reinterpret_cast<uint2 *>(row + j) = out;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (!in_output(p, i, j + e)) continue;
                float x = v[e];
                if (use_beta) x = fmaf(p.beta, __bfloat162float(row[j + e]), x);
                row[j + e] = __float2bfloat16_rn(x);
            }
        }
    } else {
        float *row = reinterpret_cast<float *>(p.C) + i * p.ldc;
        if (all) {
            if (use_beta) {
                const float4 old = *reinterpret_cast<const float4 *>(row + j);
                v[0] = fmaf(p.beta, old.x, v[0]);
                v[1] = fmaf(p.beta, old.y, v[1]);
                v[2] = fmaf(p.beta, old.z, v[2]);
                v[3] = fmaf(p.beta, old.w, v[3]);
            }
            *reinterpret_cast<float4 *>(row + j) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (!in_output(p, i, j + e)) continue;
                float x = v[e];
                if (use_beta) x = fmaf(p.beta, row[j + e], x);
                row[j + e] = x;
            }
        }
    }
}

// Out-of-line masked store for vectors on a ragged edge or the SYRK diagonal;
// keeps the epilogue's unrolled fast path small.
__device__ __noinline__ void write_c4_edge(const GemmParams &p, int64_t i, int64_t j, float4 v4)
{
    float v[4] = {v4.x, v4.y, v4.z, v4.w};
    write_c4(p, i, j, v);
}

// write_c4 for a full, unmasked 4-vector whose old C value was loaded earlier
// (raw bits: fp32 -> 4 words; bf16 -> words x, y hold 4 values).
__device__ __forceinline__ void write_c4_preloaded(const GemmParams &p, int64_t i, int64_t j, float v[4],
                                                   uint4 old)
{
    if (p.c_bf16) {
        const __nv_bfloat162 o01 = *reinterpret_cast<const __nv_bfloat162 *>(&old.x);
        const __nv_bfloat162 o23 = *reinterpret_cast<const __nv_bfloat162 *>(&old.y);
        v[0] = fmaf(p.beta, __low2float(o01), v[0]);
        v[1] = fmaf(p.beta, __high2float(o01), v[1]);
        v[2] = fmaf(p.beta, __low2float(o23), v[2]);
        v[3] = fmaf(p.beta, __high2float(o23), v[3]);
        const __nv_bfloat162 r01 = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 r23 = __floats2bfloat162_rn(v[2], v[3]);
        uint2 out;
        out.x = *reinterpret_cast<const uint32_t *>(&r01);
        out.y = *reinterpret_cast<const uint32_t *>(&r23);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.C) + i * p.ldc + j) = out;
    } else {
        v[0] = fmaf(p.beta, __uint_as_float(old.x), v[0]);
        v[1] = fmaf(p.beta, __uint_as_float(old.y), v[1]);
        v[2] = fmaf(p.beta, __uint_as_float(old.z), v[2]);
        v[3] = fmaf(p.beta, __uint_as_float(old.w), v[3]);
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.C) + i * p.ldc + j) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

// Two bf16 outputs from two fp32 accumulators and two old bf16 values (packed,
// low half first): beta * c + alpha * acc in fp32, rounded to nearest even.
// A bf16 value is the upper 16 bits of the fp32 with the same value.
__device__ __forceinline__ uint32_t combine_bf16x2(const GemmParams &p, uint32_t acc0, uint32_t acc1, uint32_t old)
{
    const float v0 = fmaf(p.beta, __uint_as_float(old << 16), p.alpha * __uint_as_float(acc0));
    const float v1 = fmaf(p.beta, __uint_as_float(old & 0xFFFF0000u), p.alpha * __uint_as_float(acc1));
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    return static_cast<uint32_t>(__bfloat16_as_ushort(h.x)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h.y)) << 16);
}

__device__ __forceinline__ uint32_t combine_f32(const GemmParams &p, uint32_t acc, uint32_t old)
{
    return __float_as_uint(fmaf(p.beta, __uint_as_float(old), p.alpha * __uint_as_float(acc)));
}

// One lane's row of a 32-row x 128-byte staging block, 128B-swizzled (16-byte
// unit u of row r at slot u ^ (r & 7)): 64 accumulator columns as bf16, or 32
// as fp32, times alpha when SCALE.
template <bool SCALE>
__device__ __forceinline__ void stage_row_bf16(uint4 *srow, const uint32_t (&r)[64], float alpha, int lane)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(r[8 * j + 2 * e]);
            const float x1 = __uint_as_float(r[8 * j + 2 * e + 1]);
            h[e] = SCALE ? __floats2bfloat162_rn(alpha * x0, alpha * x1) : __floats2bfloat162_rn(x0, x1);
        }
        srow[j ^ (lane & 7)] = *reinterpret_cast<const uint4 *>(h);
    }
}

// 64 fp32 accumulator values of a row (times alpha) as 32 packed bf16 pairs, in
// column order (the lower half of each word is the even column).
template <bool SCALE>
__device__ __forceinline__ void pack_row_bf16(uint32_t (&h)[32], const uint32_t (&r)[64], float alpha)
{
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float x0 = __uint_as_float(r[2 * i]);
        const float x1 = __uint_as_float(r[2 * i + 1]);
        const __nv_bfloat162 b = SCALE ? __floats2bfloat162_rn(alpha * x0, alpha * x1) : __floats2bfloat162_rn(x0, x1);
        h[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
}

// 32 fp32 accumulator values (times alpha) as 16 packed bf16 pairs, in column order.
template <bool SCALE>
__device__ __forceinline__ void pack_32_bf16(uint32_t *h, const uint32_t (&r)[32], float alpha)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float x0 = __uint_as_float(r[2 * i]);
        const float x1 = __uint_as_float(r[2 * i + 1]);
        const __nv_bfloat162 b = SCALE ? __floats2bfloat162_rn(alpha * x0, alpha * x1) : __floats2bfloat162_rn(x0, x1);
        h[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
}

// A row of 32 packed bf16 pairs (128 bytes) into the 128B-swizzled staging block:
// 16-byte unit j of row `lane` goes to slot j ^ (lane & 7).
__device__ __forceinline__ void stage_row_packed(uint4 *srow, const uint32_t (&h)[32], int lane)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) srow[j ^ (lane & 7)] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
}

template <bool SCALE>
__device__ __forceinline__ void stage_row_f32(uint4 *srow, const uint32_t (&r)[64], float alpha, int lane)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 q = make_uint4(r[4 * j + 0], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        if (SCALE)
            q = make_uint4(__float_as_uint(alpha * __uint_as_float(q.x)), __float_as_uint(alpha * __uint_as_float(q.y)),
                           __float_as_uint(alpha * __uint_as_float(q.z)), __float_as_uint(alpha * __uint_as_float(q.w)));
        srow[j ^ (lane & 7)] = q;
    }
}

// Is C[i, j..j+3] a full vector inside the output (no edge, no triangle mask)?
__device__ __forceinline__ bool full_vector(const GemmParams &p, int64_t i, int64_t j)
{
    bool all = (i < p.m) && (j + 3 < p.n);
    if (p.mode == MODE_SYRK_LOWER) all = all && (i >= j + 3);
    if (p.mode == MODE_SYRK_UPPER) all = all && (i <= j);
    return all;
}

// Does the 32 x 32 block at rows r0.., columns c0.. lie wholly outside the
// referenced SYRK triangle (lower: every column > every row; upper: the mirror)?
__device__ __forceinline__ bool block_outside_triangle(int mode, int64_t r0, int64_t c0)
{
    if (mode == MODE_SYRK_LOWER) return r0 + 31 < c0;
    if (mode == MODE_SYRK_UPPER) return r0 > c0 + 31;
    return false;
}

// Does C[i, j..j+3] lie wholly outside the referenced SYRK triangle?
__device__ __forceinline__ bool vector_outside_triangle(int mode, int64_t i, int64_t j)
{
    if (mode == MODE_SYRK_LOWER) return j > i;
    if (mode == MODE_SYRK_UPPER) return j + 3 < i;
    return false;
}

// ---------------------------------------------------------------- in-kernel split-K reduction
// One arrival at a region counter. The value is (tag << 16) | arrivals; a tag
// other than this launch's (a reset counter, a launch that stopped early, or
// workspace bytes left by other use) counts as no arrivals yet. Returns this
// arrival's number, 1 .. k_splits. Each failed compare-and-swap means another
// arrival went in, so the loop ends within k_splits attempts.
__device__ __forceinline__ int fixup_arrive(unsigned long long *ctr, unsigned long long seq, int k_splits)
{
    unsigned long long cur = atomicAdd(ctr, 0ull);
    for (int i = 0; i <= k_splits; ++i) {
        const int n = (cur >> 16) == seq ? static_cast<int>(cur & 0xFFFFull) + 1 : 1;
        const unsigned long long want = (seq << 16) | static_cast<unsigned long long>(n);
        const unsigned long long prev = atomicCAS(ctr, cur, want);
        if (prev == cur) return n;
        cur = prev;
    }
    return 0;
}

// A full 4-vector of C (no edge, no triangle mask) from its final value: cast
// and store, no beta term.
__device__ __forceinline__ void store_c4(const GemmParams &p, int64_t i, int64_t j, float4 v)
{
    if (p.c_bf16) {
        const __nv_bfloat162 r01 = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 r23 = __floats2bfloat162_rn(v.z, v.w);
        uint2 out;
        out.x = *reinterpret_cast<const uint32_t *>(&r01);
        out.y = *reinterpret_cast<const uint32_t *>(&r23);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.C) + i * p.ldc + j) = out;
    } else {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.C) + i * p.ldc + j) = v;
    }
}

// beta * c + v for a full 4-vector whose old C value (bf16 or fp32 bits) was loaded earlier.
__device__ __forceinline__ float4 add_beta_c4(const GemmParams &p, float4 v, uint4 old)
{
    if (p.c_bf16) {
        v.x = fmaf(p.beta, __uint_as_float(old.x << 16), v.x);
        v.y = fmaf(p.beta, __uint_as_float(old.x & 0xFFFF0000u), v.y);
        v.z = fmaf(p.beta, __uint_as_float(old.y << 16), v.z);
        v.w = fmaf(p.beta, __uint_as_float(old.y & 0xFFFF0000u), v.w);
    } else {
        v.x = fmaf(p.beta, __uint_as_float(old.x), v.x);
        v.y = fmaf(p.beta, __uint_as_float(old.y), v.y);
        v.z = fmaf(p.beta, __uint_as_float(old.z), v.z);
        v.w = fmaf(p.beta, __uint_as_float(old.w), v.w);
    }
    return v;
}

// Called by an epilogue warp once its 32 rows x (BN / 2) columns of a split
// unit's partial are stored (plain stores). The last of the tile's k_splits
// units to get here sums that region over the slots in split order and writes
// C; the others return at once. Nothing waits. With beta != 0 the unit of
// split 0 has already added beta * C to its partial at every full 4-vector
// (it read C before it counted itself in, so before anyone writes C); only
// the vectors at the edges of C take beta here.
template <int TM, int BN, int PAIR>
__device__ __forceinline__ void fixup_region(const GemmParams &p, int64_t tm, int64_t tn, int64_t slot, uint32_t rank,
                                             int quad, int half, int warp, int lane)
{
    const int64_t local = slot / p.k_splits;
    unsigned long long *ctr = p.fixup_ctr + (local * PAIR + rank) * NUM_EPI_WARPS + (warp - 2);
    __threadfence();  // this lane's partial stores, before the arrival (release)
    __syncwarp();
    int n = 0;
    if (lane == 0) {
        __threadfence();
        n = fixup_arrive(ctr, p.seq, p.k_splits);
        if (n == p.k_splits) atomicExch(ctr, 0ull);  // every arrival is in: reset for the next launch
    }
    n = __shfl_sync(0xffffffffu, n, 0);
    if (n != p.k_splits) return;
    __threadfence();  // the other units' partials, after the arrivals (acquire)
    const int row_in_tile = static_cast<int>(rank) * CTA_M + quad * 32;
    const int64_t row0 = tm * TM + row_in_tile;
    const int64_t col0 = tn * BN;
    const int64_t slot_elems = static_cast<int64_t>(TM) * BN;
    const float *base = p.partial + local * p.k_splits * slot_elems + static_cast<int64_t>(row_in_tile) * BN;
    const int cc = lane & 7;
#pragma unroll 1
    for (int ch = half; ch < BN / 32; ch += 2) {
        // 8 lanes cover one 32-column row segment, 4 rows per step, as in the stores
        const int64_t off = static_cast<int64_t>(lane >> 3) * BN + ch * 32 + cc * 4;
        float4 acc[8];
#pragma unroll
        for (int step = 0; step < 8; ++step)
            acc[step] = __ldcg(reinterpret_cast<const float4 *>(base + off + step * 4 * BN));
#pragma unroll 1
        for (int sp = 1; sp < p.k_splits; ++sp) {
            const float *src = base + sp * slot_elems + off;
            float4 t[8];
#pragma unroll
            for (int step = 0; step < 8; ++step) t[step] = __ldcg(reinterpret_cast<const float4 *>(src + step * 4 * BN));
#pragma unroll
            for (int step = 0; step < 8; ++step) {
                acc[step].x += t[step].x;
                acc[step].y += t[step].y;
                acc[step].z += t[step].z;
                acc[step].w += t[step].w;
            }
        }
        const int64_t gj = col0 + ch * 32 + cc * 4;
#pragma unroll
        for (int step = 0; step < 8; ++step) {
            const int64_t gi = row0 + step * 4 + (lane >> 3);
            if (gi >= p.m || gj >= p.n) continue;
            if (full_vector(p, gi, gj)) {
                store_c4(p, gi, gj, acc[step]);
            } else {
                float v[4] = {acc[step].x, acc[step].y, acc[step].z, acc[step].w};
                write_c4(p, gi, gj, v);
            }
        }
    }
}

// ---------------------------------------------------------------- roles
// One operand tile copy: 2-D box (x, y) into dst, CTA-local or counted on the
// pair's barrier.
template <int PAIR>
__device__ __forceinline__ void load_box(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x, int32_t y)
{
    if constexpr (PAIR == 1) tma_load_2d(dst, map, bar, x, y);
    else tma_load_2d_pair(dst, map, bar, x, y);
}

template <int PAIR>
__device__ __forceinline__ void load_box3(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x, int32_t y,
                                          int32_t z)
{
    if constexpr (PAIR == 1) tma_load_3d(dst, map, bar, x, y, z);
    else tma_load_3d_pair(dst, map, bar, x, y, z);
}

// Copies of one operand (`rows` rows of op(X) starting at row0, this CTA's
// share) for the KPS k-blocks kb, kb + 1, ... of a stage into the region at
// dst, in the stage layout above. A stage box is one 3-D copy: K-major maps
// are (k in k-block, row, k-block), M/N-major maps (m or n in chunk, k,
// chunk). Otherwise one 2-D copy per k-block (and per chunk). SYR2K swaps the
// roles of tmA and tmB from k-block syr2k_kb on; with stage boxes the host only
// allows this when syr2k_kb is a whole number of stages.
template <int PAIR, int KPS, int ROWS, int KB_ELEMS>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap *map, const CUtensorMap *alt,
                                             bool box3, bool mn_major, uint32_t bar, int32_t row0, int kb,
                                             int syr2k_kb)
{
    if (box3) {
        const bool swap = syr2k_kb > 0 && kb >= syr2k_kb;
        const CUtensorMap *m = swap ? alt : map;
        const int kbs = swap ? kb - syr2k_kb : kb;
        if (mn_major) load_box3<PAIR>(dst, m, bar, 0, kbs * KB_ELEMS, row0 / 64);
        else load_box3<PAIR>(dst, m, bar, 0, row0, kbs);
        return;
    }
#pragma unroll
    for (int sub = 0; sub < KPS; ++sub) {
        const int kbs = kb + sub;
        const bool swap = syr2k_kb > 0 && kbs >= syr2k_kb;
        const CUtensorMap *m = swap ? alt : map;
        const int32_t kx = (swap ? kbs - syr2k_kb : kbs) * KB_ELEMS;
        if (mn_major) {
#pragma unroll
            for (int c = 0; c < ROWS / 64; ++c)
                load_box<PAIR>(dst + c * KPS * 8192 + sub * 8192, m, bar, row0 + 64 * c, kx);
        } else {
            load_box<PAIR>(dst + sub * ROWS * 128, m, bar, kx, row0);
        }
    }
}

// L2 prefetch of the stage boxes the producer will copy first (this CTA's
// share of its first unit's first 8 stages), in the coordinates of
// load_operand's stage-box branch. Measured: 8 stages beat the ring's 3 at
// K = 1024 (28.7 vs 29.5 us at 4096^2) and tie elsewhere; 32 stages made dX
// 5 % slower.
template <int BN, int STAGES, int PAIR, int ELEM, int KPS, int EPI>
__device__ __forceinline__ void prefetch_first_stages(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                                      const GemmParams &p, uint32_t rank)
{
    using Cfg = KernelCfg<BN, STAGES, PAIR, ELEM, KPS>;
    const int64_t u = first_unit<PAIR>();
    if (u >= p.num_units) return;
    const Unit w = map_unit<Cfg::TILE_M, BN, syrk_capable(ELEM, EPI)>(p, u);
    const int32_t row_a = static_cast<int32_t>(w.tm * Cfg::TILE_M + rank * CTA_M);
    const int32_t row_b = static_cast<int32_t>(w.tn * BN + rank * Cfg::B_ROWS);
    for (int s = 0, kb = w.kb0; s < 8 && kb < w.kb1; ++s, kb += KPS) {
        if (p.a_mn_major) tma_prefetch_3d(tmA, 0, kb * Cfg::KB_ELEMS, row_a / 64);
        else tma_prefetch_3d(tmA, 0, row_a, kb);
        if (p.b_mn_major) tma_prefetch_3d(tmB, 0, kb * Cfg::KB_ELEMS, row_b / 64);
        else tma_prefetch_3d(tmB, 0, row_b, kb);
    }
}

template <int PAIR>
__device__ __forceinline__ void load_box4(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t z, int32_t w)
{
    if constexpr (PAIR == 1) tma_load_4d(dst, map, bar, 0, 0, z, w);
    else tma_load_4d_pair(dst, map, bar, 0, 0, z, w);
}

template <int BN, int STAGES, int PAIR, int ELEM, int KPS, int EPI>
__device__ __forceinline__ void run_producer(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                             const CUtensorMap *tmSA, const CUtensorMap *tmSB,
                                             const GemmParams &p, uint32_t ring, uint32_t bar0, uint32_t rank,
                                             volatile int *abort_flag)
{
    using Cfg = KernelCfg<BN, STAGES, PAIR, ELEM, KPS>;
    const int64_t units = p.num_units;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;  // per stage: armed at least once / parity of last arming
    bool ok = true, first = true, issued_any = false;
    for (int64_t u = first_unit<PAIR>(); u < units && ok; u += unit_stride<PAIR>()) {
        const Unit w = map_unit<Cfg::TILE_M, BN, syrk_capable(ELEM, EPI)>(p, u);
        const int kb0 = w.kb0;
        const int kb1 = w.kb1;
        const int32_t row_a = static_cast<int32_t>(w.tm * Cfg::TILE_M + rank * CTA_M);
        const int32_t row_b = static_cast<int32_t>(w.tn * BN + rank * Cfg::B_ROWS);
        for (int kb = kb0; kb < kb1; kb += KPS) {
            const uint32_t empty = bar0 + 8u * (STAGES + stage);
            if (!wait_one<PAIR == 2>(empty, phase ^ 1u, abort_flag, p.timeout_ns)) {
                ok = false;
                break;
            }
            // Every stage copies KPS whole k-blocks; those past K (or past this
            // unit's K range, in the last stage of an odd-length unit) are zeros
            // or unused, but their bytes still count on the barrier.
            const uint32_t full = bar0 + 8u * stage;
            if (rank == 0) {
                mbar_arrive_expect_tx(full, static_cast<uint32_t>((Cfg::STAGE_BYTES + Cfg::SF_STAGE_BYTES) * PAIR));
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            }
            if (!(p.debug_stall && first)) {
                issued_any = true;
                // the pair's CTA 0 counts both CTAs' bytes
                const uint32_t bar = PAIR == 2 ? map_shared_to_rank(full, 0) : full;
                const uint32_t sa = ring + stage * Cfg::STAGE_BYTES;
                load_operand<PAIR, KPS, CTA_M, Cfg::KB_ELEMS>(sa, tmA, tmB, p.a_box3 != 0, p.a_mn_major != 0, bar,
                                                              row_a, kb, p.syr2k_kb);
                load_operand<PAIR, KPS, Cfg::B_ROWS, Cfg::KB_ELEMS>(sa + Cfg::B_OFFSET, tmB, tmA, p.b_box3 != 0,
                                                                    p.b_mn_major != 0, bar, row_b, kb, p.syr2k_kb);
                if constexpr (Cfg::SCALED) {
                    // this CTA's A scale atoms and all B scale atoms of the tile, KPS k-blocks
                    // (boxes past K or past the last row block are zero-filled and unused)
                    const uint32_t sf = ring + Cfg::RING_BYTES + stage * Cfg::SF_STAGE_BYTES;
                    load_box4<PAIR>(sf, tmSA, bar, kb, row_a / 128);
                    load_box4<PAIR>(sf + KPS * SF_ATOM_BYTES, tmSB, bar, kb, static_cast<int32_t>(w.tn * (BN / 128)));
                }
            }
            first = false;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        signal_timeout(p, abort_flag);
        // Let every copy this thread started land before shared memory is released.
        for (int s = 0; s < STAGES; ++s)
            if ((armed >> s) & 1u) wait_one(bar0 + 8u * s, (armed_parity >> s) & 1u, nullptr, p.timeout_ns);
        if (PAIR == 2 && issued_any) spin_ns(100000);  // copies counted on the other CTA's barrier
    }
}

template <int BN, int STAGES, int PAIR, int ELEM, int KPS, int EPI>
// The whole warp runs the loop and waits; lane 0 issues the MMAs and commits
// (a converged warp keeps the issue stream tighter than a lone diverged lane).
__device__ __forceinline__ void run_mma(const GemmParams &p, uint32_t ring, uint32_t bar0, uint32_t tmem_base,
                                        volatile int *abort_flag, int lane)
{
    using Cfg = KernelCfg<BN, STAGES, PAIR, ELEM, KPS>;
    const int64_t units = p.num_units;

    // Shared-memory descriptors are built once: a template with the start address
    // left at 0, plus the address >> 4 in the low 14 bits per MMA. Shared addresses
    // are below 256 KB, so the sum never carries into the next field. Steps, in
    // 16-byte units: K-major operands advance 32 B per 16 k and one tile per
    // k-block of the stage; M/N-major ones two 1024-byte row groups per 16 k and
    // 8 KB per k-block (the next 64 M/N lines are one chunk, KPS x 8 KB, further).
    // This keeps the issuing warp to a few instructions per MMA: it shares its SM
    // sub-partition with two epilogue warps.
    const uint64_t a_tpl = p.a_mn_major ? smem_desc_sw128(0u, Cfg::CHUNK_BYTES, 1024u) : smem_desc_sw128(0u, 16u, 1024u);
    const uint64_t b_tpl = p.b_mn_major ? smem_desc_sw128(0u, Cfg::CHUNK_BYTES, 1024u) : smem_desc_sw128(0u, 16u, 1024u);
    const uint32_t a_kk = p.a_mn_major ? 2048u / 16u : 32u / 16u;
    const uint32_t b_kk = p.b_mn_major ? 2048u / 16u : 32u / 16u;
    const uint32_t a_sub = p.a_mn_major ? 8192u / 16u : static_cast<uint32_t>(Cfg::A_BYTES) / 16u;
    const uint32_t b_sub = p.b_mn_major ? 8192u / 16u : static_cast<uint32_t>(Cfg::B_BYTES) / 16u;
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued_any = false;
    for (int64_t u = first_unit<PAIR>(); u < units && ok; u += unit_stride<PAIR>()) {
        const Unit w = map_unit<Cfg::TILE_M, BN, syrk_capable(ELEM, EPI)>(p, u);
        const int kb0 = w.kb0;
        const int kb1 = w.kb1;
        const uint32_t acc_empty = bar0 + 8u * (2 * STAGES + 2 + acc);
        if (!wait_one<PAIR == 2>(acc_empty, acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        // N halves (pair 256 x 256 tiles): N = BN / 2 over rows nh * 64 .. of each CTA's
        // B tile; the second half starts one 64-row chunk (M/N-major) or 64 x 128 bytes
        // (K-major) in.
        const uint32_t idesc = idesc_f32acc(Cfg::TILE_M, w.nh < 0 ? BN : BN / 2, ELEM == ELEM_BF16 ? 1u : 0u,
                                            p.a_mn_major, p.b_mn_major);
        const uint32_t b_nh =
            w.nh > 0 ? (p.b_mn_major ? static_cast<uint32_t>(Cfg::CHUNK_BYTES) : 64u * 128u) / 16u : 0u;
        for (int kb = kb0; kb < kb1; kb += KPS) {
            if (!wait_one(bar0 + 8u * stage, phase, abort_flag, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int nkb = kb1 - kb < KPS ? kb1 - kb : KPS;
            const uint32_t st = ring + stage * Cfg::STAGE_BYTES;
            for (int sub = 0; sub < nkb; ++sub) {
                // k-block `sub` of the stage
                const uint64_t a0 = a_tpl + (st >> 4) + a_sub * sub;
                const uint64_t b0 = b_tpl + ((st + Cfg::B_OFFSET) >> 4) + b_sub * sub + b_nh;
                // MXFP8: the k-block's scale atoms into this ring slot's tensor-memory
                // columns (A's, then B's), ahead of the MMAs that read them. A slot is
                // rewritten only after the MMAs of its last use have completed: its
                // stage's full barrier follows the empty barrier those MMAs' commit
                // arrived on.
                uint32_t sf_tmem = 0;
                if constexpr (Cfg::SCALED) {
                    const uint32_t sf = ring + Cfg::RING_BYTES + stage * Cfg::SF_STAGE_BYTES;
                    sf_tmem = tmem_base + static_cast<uint32_t>(Cfg::ACC_COLS + (stage * KPS + sub) * Cfg::SF_KB_COLS);
                    if (lane == 0) {
#pragma unroll
                        for (int at = 0; at <= Cfg::SF_B_ATOMS; ++at) {
                            // atom 0: A's (box offset sub); atoms 1..: B's (box offset KPS + (at-1) KPS + sub)
                            const uint32_t src = sf + static_cast<uint32_t>(
                                (at == 0 ? sub : KPS + (at - 1) * KPS + sub) * SF_ATOM_BYTES);
                            const uint64_t sd = smem_desc_plain(src, 16u, 128u);
                            if constexpr (PAIR == 1) tmem_cp_32x128b_x4(sf_tmem + 4u * at, sd);
                            else tmem_cp_32x128b_x4_pair(sf_tmem + 4u * at, sd);
                        }
                    }
                }
#pragma unroll
                for (int kk = 0; kk < TILE_K / UMMA_K; ++kk) {
                    const uint64_t ad = a0 + a_kk * kk;
                    const uint64_t bd = b0 + b_kk * kk;
                    const uint32_t accumulate = (kb > kb0 || sub > 0 || kk > 0) ? 1u : 0u;
                    if (lane == 0) {
                        if constexpr (ELEM == ELEM_MXF8) {
                            // scale byte kk: the kk-th group of 32 elements of this k-block
                            const uint32_t id = idesc_mxf8(Cfg::TILE_M, BN, static_cast<uint32_t>(kk));
                            if constexpr (PAIR == 1) umma_mxf8(d_tmem, ad, bd, id, sf_tmem, sf_tmem + 4u, accumulate);
                            else umma_mxf8_pair(d_tmem, ad, bd, id, sf_tmem, sf_tmem + 4u, accumulate);
                        } else if constexpr (ELEM == ELEM_E4M3) {
                            if constexpr (PAIR == 1) umma_f8(d_tmem, ad, bd, idesc, accumulate);
                            else umma_f8_pair(d_tmem, ad, bd, idesc, accumulate);
                        } else {
                            if constexpr (PAIR == 1) umma_bf16(d_tmem, ad, bd, idesc, accumulate);
                            else umma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
                        }
                    }
                }
            }
            issued_any = true;
            // the stage is free (in both CTAs) once these MMAs finish
            if (lane == 0) {
                if constexpr (PAIR == 1) umma_commit(bar0 + 8u * (STAGES + stage));
                else umma_commit_pair(bar0 + 8u * (STAGES + stage), 0x3);
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs)
        if (lane == 0) {
            if constexpr (PAIR == 1) umma_commit(bar0 + 8u * (2 * STAGES + acc));
            else umma_commit_pair(bar0 + 8u * (2 * STAGES + acc), 0x3);
        }
        if (++acc == Cfg::NUM_ACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
    if (!ok) {
        signal_timeout(p, abort_flag);
        if (issued_any) {  // drain: MMAs in flight must finish before TMEM is freed
            const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);
            if (lane == 0) {
                if constexpr (PAIR == 1) umma_commit(drain);
                else umma_commit_pair(drain, 0x1);
            }
            wait_one(drain, 0u, nullptr, p.timeout_ns);
        }
    }
}

// EPI selects the epilogue paths compiled in. EPI_FULL has them all (SYRK needs
// the triangle masks of the transposing path for tiles across the diagonal). The
// GEMM copies keep only what they use, which keeps them free of register spills:
// EPI_STORE (beta == 0) stores whole tiles with per-warp TMA stores, EPI_COMBINE
// (beta != 0) through the group path; split units take the slot-map TMA stores,
// or the transposing path with the in-kernel sum.
template <int BN, int STAGES, int PAIR, int ELEM, int KPS, int EPI = EPI_FULL>
__device__ __forceinline__ void run_epilogue(const CUtensorMap *tmC, const CUtensorMap *tmP, const GemmParams &p,
                                             uint32_t bar0, uint32_t tmem_base, float *epi, uint32_t rank,
                                             volatile int *abort_flag, int warp, int lane)
{
    using Cfg = KernelCfg<BN, STAGES, PAIR, ELEM, KPS>;
    const int64_t units = p.num_units;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31 are this warp's rows
    const int half = (warp - 2) >> 2;  // which of the two warps on this quadrant: even or odd chunks
    const int group_bar = 1 + half;    // named barrier of the four warps of this half
    float *stage_buf = epi + (warp - 2) * EPI_WARP_FLOATS;  // this warp's own block (per-warp path)
    const bool beta_nonzero = p.beta != 0.0f;
    const bool issuer = quad == 0 && lane == 0;  // issues this half's TMA copies in the group path
    int acc = 0;
    uint32_t acc_phase = 0, c_phase = 0;
    // This half's staging block has nothing in flight: no unit yet, or the last unit
    // took the group path (its stores have read the block and the half has met).
    // After other paths a warp of the half may still be using its own staging area
    // inside the block.
    bool block_free = true;
    for (int64_t u = first_unit<PAIR>(); u < units; u += unit_stride<PAIR>()) {
        const Unit w = map_unit<Cfg::TILE_M, BN, syrk_capable(ELEM, EPI)>(p, u);
        const bool to_slot = w.slot >= 0;
        // Paths: beta != 0 tiles of GEMM (and SYRK tiles inside the triangle) go through
        // the group path (TMA load of C, combine, TMA store); beta == 0 tiles and the
        // split units of the reduce-kernel plan through the per-warp TMA-store path; SYRK
        // tiles across the diagonal, split units of the in-kernel reduction and calls
        // without a C tensor map through the per-warp transposing path.
        const bool inside = tile_inside_triangle<Cfg::TILE_M, BN>(p.mode, w.tm, w.tn);
        const bool group = EPI == EPI_COMBINE ? !to_slot
                                              : EPI == EPI_FULL && !to_slot && beta_nonzero && p.tma_c && inside;
        const bool slot_tma = p.store_p_tma != 0 && !p.fixup;  // split units of the reduce-kernel plan
        // (split units of the in-kernel reduction store their partials with plain
        // stores, which the arrival's fence orders before the counter update)
        const bool warp_tma = EPI == EPI_STORE   ? !to_slot || slot_tma
                              : EPI == EPI_COMBINE ? to_slot && slot_tma
                                                   : (to_slot ? slot_tma : (!beta_nonzero && p.tma_c && inside));
        // Group path: this half's staging block and C-load barrier. When the block is
        // free, the tile's first chunk of C is loaded before the accumulator is ready,
        // so that its latency overlaps the tile's last MMAs instead of the epilogue.
        uint8_t *block = reinterpret_cast<uint8_t *>(epi) + half * GROUP_BLOCK_BYTES;
        const uint32_t block_addr = smem_addr(block);
        const uint32_t cbar = bar0 + 8u * (2 * STAGES + 5 + half);
        const int32_t ys = static_cast<int32_t>(w.tm * Cfg::TILE_M + rank * CTA_M);
        const int32_t xs0 = static_cast<int32_t>(unit_col<BN, PAIR>(w.tn * BN, w.nh, half * (p.c_bf16 ? 64 : 32)));
        const bool pre = group && block_free && issuer && ys < p.m && xs0 < p.n;
        if (pre) {
            mbar_arrive_expect_tx(cbar, GROUP_BLOCK_BYTES);
            tma_load_2d(block_addr, tmC, cbar, xs0, ys);
        }
        bool ready = wait_warp<PAIR == 2>(bar0 + 8u * (2 * STAGES + acc), acc_phase, abort_flag, p.timeout_ns);
        // A half that will meet at named barriers decides together, so that none of its
        // warps is left waiting at one.
        if (group) ready = group_all(ready, group_bar, 128);
        if (!ready) {
            if (lane == 0) signal_timeout(p, abort_flag);
            if (pre) spin_ns(100000);  // the C copy may still land in the block
            break;
        }
        tc_fence_after_sync();
        // split 0 of an in-kernel reduction adds beta * C to its partial (full vectors)
        const bool fold_beta = to_slot && p.fixup && beta_nonzero && w.kb0 == 0;
        const bool use_beta_fast = beta_nonzero && (w.slot < 0 || fold_beta);
        // split units: this CTA's rows of the tile's fp32 partial slot
        float *slot_rows = w.slot < 0 ? nullptr
                                      : p.partial + w.slot * static_cast<int64_t>(Cfg::TILE_M * BN) +
                                            static_cast<int64_t>(rank * CTA_M + quad * 32) * BN;
        const int64_t row0 = w.tm * Cfg::TILE_M + rank * CTA_M + quad * 32;
        const int64_t col0 = w.tn * BN;
        // accumulator columns of this unit (half units exist only for 256 x 256 pair tiles)
        const int acc_cols = (PAIR == 2 && BN == 256 && w.nh >= 0) ? BN / 2 : BN;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
        if (group) {
            // Per chunk of 128 bytes per row (64 bf16 or 32 fp32 columns), one thread of
            // this half loads the chunk of C (its 128 rows) into one 128B-swizzled
            // staging block with a single TMA copy; the four warps each combine their
            // 32 rows in place (beta * c + alpha * acc, as the other paths) and one
            // TMA copy stores the block back (the map clips rows >= m and columns >= n;
            // C has a map only when its rows end on a 16-byte boundary, the unit the
            // store clips columns to).
            const CUtensorMap *map = tmC;
            const bool bf16_out = p.c_bf16 != 0;
            const int cw = bf16_out ? 64 : 32;
            const int nchunks = acc_cols / cw;
            uint4 *myrow = reinterpret_cast<uint4 *>(block + (quad * 32 + lane) * 128);
            const bool rows_in = ys < p.m;
            bool gok = true, loading = pre;
            for (int c = half; c < nchunks; c += 2) {
                const int32_t xs = static_cast<int32_t>(unit_col<BN, PAIR>(col0, w.nh, c * cw));
                const bool live = rows_in && xs < p.n;  // the same for the whole half
                if (issuer && live && !(c == half && pre)) {  // (or it went out before the wait)
                    mbar_arrive_expect_tx(cbar, GROUP_BLOCK_BYTES);
                    tma_load_2d(block_addr, map, cbar, xs, ys);
                    loading = true;
                }
                bool ok = true;
                if (live) {
                    ok = wait_warp<false>(cbar, c_phase, abort_flag, p.timeout_ns);
                    c_phase ^= 1u;
                }
                // 32 accumulator columns at a time: 16-byte units 0-3 of the row (bf16) or
                // all 8 (fp32, one pass)
                for (int part = 0; part < cw / 32; ++part) {
                    uint32_t r[32];
                    tmem_load_32cols(taddr + static_cast<uint32_t>(c * cw + 32 * part), r);
                    if (ok) {
                        if (bf16_out) {
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                uint4 *slot = myrow + ((4 * part + jj) ^ (lane & 7));
                                const uint4 old = *slot;
                                uint4 q;
                                q.x = combine_bf16x2(p, r[8 * jj + 0], r[8 * jj + 1], old.x);
                                q.y = combine_bf16x2(p, r[8 * jj + 2], r[8 * jj + 3], old.y);
                                q.z = combine_bf16x2(p, r[8 * jj + 4], r[8 * jj + 5], old.z);
                                q.w = combine_bf16x2(p, r[8 * jj + 6], r[8 * jj + 7], old.w);
                                *slot = q;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                uint4 *slot = myrow + (j ^ (lane & 7));
                                const uint4 old = *slot;
                                uint4 q;
                                q.x = combine_f32(p, r[4 * j + 0], old.x);
                                q.y = combine_f32(p, r[4 * j + 1], old.y);
                                q.z = combine_f32(p, r[4 * j + 2], old.z);
                                q.w = combine_f32(p, r[4 * j + 3], old.w);
                                *slot = q;
                            }
                        }
                    }
                }
                if (c + 2 >= nchunks) {  // this warp's last chunk of the tile: release the accumulator
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t acc_empty = bar0 + 8u * (2 * STAGES + 2 + acc);
                        if constexpr (PAIR == 1) mbar_arrive(acc_empty);
                        else mbar_arrive_remote(map_shared_to_rank(acc_empty, 0));
                    }
                }
                fence_proxy_async_shared();
                gok = group_all(ok, group_bar, 128);  // every row of the block is written
                if (!gok) break;
                loading = false;
                if (issuer && live) {
                    tma_store_2d(map, block_addr, xs, ys);
                    bulk_commit_group();
                    bulk_wait_group_read0();  // the store has read the block
                }
                group_sync(group_bar, 128);  // the block may be written again
            }
            if (!gok) {
                if (lane == 0) signal_timeout(p, abort_flag);
                if (issuer && loading) spin_ns(100000);  // a C copy may still land in the block
                break;
            }
        } else if (warp_tma) {
            // Chunks of 128 bytes per row (64 bf16 or 32 fp32 columns), 32 rows: each lane
            // converts its row into a 128B-swizzled staging block, one lane stores it with
            // TMA, into C (the map clips rows >= m and columns >= n; C has a map only
            // when its rows end on a 16-byte boundary) or into the unit's fp32 partial slot.
            const CUtensorMap *map = to_slot ? tmP : tmC;
            const bool bf16_out = !to_slot && p.c_bf16;
            const int cw = bf16_out ? 64 : 32;
            const int nchunks = acc_cols / cw;
            const uint32_t stage_addr = smem_addr(stage_buf);
            const int64_t slot_row = to_slot ? w.slot * Cfg::TILE_M + rank * CTA_M + quad * 32 : 0;
            constexpr bool kReadAllFirst = BN == 256 && EPI == EPI_STORE;
            if (kReadAllFirst && bf16_out) {
                // Both chunks of this warp (64-column chunks half and half + 2; a half unit
                // has only the first) are read from tensor memory and packed to bf16 before
                // any store, so the accumulator goes back to the MMA warp without waiting
                // behind a store: the C stores queue on the SM's TMA unit with the operand
                // copies, and with short K the next tile's MMAs are ready long before the
                // stores have drained.
                const bool two = w.nh < 0;
                uint32_t h[2][32];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (j == 1 && !two) continue;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {  // 32 columns at a time
                        uint32_t r[32];
                        tmem_load_32cols(taddr + static_cast<uint32_t>((half + 2 * j) * 64 + 32 * part), r);
                        if (p.alpha == 1.0f) pack_32_bf16<false>(h[j] + 16 * part, r, p.alpha);
                        else pack_32_bf16<true>(h[j] + 16 * part, r, p.alpha);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t acc_empty = bar0 + 8u * (2 * STAGES + 2 + acc);
                    if constexpr (PAIR == 1) mbar_arrive(acc_empty);
                    else mbar_arrive_remote(map_shared_to_rank(acc_empty, 0));
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (j == 1 && !two) continue;
                    if (lane == 0) bulk_wait_group_read0();  // the previous store has read the staging block
                    __syncwarp();
                    stage_row_packed(reinterpret_cast<uint4 *>(stage_buf) + lane * 8, h[j], lane);
                    fence_proxy_async_shared();
                    __syncwarp();
                    const int64_t cx = unit_col<BN, PAIR>(col0, w.nh, (half + 2 * j) * 64);
                    if (lane == 0 && row0 < p.m && cx < p.n) {
                        tma_store_2d(map, stage_addr, static_cast<int32_t>(cx), static_cast<int32_t>(row0));
                        bulk_commit_group();
                    }
                }
            } else {
                for (int c = half; c < nchunks; c += 2) {
                    uint32_t r[64];
                    tmem_load_32cols(taddr + static_cast<uint32_t>(c * cw),
                                     *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                    if (bf16_out)
                        tmem_load_32cols(taddr + static_cast<uint32_t>(c * cw + 32),
                                         *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                    if (c + 2 >= nchunks) {  // this warp's last chunk of the tile: release the accumulator
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            const uint32_t acc_empty = bar0 + 8u * (2 * STAGES + 2 + acc);
                            if constexpr (PAIR == 1) mbar_arrive(acc_empty);
                            else mbar_arrive_remote(map_shared_to_rank(acc_empty, 0));
                        }
                    }
                    if (lane == 0) bulk_wait_group_read0();  // the previous store has read the staging block
                    __syncwarp();
                    uint4 *srow = reinterpret_cast<uint4 *>(stage_buf) + lane * 8;
                    // (alpha == 1 skips the multiplies: fewer instructions for the warps that
                    // share sub-partitions with the producer and MMA warps)
                    if (bf16_out) {
                        if (p.alpha == 1.0f) stage_row_bf16<false>(srow, r, p.alpha, lane);
                        else stage_row_bf16<true>(srow, r, p.alpha, lane);
                    } else {
                        if (p.alpha == 1.0f) stage_row_f32<false>(srow, r, p.alpha, lane);
                        else stage_row_f32<true>(srow, r, p.alpha, lane);
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        if (to_slot) {
                            tma_store_2d(map, stage_addr, c * cw, static_cast<int32_t>(slot_row));
                            bulk_commit_group();
                        } else {
                            const int64_t cx = unit_col<BN, PAIR>(col0, w.nh, c * cw);
                            if (row0 < p.m && cx < p.n) {
                                tma_store_2d(map, stage_addr, static_cast<int32_t>(cx), static_cast<int32_t>(row0));
                                bulk_commit_group();
                            }
                        }
                    }
                }
            }
        } else {
#pragma unroll 1
        for (int ch = half; ch < BN / 32; ch += 2) {
            uint32_t r[32];
            tmem_load_32cols(taddr + 32u * ch, r);
            if (ch >= BN / 32 - 2) {  // this warp's last chunk: its part of the accumulator is read
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t acc_empty = bar0 + 8u * (2 * STAGES + 2 + acc);
                    if constexpr (PAIR == 1) mbar_arrive(acc_empty);
                    else mbar_arrive_remote(map_shared_to_rank(acc_empty, 0));
                }
            }
            // SYRK tiles across the diagonal: a block wholly outside the triangle is
            // skipped (the other triangle is neither read nor written).
            if (block_outside_triangle(p.mode, row0, col0 + 32 * ch)) continue;
            // Row `lane` of this 32 x 32 block into shared memory; 16-byte chunk c of
            // row r goes to slot c ^ (r & 7) so that both passes are conflict-free.
            float4 *srow = reinterpret_cast<float4 *>(stage_buf + lane * 32);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                srow[c ^ (lane & 7)] =
                    make_float4(p.alpha * __uint_as_float(r[4 * c + 0]), p.alpha * __uint_as_float(r[4 * c + 1]),
                                p.alpha * __uint_as_float(r[4 * c + 2]), p.alpha * __uint_as_float(r[4 * c + 3]));
            __syncwarp();
            // Coalesced pass: 8 lanes cover one 32-column row segment, 4 rows per step.
            // With beta != 0 the old C values of all 8 steps are loaded first, so the
            // loads are in flight together instead of one load latency per step.
            const int cc = lane & 7;
            const int64_t gj0 = col0 + ch * 32 + cc * 4;
            uint4 old[8];
            if (use_beta_fast) {
#pragma unroll
                for (int step = 0; step < 8; ++step) {
                    const int64_t gi = row0 + step * 4 + (lane >> 3);
                    old[step] = make_uint4(0u, 0u, 0u, 0u);
                    if (!full_vector(p, gi, gj0)) continue;
                    if (p.c_bf16) {
                        const uint2 o = *reinterpret_cast<const uint2 *>(
                            reinterpret_cast<const __nv_bfloat16 *>(p.C) + gi * p.ldc + gj0);
                        old[step].x = o.x;
                        old[step].y = o.y;
                    } else {
                        old[step] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const float *>(p.C) +
                                                                      gi * p.ldc + gj0);
                    }
                }
            }
#pragma unroll
            for (int step = 0; step < 8; ++step) {
                const int rr = step * 4 + (lane >> 3);
                const float4 v4 = reinterpret_cast<const float4 *>(stage_buf + rr * 32)[cc ^ (rr & 7)];
                const int64_t gi = row0 + rr;
                if (slot_rows != nullptr) {  // whole tile row segment, edges included
                    const float4 x = fold_beta && full_vector(p, gi, gj0) ? add_beta_c4(p, v4, old[step]) : v4;
                    *reinterpret_cast<float4 *>(slot_rows + rr * BN + ch * 32 + cc * 4) = x;
                } else if (full_vector(p, gi, gj0)) {
                    float v[4] = {v4.x, v4.y, v4.z, v4.w};
                    if (use_beta_fast) {
                        write_c4_preloaded(p, gi, gj0, v, old[step]);
                    } else if (p.c_bf16) {
                        const __nv_bfloat162 r01 = __floats2bfloat162_rn(v[0], v[1]);
                        const __nv_bfloat162 r23 = __floats2bfloat162_rn(v[2], v[3]);
                        uint2 out;
                        out.x = *reinterpret_cast<const uint32_t *>(&r01);
                        out.y = *reinterpret_cast<const uint32_t *>(&r23);
                        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.C) + gi * p.ldc + gj0) = out;
                    } else {
                        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.C) + gi * p.ldc + gj0) = v4;
                    }
                } else if (gi < p.m && gj0 < p.n && !vector_outside_triangle(p.mode, gi, gj0)) {
                    write_c4_edge(p, gi, gj0, v4);
                }
            }
            __syncwarp();
        }
        if (to_slot && p.fixup) fixup_region<Cfg::TILE_M, BN, PAIR>(p, w.tm, w.tn, w.slot, rank, quad, half, warp, lane);
        }
        block_free = group;
        if (++acc == Cfg::NUM_ACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
    // Every thread that issued bulk stores (lane 0 of each warp in the per-warp path,
    // the half's issuer in the group path) waits for them: the CTA's shared memory
    // must outlive the copies that read it.
    if ((p.tma_c || p.store_p_tma) && lane == 0) bulk_wait_group0();
}

// ---------------------------------------------------------------- kernels
template <int BN, int STAGES, int PAIR, int ELEM, int KPS, int EPI = EPI_FULL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bm_gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
                           const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                           const GemmParams p)
{
    using Cfg = KernelCfg<BN, STAGES, PAIR, ELEM, KPS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t *smem = smem_raw + pad;
    const uint32_t ring = raw + pad;  // identical offset in both CTAs of a pair
    float *epi = reinterpret_cast<float *>(smem + Cfg::RING_BYTES + Cfg::SF_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::RING_BYTES + Cfg::SF_BYTES + Cfg::EPI_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = smem_addr(bars);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR == 2 ? cluster_cta_rank() : 0u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8u * s, 1);             // full: CTA 0's expect_tx arrival (+ bytes)
            mbar_init(bar0 + 8u * (STAGES + s), 1);  // empty: one tcgen05.commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar0 + 8u * (2 * STAGES + b), 1);                         // accumulator full
            mbar_init(bar0 + 8u * (2 * STAGES + 2 + b), NUM_EPI_WARPS * PAIR);  // accumulator empty
        }
        mbar_init(bar0 + 8u * (2 * STAGES + 4), 1);  // drain (abort path only)
        mbar_init(bar0 + 8u * (2 * STAGES + 5), 1);  // C load, epilogue half 0
        mbar_init(bar0 + 8u * (2 * STAGES + 6), 1);  // C load, epilogue half 1
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        if constexpr (Cfg::SCALED) {
            tma_prefetch_map(&tmSA);
            tma_prefetch_map(&tmSB);
        }
        if (p.tma_c) tma_prefetch_map(&tmC);
        if (p.store_p_tma) tma_prefetch_map(&tmP);
    }
    if (warp == 1) {
        if constexpr (PAIR == 1) {
            tmem_alloc(smem_addr(tmem_slot), Cfg::TMEM_COLS);
            tmem_relinquish();
        } else {
            tmem_alloc_pair(smem_addr(tmem_slot), Cfg::TMEM_COLS);
            tmem_relinquish_pair();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR == 2) cluster_sync();  // peer barriers initialised before any remote arrival
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // The set-up above overlaps the end of the previous kernel on the stream; no
    // global memory (A, B, C, workspace) is read into the SM or written before that
    // kernel is complete (the L2 prefetch below brings no data into the SM).
    griddep_launch_dependents();
    // While the previous kernel finishes, bring this CTA's operand boxes for its
    // first stages into L2 (a prefetch only warms the cache, so
    // it is safe before the wait even if that kernel writes A or B).
    if (warp == 0 && lane == 0 && p.a_box3 && p.b_box3 && p.syr2k_kb == 0)
        prefetch_first_stages<BN, STAGES, PAIR, ELEM, KPS, EPI>(&tmA, &tmB, p, rank);
    griddep_wait();

    if (warp == 0) {
        if (lane == 0) run_producer<BN, STAGES, PAIR, ELEM, KPS, EPI>(&tmA, &tmB, &tmSA, &tmSB, p, ring, bar0, rank,
                                                                        abort_flag);
    } else if (warp == 1) {
        if (rank == 0) run_mma<BN, STAGES, PAIR, ELEM, KPS, EPI>(p, ring, bar0, tmem_base, abort_flag, lane);
    } else {
        run_epilogue<BN, STAGES, PAIR, ELEM, KPS, EPI>(&tmC, &tmP, p, bar0, tmem_base, epi, rank,
                                       abort_flag,
                                       warp, lane);
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR == 2) cluster_sync();  // no CTA leaves while its peer may still touch it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        if constexpr (PAIR == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
        else tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

// Split tiles: sum of the K-split partial slots in split order, then beta * C,
// cast and masked store. TM x BN is the tile of the kernel that wrote them.
template <int TM, int BN>
__global__ void __launch_bounds__(256) bm_splitk_reduce_kernel(const GemmParams p)
{
    griddep_launch_dependents();
    griddep_wait();  // the partial slots come from the previous kernel
    const int64_t split_tiles = p.num_tiles - p.full_tiles;
    const int64_t per_tile = static_cast<int64_t>(TM) * (BN / 4);
    const int64_t total = split_tiles * per_tile;
    const int64_t slot_elems = static_cast<int64_t>(TM) * BN;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t local = idx / per_tile;
        const int64_t rem = idx - local * per_tile;
        const int r = static_cast<int>(rem / (BN / 4));
        const int c = static_cast<int>(rem - static_cast<int64_t>(r) * (BN / 4)) * 4;
        int64_t tm, tn;
        tile_coords<TM, BN>(p, p.full_tiles + local, tm, tn);
        const int64_t i = tm * TM + r;
        const int64_t j = tn * BN + c;
        if (i >= p.m || j >= p.n) continue;
        const float *src = p.partial + local * p.k_splits * slot_elems + static_cast<int64_t>(r) * BN + c;
        float4 s = *reinterpret_cast<const float4 *>(src);
        // Loads of up to 8 slots are issued together, then added one after the
        // other in split order (the sum itself is sequential).
        int sp = 1;
        for (; sp + 8 <= p.k_splits; sp += 8) {
            float4 t[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) t[q] = *reinterpret_cast<const float4 *>(src + (sp + q) * slot_elems);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                s.x += t[q].x;
                s.y += t[q].y;
                s.z += t[q].z;
                s.w += t[q].w;
            }
        }
        for (; sp < p.k_splits; ++sp) {
            const float4 t = *reinterpret_cast<const float4 *>(src + sp * slot_elems);
            s.x += t.x;
            s.y += t.y;
            s.z += t.z;
            s.w += t.w;
        }
        float v[4] = {s.x, s.y, s.z, s.w};
        write_c4(p, i, j, v);
    }
}

// alpha == 0 or k == 0: C = beta * C on the output region (C unread when beta == 0).
__global__ void __launch_bounds__(256) bm_scale_kernel(const GemmParams p)
{
    griddep_launch_dependents();
    griddep_wait();
    const int64_t cols4 = (p.n + 3) / 4;
    const int64_t total = p.m * cols4;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = idx / cols4;
        const int64_t j = (idx - i * cols4) * 4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        write_c4(p, i, j, v);
    }
}

}  // namespace bm
